// Device helpers shared by the attention backward kernels (the split dK/dV and
// dQ kernels and the fused kernel): tile constants, warp roles, bf16 packing,
// the key-mask bits of a key tile and the work-item decoding.
#pragma once

#include "uaa_common.cuh"

namespace uaa {
namespace {

constexpr int kBT = 128;  // rows per query tile and per key tile
constexpr int kChunkBytes = 128 * 128;
constexpr int kComputeThreads = 256;  // warps 0-7
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;    // the MMA issuer (dQ and fused kernels: the first of two)
constexpr int kMmaWarp1 = 10;  // the second MMA issuer of the dQ and fused kernels
constexpr int kThreads = 352;  // the dQ and fused kernels' block (the dK/dV kernel uses warps 0-9)

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}


// Warp-collective: the attended-key bits of key tile j of sequence kd (bit c of
// word t = key c' = 32t + c of the tile); keys past the tile's segment count as
// masked.  Every lane gets all 4 words.  key_mask is (B, kd.total) in sequence order.
__device__ __forceinline__ void key_tile_bits(const uint8_t* __restrict__ key_mask, const SeqDesc& kd, int b, int j,
                                              uint32_t (&w)[4]) {
  const int lane = threadIdx.x & 31;
  const SeqTile kt = seq_tile(kd, j);
  const size_t base = (size_t)b * kd.total + kd.off[kt.seg] + kt.row0;
#pragma unroll
  for (int t = 0; t < 4; ++t) {
    const int c = 32 * t + lane;
    const bool valid = c < kt.valid && (key_mask == nullptr || key_mask[base + c] != 0);
    w[t] = __ballot_sync(0xffffffffu, valid);
  }
}

__device__ __forceinline__ bool key_tile_any(const uint8_t* __restrict__ key_mask, const SeqDesc& kd, int b, int j) {
  uint32_t w[4];
  key_tile_bits(key_mask, kd, b, j, w);
  return (w[0] | w[1] | w[2] | w[3]) != 0;
}

// Packed bf16 pairs of 64 consecutive columns -> 32 TMEM columns (two stores).
__device__ __forceinline__ void store_packed64(uint32_t taddr, const float (&x)[64]) {
  uint32_t pk[32];
#pragma unroll
  for (int c = 0; c < 32; ++c) pk[c] = pack_bf16(x[2 * c], x[2 * c + 1]);
  tmem_st32_bits(taddr, pk);
}

struct Item3 {
  int t, h, b;
};
__device__ __forceinline__ Item3 decode_item(int item, int ntiles, int H) {
  Item3 it;
  it.t = item % ntiles;
  const int bh = item / ntiles;
  it.h = bh % H;
  it.b = bh / H;
  return it;
}
// The same items with the head innermost: (b, t, h).  With a key mask the empty key
// tiles of a batch (the cheap items) then form runs of H consecutive items, which the
// round-robin hand-out spreads evenly over the CTAs; the Q / dO streams in flight at
// once are those of all heads of one batch instead of a few heads.
__device__ __forceinline__ Item3 decode_item_head_inner(int item, int ntiles, int H) {
  Item3 it;
  it.h = item % H;
  const int bt = item / H;
  it.t = bt % ntiles;
  it.b = bt / ntiles;
  return it;
}

// TMEM column of the A operand for K step kk (16 elements = 8 packed columns)
// when the 128 packed K elements sit as two runs of 32 columns at base and
// base + 64 (column half hf of the compute warps writes its 64 elements into
// the first 32 columns of its own 64-column region).
__device__ __forceinline__ uint32_t packed_a_col(int kk) { return kk < 4 ? kk * 8 : 64 + (kk - 4) * 8; }

__host__ __device__ constexpr int padded_rows(int S) { return (S + 127) / 128 * 128; }

}  // namespace
}  // namespace uaa
