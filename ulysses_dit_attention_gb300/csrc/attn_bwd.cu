// Attention backward on sm_103a: dQ, dK, dV from Q, K, V, O, dO and the LSE.
//
// "Fix double transpose of K/V in templated attention backward", description
// and Test: the backward op takes Q, K, V in one layout (BSHD here, no second
// transpose), the output gradient in BSHD and the saved log-sum-exp, and must
// match an eager reference on all three gradients.  "[attention] Add Ulysses
// Anything backward", What does this PR do: the auxiliary LSE output is not
// differentiated; the backward of each head group is the plain attention
// backward.
//
// Three kernels:
//  1. bwd_preprocess_kernel: Delta_i = sum_d dO_id * O_id (fp32), equal to
//     sum_j P_ij dP_ij, and zeroes the fp32 dQ accumulator.
//  2. attn_bwd_kernel: one CTA per 128-key tile of one (batch, head), looping
//     over all 128-row query tiles (K/V-tile-major):
//        S^T  = K Q^T          (TMEM, M = keys)        P^T = exp2(S^T*c - lse2)
//        dP^T = V dO^T         (TMEM)                  dS^T = P^T (dP^T - Delta)
//        dV  += P^T dO         (TMEM accumulator, A = P^T from shared memory)
//        dK  += dS^T Q         (TMEM accumulator, A = dS^T from shared memory)
//        dQ_i = dS K           (TMEM, A = the same dS^T buffer read MN-major)
//     The fp32 dQ_i tile is staged in shared memory and added to the
//     accumulator with TMA tensor reduce-adds.
//     warp 8 = TMA producer, warp 9 = tcgen05 issuer, warps 0-7 = compute
//     (thread = key row; warps 0-3 take query columns 0-63, warps 4-7 64-127).
//     Keys outside the mask get P = 0, hence dK = dV = 0 exactly; a key tile
//     with no attended key writes zeros and skips all work.
//  3. dq_convert_kernel: dQ = bf16(scale * accumulator).
// TMEM columns: [0,128) S^T, [128,256) dP^T then dQ, [256,256+D) dV,
// [256+D,256+2D) dK.
#include <math.h>

#include <mutex>

#include "uaa_common.cuh"

namespace uaa {

int validate_attn_sizes(const char* fn, int B, int S, int H, int D, float scale);
int check_dev_ptr(const char* fn, const char* name, const void* p);

namespace {

constexpr int kBK = 128;  // keys per CTA (TMEM lanes)
constexpr int kBQ = 128;  // queries per inner tile
constexpr int kChunkBytes = 128 * 128;
constexpr int kComputeThreads = 256;  // warps 0-7
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr int kThreads = 320;

template <int D>
struct BwdLayout {
  static constexpr int kQStages = 2;
  static constexpr int kDStages = (D == 128) ? 1 : 2;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;
  static constexpr int kDO = kQ + kQStages * kTileBytes;
  static constexpr int kPDS = kDO + kDStages * kTileBytes;          // P^T, then dS^T, then half the dQ staging
  static constexpr int kSTG = kPDS + kBK * kBQ * 2;                 // the other half of the fp32 dQ staging
  static constexpr int kLse = kSTG + kBQ * (D / 2) * 4;
  static constexpr int kDelta = kLse + kQStages * kBQ * 4;
  static constexpr int kCtl = kDelta + kQStages * kBQ * 4;
  static constexpr int kSmem = kCtl + 256;
  static_assert(kSmem <= 232448, "backward shared memory exceeds the per-CTA limit");
  static_assert(kBQ * (D / 2) * 4 <= kBK * kBQ * 2, "dQ staging half must fit the P/dS buffer");
};

struct BwdCtl {
  uint64_t bar_kv;
  uint64_t bar_q_full[2];
  uint64_t bar_q_empty[2];
  uint64_t bar_do_full[2];
  uint64_t bar_do_empty[2];
  uint64_t bar_s_full;
  uint64_t bar_dp_full;
  uint64_t bar_p_ready;
  uint64_t bar_dv_done;
  uint64_t bar_ds_ready;
  uint64_t bar_dq_full;
  uint64_t bar_dq_free;
  uint64_t bar_pds_free;
  uint64_t bar_staged;
  uint64_t bar_kv_done;
  uint64_t bar_final;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(BwdCtl) <= 256, "control block");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const DevCtx& ctx, BwdCtl* ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ctl->abort)) return false;
    if (*reinterpret_cast<volatile unsigned int*>(ctx.status) & kStatusTimeout) {
      // another CTA already gave up: stop waiting (the launch has failed)
      *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
      return false;
    }
    if (globaltimer_ns() - t0 > ctx.timeout_ns) {
      atomicOr(ctx.status, kStatusTimeout);
      *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
      return false;
    }
  }
}

__device__ __forceinline__ void settle(uint64_t* bar, uint32_t parity, const DevCtx& ctx) {
  if (!mbar_wait(bar, parity, ctx.timeout_ns)) atomicOr(ctx.status, kStatusTimeout);
}

// Write 64 consecutive values of row `row` as bf16 into a 128-byte-swizzled
// K-major tile chunk (128 rows x 64 columns).
__device__ __forceinline__ void store_row_chunk_sw128(uint8_t* chunk, int row, const float (&x)[64]) {
#pragma unroll
  for (int pc = 0; pc < 8; ++pc) {
    uint4 v;
    v.x = pack_bf16(x[pc * 8 + 0], x[pc * 8 + 1]);
    v.y = pack_bf16(x[pc * 8 + 2], x[pc * 8 + 3]);
    v.z = pack_bf16(x[pc * 8 + 4], x[pc * 8 + 5]);
    v.w = pack_bf16(x[pc * 8 + 6], x[pc * 8 + 7]);
    *reinterpret_cast<uint4*>(chunk + row * 128 + ((pc ^ (row & 7)) << 4)) = v;
  }
}

// ---------------------------------------------------------------------------
// 1. Delta = rowsum(dO * O); zero the dQ accumulator.
// Eight lanes per (b, s, h) row, 16-byte loads; Delta stored as (B, H, S).
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             float* __restrict__ delta, float4* __restrict__ dq_acc,
                                                             int B, int S, int H, size_t acc_vec4) {
  constexpr int kVecPerRow = D / 8;        // 16-byte vectors per row
  constexpr int kPerLane = kVecPerRow / 8;  // vectors per lane (8 lanes per row)
  const size_t rows = (size_t)B * S * H;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  const int sub = threadIdx.x & 7;
  for (size_t base = tid >> 3; base < ((rows + 3) / 4) * 4; base += nthreads >> 3) {
    const size_t r = base;
    float acc = 0.f;
    if (r < rows) {
      const uint4* po = reinterpret_cast<const uint4*>(o + r * D);
      const uint4* pd = reinterpret_cast<const uint4*>(dout + r * D);
#pragma unroll
      for (int t = 0; t < kPerLane; ++t) {
        const uint4 a = __ldg(po + sub + 8 * t);
        const uint4 g = __ldg(pd + sub + 8 * t);
        const __nv_bfloat162* a2 = reinterpret_cast<const __nv_bfloat162*>(&a);
        const __nv_bfloat162* g2 = reinterpret_cast<const __nv_bfloat162*>(&g);
#pragma unroll
        for (int e = 0; e < 4; ++e) {
          const float2 af = __bfloat1622float2(a2[e]);
          const float2 gf = __bfloat1622float2(g2[e]);
          acc = fmaf(af.x, gf.x, acc);
          acc = fmaf(af.y, gf.y, acc);
        }
      }
    }
    acc += __shfl_xor_sync(0xffffffffu, acc, 4);
    acc += __shfl_xor_sync(0xffffffffu, acc, 2);
    acc += __shfl_xor_sync(0xffffffffu, acc, 1);
    if (r < rows && sub == 0) {
      const int h = (int)(r % H);
      const size_t bs = r / H;
      const int s = (int)(bs % S);
      const int b = (int)(bs / S);
      delta[((size_t)b * H + h) * S + s] = acc;
    }
  }
  const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
  for (size_t i = tid; i < acc_vec4; i += nthreads) dq_acc[i] = z;
}

// ---------------------------------------------------------------------------
// 3. dQ = bf16(scale * accumulator), 8 elements per thread.
__global__ void __launch_bounds__(256) dq_convert_kernel(const float4* __restrict__ acc, uint4* __restrict__ dq,
                                                         float scale, size_t n8) {
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < n8; i += (size_t)gridDim.x * blockDim.x) {
    const float4 a = __ldcs(acc + 2 * i);
    const float4 c = __ldcs(acc + 2 * i + 1);
    uint4 v;
    v.x = pack_bf16(a.x * scale, a.y * scale);
    v.y = pack_bf16(a.z * scale, a.w * scale);
    v.z = pack_bf16(c.x * scale, c.y * scale);
    v.w = pack_bf16(c.z * scale, c.w * scale);
    dq[i] = v;
  }
}

// ---------------------------------------------------------------------------
// 2. main backward kernel
//
// Per query tile i the tensor core runs, in this order,
//   dP^T_i = V dO_i^T             (TMEM columns [128,256))
//   dV    += P^T_i dO_i           (A = P^T in the shared P/dS buffer)
//   dK    += dS^T_i Q_i           (A = dS^T in the same buffer, after dV is done)
//   dQ_i   = dS_i K               (A = dS^T read MN-major; into the dP^T columns)
//   S^T_{i+1} = K Q_{i+1}^T       (TMEM columns [0,128))
// so S^T_{i+1} runs while the compute warps read dQ_i out of TMEM, and the
// fp32 dQ partial tile leaves through shared memory with TMA reduce-adds
// (cp.reduce.async.bulk.tensor ... .add) instead of per-thread atomics.
template <int D, bool kMask>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const __grid_constant__ CUtensorMap tmDO,
                    const __grid_constant__ CUtensorMap tmAcc, const float* __restrict__ lse,
                    const float* __restrict__ delta, const uint8_t* __restrict__ key_mask,
                    __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int S, int H, float scale,
                    float scale_log2, DevCtx ctx) {
  using L = BwdLayout<D>;
  constexpr int kChunks = D / 64;
  constexpr int QST = L::kQStages;
  constexpr int DST = L::kDStages;
  constexpr int kBoxes = D / 32;  // 32-column fp32 boxes of the dQ tile
  constexpr uint32_t kIdescKK = idesc_bf16_f32(128, kBQ, false, false);  // S^T, dP^T
  constexpr uint32_t kIdescKM = idesc_bf16_f32(128, D, false, true);     // dV, dK
  constexpr uint32_t kIdescMM = idesc_bf16_f32(128, D, true, true);      // dQ
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;

  extern __shared__ __align__(1024) uint8_t smem_raw[];
  uint8_t* smem = smem_raw;
  BwdCtl* ctl = reinterpret_cast<BwdCtl*>(smem + L::kCtl);
  float* sLse = reinterpret_cast<float*>(smem + L::kLse);
  float* sDelta = reinterpret_cast<float*>(smem + L::kDelta);
  const uint32_t sbase = smem_u32(smem);

  if (sbase & 1023u) {
    // the swizzled operand tiles need 1024-byte alignment; never expected to trigger
    if (threadIdx.x == 0) atomicOr(ctx.status, kStatusBadLaunch);
    return;
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int kt = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int k0 = kt * kBK;
  const int nqt = (S + kBQ - 1) / kBQ;

  if (kMask) {
    // A key tile without any attended key contributes nothing: dK = dV = 0.
    int valid = 0;
    if (threadIdx.x < kBK) {
      const int key = k0 + threadIdx.x;
      valid = key < S && key_mask[(size_t)b * S + key] != 0;
    }
    if (!__syncthreads_or(valid)) {
      constexpr int kVec = D / 8;
      for (int idx = threadIdx.x; idx < kBK * kVec; idx += kThreads) {
        const int r = idx / kVec;
        const int c = idx % kVec;
        if (k0 + r < S) {
          const size_t off = (((size_t)b * S + k0 + r) * H + h) * D + c * 8;
          *reinterpret_cast<uint4*>(dk + off) = make_uint4(0u, 0u, 0u, 0u);
          *reinterpret_cast<uint4*>(dv + off) = make_uint4(0u, 0u, 0u, 0u);
        }
      }
      return;
    }
  }

  if (threadIdx.x == 0) {
    mbar_init(&ctl->bar_kv, 1);
    for (int s = 0; s < 2; ++s) {
      mbar_init(&ctl->bar_q_full[s], 1);
      mbar_init(&ctl->bar_q_empty[s], 1);
      mbar_init(&ctl->bar_do_full[s], 1);
      mbar_init(&ctl->bar_do_empty[s], 1);
    }
    mbar_init(&ctl->bar_s_full, 1);
    mbar_init(&ctl->bar_dp_full, 1);
    mbar_init(&ctl->bar_p_ready, kComputeThreads);
    mbar_init(&ctl->bar_dv_done, 1);
    mbar_init(&ctl->bar_ds_ready, kComputeThreads);
    mbar_init(&ctl->bar_dq_full, 1);
    mbar_init(&ctl->bar_dq_free, kComputeThreads);
    mbar_init(&ctl->bar_pds_free, 1);
    mbar_init(&ctl->bar_staged, kComputeThreads);
    mbar_init(&ctl->bar_kv_done, 1);
    mbar_init(&ctl->bar_final, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
    tma_prefetch_desc(&tmDO);
    tma_prefetch_desc(&tmAcc);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  uint32_t q_armed[2] = {0, 0};
  uint32_t do_armed[2] = {0, 0};
  bool kv_armed = false;
  bool mma_issued = false;
  bool bulk_issued = false;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    if (lane == 0) {
      mbar_arrive_expect_tx(&ctl->bar_kv, 2 * L::kTileBytes);
#pragma unroll
      for (int c = 0; c < kChunks; ++c) {
        tma_load_4d(smem + L::kK + c * kChunkBytes, &tmK, &ctl->bar_kv, c * 64, h, k0, b);
        tma_load_4d(smem + L::kV + c * kChunkBytes, &tmV, &ctl->bar_kv, c * 64, h, k0, b);
      }
      kv_armed = true;
    }
    const float* lse_bh = lse + ((size_t)b * H + h) * S;
    const float* delta_bh = delta + ((size_t)b * H + h) * S;
    for (int i = 0; i < nqt; ++i) {
      const int qs = i % QST;
      const uint32_t qu = i / QST;
      if (lane == 0 && qu > 0) ok = wait_or_abort(&ctl->bar_q_empty[qs], (qu - 1) & 1, ctx, ctl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
#pragma unroll
      for (int t = 0; t < 4; ++t) {
        const int q = i * kBQ + 32 * t + lane;
        float l2 = INFINITY;  // rows past the end, and fully masked rows, get P = 0
        if (q < S) {
          const float l = lse_bh[q];
          if (l != -INFINITY) l2 = l * kLog2e;
        }
        sLse[qs * kBQ + 32 * t + lane] = l2;
        sDelta[qs * kBQ + 32 * t + lane] = q < S ? delta_bh[q] : 0.f;
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctl->bar_q_full[qs], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d(smem + L::kQ + qs * L::kTileBytes + c * kChunkBytes, &tmQ, &ctl->bar_q_full[qs], c * 64, h,
                      i * kBQ, b);
        q_armed[qs] = qu + 1;
      }
      const int ds = i % DST;
      const uint32_t du = i / DST;
      if (lane == 0 && du > 0) ok = wait_or_abort(&ctl->bar_do_empty[ds], (du - 1) & 1, ctx, ctl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctl->bar_do_full[ds], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d(smem + L::kDO + ds * L::kTileBytes + c * kChunkBytes, &tmDO, &ctl->bar_do_full[ds], c * 64,
                      h, i * kBQ, b);
        do_armed[ds] = du + 1;
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      const uint32_t sK = sbase + L::kK;
      const uint32_t sV = sbase + L::kV;
      const uint32_t sPDS = sbase + L::kPDS;
      auto issue_s = [&](int i) -> bool {
        const int qs = i % QST;
        if (!wait_or_abort(&ctl->bar_q_full[qs], (i / QST) & 1, ctx, ctl)) return false;
        tc_fence_after();
        const uint32_t sQ = sbase + L::kQ + qs * L::kTileBytes;
        // S^T = K Q^T  (M = keys, N = queries, K = D; both K-major)
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          mma_bf16(tmem + kColS, sdesc_sw128(sK + off, 16, 1024), sdesc_sw128(sQ + off, 16, 1024), kIdescKK,
                   kk > 0);
        }
        mma_commit(&ctl->bar_s_full);
        mma_issued = true;
        return true;
      };
      bool ok = wait_or_abort(&ctl->bar_kv, 0, ctx, ctl);
      tc_fence_after();
      if (ok) ok = issue_s(0);
      for (int i = 0; ok && i < nqt; ++i) {
        const int qs = i % QST;
        const int ds = i % DST;
        const uint32_t sQ = sbase + L::kQ + qs * L::kTileBytes;
        const uint32_t sDO = sbase + L::kDO + ds * L::kTileBytes;
        // dP^T = V dO^T into the columns dQ_{i-1} used: wait until it was read out
        if (i > 0) {
          if (!(ok = wait_or_abort(&ctl->bar_dq_free, (i - 1) & 1, ctx, ctl))) break;
          tc_fence_after();
        }
        if (!(ok = wait_or_abort(&ctl->bar_do_full[ds], (i / DST) & 1, ctx, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          mma_bf16(tmem + kColDP, sdesc_sw128(sV + off, 16, 1024), sdesc_sw128(sDO + off, 16, 1024), kIdescKK,
                   kk > 0);
        }
        mma_commit(&ctl->bar_dp_full);
        // dV += P^T dO  (A = P^T, K-major over queries; B = dO MN-major)
        if (!(ok = wait_or_abort(&ctl->bar_p_ready, i & 1, ctx, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          mma_bf16(tmem + kColDV, sdesc_sw128(sPDS + aoff, 16, 1024),
                   sdesc_sw128(sDO + kk * 2048, kChunkBytes, 1024), kIdescKM, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl->bar_do_empty[ds]);
        mma_commit(&ctl->bar_dv_done);
        // dK += dS^T Q  (A = dS^T, K-major over queries; B = Q MN-major)
        if (!(ok = wait_or_abort(&ctl->bar_ds_ready, i & 1, ctx, ctl))) break;
        tc_fence_after();
#pragma unroll
        for (int kk = 0; kk < kBQ / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          mma_bf16(tmem + kColDK, sdesc_sw128(sPDS + aoff, 16, 1024),
                   sdesc_sw128(sQ + kk * 2048, kChunkBytes, 1024), kIdescKM, (i > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl->bar_q_empty[qs]);
        // dQ_i = dS K  (A = dS^T read MN-major: M = queries, K = keys; B = K MN-major)
#pragma unroll
        for (int kk = 0; kk < kBK / 16; ++kk) {
          mma_bf16(tmem + kColDP, sdesc_sw128(sPDS + kk * 2048, kChunkBytes, 1024),
                   sdesc_sw128(sK + kk * 2048, kChunkBytes, 1024), kIdescMM, kk > 0);
        }
        mma_commit(&ctl->bar_dq_full);
        // S^T of the next tile (its columns were freed when P_i was formed)
        if (i + 1 < nqt && !(ok = issue_s(i + 1))) break;
      }
      if (ok) mma_commit(&ctl->bar_kv_done);
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ compute warps 0..7
    const int ctid = threadIdx.x;  // 0..255
    const int qd = warp & 3;
    const int hf = warp >> 2;
    const int jrow = qd * 32 + lane;  // key row (TMEM lane) in the S^T / dP^T phase; query row for dQ
    const uint32_t tl = tmem + ((uint32_t)(qd * 32) << 16);
    const int key = k0 + jrow;
    const bool kvalid = key < S && (!kMask || key_mask[(size_t)b * S + key] != 0);
    uint8_t* sPDSc = smem + L::kPDS + hf * kChunkBytes;
    // fp32 dQ staging: boxes [0, kBoxes/2) in the staging buffer, the rest in the P/dS buffer
    uint8_t* stg = hf == 0 ? smem + L::kSTG : smem + L::kPDS;
    bool ok = true;
    for (int i = 0; i < nqt; ++i) {
      const int qs = i % QST;
      ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_s_full, i & 1, ctx, ctl));
      if (!ok) break;
      tc_fence_after();
      float p[64];
      tmem_ld32(tl + kColS + 64 * hf, *reinterpret_cast<float(*)[32]>(&p[0]));
      tmem_ld32(tl + kColS + 64 * hf + 32, *reinterpret_cast<float(*)[32]>(&p[32]));
      ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_q_full[qs], (i / QST) & 1, ctx, ctl));
      if (!ok) break;
      {
        const float4* l2 = reinterpret_cast<const float4*>(sLse + qs * kBQ + 64 * hf);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 l = l2[c4];
          p[4 * c4 + 0] = kvalid ? ex2(fmaf(p[4 * c4 + 0], scale_log2, -l.x)) : 0.f;
          p[4 * c4 + 1] = kvalid ? ex2(fmaf(p[4 * c4 + 1], scale_log2, -l.y)) : 0.f;
          p[4 * c4 + 2] = kvalid ? ex2(fmaf(p[4 * c4 + 2], scale_log2, -l.z)) : 0.f;
          p[4 * c4 + 3] = kvalid ? ex2(fmaf(p[4 * c4 + 3], scale_log2, -l.w)) : 0.f;
        }
      }
      if (i > 0) {
        // the P/dS buffer also held the previous dQ staging: its TMA reads must be done
        if (ctid == 0) {
          bulk_wait_read_all();
          mbar_arrive(&ctl->bar_pds_free);
        }
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_pds_free, (i - 1) & 1, ctx, ctl));
        if (!ok) break;
      }
      store_row_chunk_sw128(sPDSc, jrow, p);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ctl->bar_p_ready);
      ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_dp_full, i & 1, ctx, ctl));
      if (!ok) break;
      tc_fence_after();
      float dp[64];
      tmem_ld32(tl + kColDP + 64 * hf, *reinterpret_cast<float(*)[32]>(&dp[0]));
      tmem_ld32(tl + kColDP + 64 * hf + 32, *reinterpret_cast<float(*)[32]>(&dp[32]));
      {
        // Delta_i sits with the Q_i stage (q_full was waited on above)
        const float4* dl = reinterpret_cast<const float4*>(sDelta + qs * kBQ + 64 * hf);
#pragma unroll
        for (int c4 = 0; c4 < 16; ++c4) {
          const float4 d = dl[c4];
          dp[4 * c4 + 0] = p[4 * c4 + 0] * (dp[4 * c4 + 0] - d.x);
          dp[4 * c4 + 1] = p[4 * c4 + 1] * (dp[4 * c4 + 1] - d.y);
          dp[4 * c4 + 2] = p[4 * c4 + 2] * (dp[4 * c4 + 2] - d.z);
          dp[4 * c4 + 3] = p[4 * c4 + 3] * (dp[4 * c4 + 3] - d.w);
        }
      }
      // P^T must have been consumed by the dV MMA before dS^T overwrites it
      ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_dv_done, i & 1, ctx, ctl));
      if (!ok) break;
      store_row_chunk_sw128(sPDSc, jrow, dp);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ctl->bar_ds_ready);
      // dQ_i: TMEM lane = query row of tile i; this thread takes columns [hf*D/2, (hf+1)*D/2)
      ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_dq_full, i & 1, ctx, ctl));
      if (!ok) break;
      tc_fence_after();
      float g[D / 2];
#pragma unroll
      for (int c = 0; c < D / 64; ++c)
        tmem_ld32(tl + kColDP + hf * (D / 2) + 32 * c, *reinterpret_cast<float(*)[32]>(&g[32 * c]));
      tc_fence_before();
      mbar_arrive(&ctl->bar_dq_free);
      // stage the fp32 partial tile (128-byte swizzled boxes of 32 columns) and reduce-add it
#pragma unroll
      for (int bx = 0; bx < D / 64; ++bx) {
        uint8_t* box = stg + bx * (kBQ * 128);
#pragma unroll
        for (int c4 = 0; c4 < 8; ++c4) {
          const float* src = &g[32 * bx + 4 * c4];
          *reinterpret_cast<float4*>(box + jrow * 128 + ((c4 ^ (jrow & 7)) << 4)) =
              make_float4(src[0], src[1], src[2], src[3]);
        }
      }
      fence_proxy_async_smem();
      mbar_arrive(&ctl->bar_staged);
      if (warp == 0) {
        bool staged = true;
        if (lane == 0) staged = wait_or_abort(&ctl->bar_staged, i & 1, ctx, ctl);
        ok = __all_sync(0xffffffffu, staged);
        if (!ok) break;
      }
      if (ctid == 0) {
#pragma unroll
        for (int bx = 0; bx < kBoxes; ++bx) {
          const uint8_t* box = (bx < kBoxes / 2 ? smem + L::kSTG : smem + L::kPDS) + (bx % (kBoxes / 2)) * (kBQ * 128);
          tma_reduce_add_4d(box, &tmAcc, 32 * bx, h, i * kBQ, b);
        }
        bulk_commit_group();
        bulk_issued = true;
      }
    }
    if (ctid == 0 && bulk_issued) bulk_wait_all();  // the reductions have landed before the kernel ends
    if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_kv_done, 0, ctx, ctl));
    if (ok) {
      tc_fence_after();
      const size_t off = (((size_t)b * S + key) * H + h) * D + hf * (D / 2);
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        float g[32];
        tmem_ld32(tl + kColDV + hf * (D / 2) + 32 * c, g);
        if (key < S) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 v;
            v.x = pack_bf16(g[8 * t + 0], g[8 * t + 1]);
            v.y = pack_bf16(g[8 * t + 2], g[8 * t + 3]);
            v.z = pack_bf16(g[8 * t + 4], g[8 * t + 5]);
            v.w = pack_bf16(g[8 * t + 6], g[8 * t + 7]);
            *reinterpret_cast<uint4*>(dv + off + 32 * c + 8 * t) = v;
          }
        }
        tmem_ld32(tl + kColDK + hf * (D / 2) + 32 * c, g);
        if (key < S) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 v;
            v.x = pack_bf16(g[8 * t + 0] * scale, g[8 * t + 1] * scale);
            v.y = pack_bf16(g[8 * t + 2] * scale, g[8 * t + 3] * scale);
            v.z = pack_bf16(g[8 * t + 4] * scale, g[8 * t + 5] * scale);
            v.w = pack_bf16(g[8 * t + 6] * scale, g[8 * t + 7] * scale);
            *reinterpret_cast<uint4*>(dk + off + 32 * c + 8 * t) = v;
          }
        }
      }
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp && lane == 0 && mma_issued) {
    mma_commit(&ctl->bar_final);
    settle(&ctl->bar_final, 0, ctx);
  }
  if (warp == kProducerWarp && lane == 0) {
    if (kv_armed) settle(&ctl->bar_kv, 0, ctx);
    for (int s = 0; s < 2; ++s) {
      if (q_armed[s]) settle(&ctl->bar_q_full[s], (q_armed[s] - 1) & 1, ctx);
      if (do_armed[s]) settle(&ctl->bar_do_full[s], (do_armed[s] - 1) & 1, ctx);
    }
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int grid_cap(size_t work, int per_block) {
  int dev = 0, sms = 148;
  if (cudaGetDevice(&dev) == cudaSuccess) cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const size_t need = (work + per_block - 1) / per_block;
  const size_t cap = (size_t)sms * 8;
  return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

template <int D, bool kMask>
int launch_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
               const uint8_t* mask, void* dq, void* dk, void* dv, int B, int S, int H, float scale, float* delta,
               float* acc, cudaStream_t stream, const DevCtx& ctx) {
  const size_t rows = (size_t)B * S * H;
  const size_t acc_vec4 = rows * D / 4;
  bwd_preprocess_kernel<D><<<grid_cap(rows * 8, 256), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), delta,
      reinterpret_cast<float4*>(acc), B, S, H, acc_vec4);
  int st = check_launch("uaa_attn_bwd (preprocess)");
  if (st) return st;
  CUtensorMap mq, mk, mv, mdo, macc;
  if ((st = encode_bshd_map(&mq, q, B, S, H, D, 128))) return st;
  if ((st = encode_bshd_map(&mk, k, B, S, H, D, 128))) return st;
  if ((st = encode_bshd_map(&mv, v, B, S, H, D, 128))) return st;
  if ((st = encode_bshd_map(&mdo, dout, B, S, H, D, 128))) return st;
  if ((st = encode_bshd_map_f32(&macc, acc, B, S, H, D, 128))) return st;
  auto kern = attn_bwd_kernel<D, kMask>;
  const int smem = BwdLayout<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "uaa_attn_bwd: smem attribute: %s", cudaGetErrorString(e));
  dim3 grid((S + kBK - 1) / kBK, H, B);
  kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, mdo, macc, lse, delta, mask, static_cast<__nv_bfloat16*>(dk),
                                         static_cast<__nv_bfloat16*>(dv), S, H, scale, scale * kLog2e, ctx);
  if ((st = check_launch("uaa_attn_bwd (main)"))) return st;
  const size_t n8 = rows * D / 8;
  dq_convert_kernel<<<grid_cap(n8, 256), 256, 0, stream>>>(reinterpret_cast<const float4*>(acc),
                                                            static_cast<uint4*>(dq), scale, n8);
  return check_launch("uaa_attn_bwd (dq convert)");
}

size_t delta_bytes(int B, int S, int H) {
  return (((size_t)B * H * S * 4) + 255) & ~(size_t)255;
}

}  // namespace
}  // namespace uaa

using namespace uaa;

extern "C" size_t uaa_attn_bwd_workspace_bytes(int B, int S, int H, int D) {
  if (B < 0 || S < 0 || H < 0 || (D != 64 && D != 128)) return 0;
  return delta_bytes(B, S, H) + (size_t)B * S * H * D * 4;
}

extern "C" int uaa_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                            const float* lse, const uint8_t* key_mask, void* dq, void* dk, void* dv, int B, int S,
                            int H, int D, float scale, void* workspace, size_t workspace_bytes,
                            uaa_stream_t stream) {
  const char* fn = "uaa_attn_bwd";
  int st = validate_attn_sizes(fn, B, S, H, D, scale);
  if (st) return st;
  if ((uint64_t)B * S * H == 0) return UAA_OK;
  if ((st = check_dev_ptr(fn, "q", q)) || (st = check_dev_ptr(fn, "k", k)) || (st = check_dev_ptr(fn, "v", v)) ||
      (st = check_dev_ptr(fn, "out", out)) || (st = check_dev_ptr(fn, "dout", dout)) ||
      (st = check_dev_ptr(fn, "dq", dq)) || (st = check_dev_ptr(fn, "dk", dk)) || (st = check_dev_ptr(fn, "dv", dv)))
    return st;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: lse is NULL or not 4-byte aligned", fn);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace is NULL or not 256-byte aligned", fn);
  const size_t need = uaa_attn_bwd_workspace_bytes(B, S, H, D);
  if (workspace_bytes < need)
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace has %zu bytes, %zu needed", fn, workspace_bytes, need);
  DevCtx ctx;
  if ((st = get_dev_ctx(&ctx))) return st;
  float* delta = static_cast<float*>(workspace);
  float* acc = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) + delta_bytes(B, S, H));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 64)
    return key_mask ? launch_bwd<64, true>(q, k, v, out, dout, lse, key_mask, dq, dk, dv, B, S, H, scale, delta, acc,
                                           s, ctx)
                    : launch_bwd<64, false>(q, k, v, out, dout, lse, key_mask, dq, dk, dv, B, S, H, scale, delta,
                                            acc, s, ctx);
  return key_mask ? launch_bwd<128, true>(q, k, v, out, dout, lse, key_mask, dq, dk, dv, B, S, H, scale, delta, acc,
                                          s, ctx)
                  : launch_bwd<128, false>(q, k, v, out, dout, lse, key_mask, dq, dk, dv, B, S, H, scale, delta, acc,
                                           s, ctx);
}

// ---------------------------------------------------------------------------
// Allocation-free variant of the backward.
//
// Some callers cannot call cudaMalloc at the point where they run the backward:
// code inside a custom allocator callback, a plugin that may only launch work
// on a stream it was handed, a runtime that has pre-planned every device
// allocation and forbids new ones, or a latency-bound loop that must not take
// the allocator's locks.  They cannot size and hand over the workspace that
// uaa_attn_bwd asks for, so this entry point uses a fixed scratch array that
// lives in the library itself.
//
// The array is a file-scope device variable: every GPU that loads the library
// holds kNoAllocScratchBytes of it until the process exits.  Host code cannot
// use the array's name as a device address, so the first call on each device
// looks the address up (cudaGetSymbolAddress, with that device current) and
// caches it; make that first call before any stream capture begins.  All calls
// share the one array: two calls whose kernels overlap on the GPU (different
// streams, no ordering between them) race on it and give wrong results.
// Nothing in the array needs to start at zero: the Delta part is fully written
// and the dQ accumulator is zeroed by the preprocess kernel of every call.
namespace uaa {
namespace {

constexpr size_t kNoAllocScratchBytes = 64ull << 20;  // 64 MiB
__device__ __align__(256) uint8_t g_bwd_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {nullptr};

int scratch_address(void** out) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= 64) return set_error(UAA_ERR_CUDA, "device index %d out of range", dev);
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (!g_scratch_addr[dev]) {
    void* p = nullptr;
    e = cudaGetSymbolAddress(&p, g_bwd_scratch);
    if (e != cudaSuccess)
      return set_error(UAA_ERR_CUDA, "cudaGetSymbolAddress(backward scratch): %s", cudaGetErrorString(e));
    g_scratch_addr[dev] = p;
  }
  *out = g_scratch_addr[dev];
  return UAA_OK;
}

}  // namespace
}  // namespace uaa

extern "C" size_t uaa_attn_bwd_noalloc_max_bytes(void) { return uaa::kNoAllocScratchBytes; }

extern "C" int uaa_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                    const float* lse, const uint8_t* key_mask, void* dq, void* dk, void* dv, int B,
                                    int S, int H, int D, float scale, uaa_stream_t stream) {
  const char* fn = "uaa_attn_bwd_noalloc";
  int st = validate_attn_sizes(fn, B, S, H, D, scale);
  if (st) return st;
  if ((uint64_t)B * S * H == 0) return UAA_OK;
  const size_t need = uaa_attn_bwd_workspace_bytes(B, S, H, D);
  if (need > kNoAllocScratchBytes)
    return set_error(UAA_ERR_UNSUPPORTED,
                     "%s: B*S*H*D too large for the built-in scratch (%zu bytes needed, %zu available); "
                     "use uaa_attn_bwd with a caller-provided workspace",
                     fn, need, kNoAllocScratchBytes);
  void* scratch = nullptr;
  if ((st = scratch_address(&scratch))) return st;
  return uaa_attn_bwd(q, k, v, out, dout, lse, key_mask, dq, dk, dv, B, S, H, D, scale, scratch, need, stream);
}
