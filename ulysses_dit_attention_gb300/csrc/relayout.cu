// Ulysses re-layout kernels on one device: the forward exchange (sequence
// shards -> head groups), its inverse (head groups -> sequence shards, padding
// rows zeroed) and the trim-before-concat key-mask assembly.
//
// "[attention] Add Ulysses Anything backward", What does this PR do: the
// exchange reuses all-to-all helpers with saved query/key partition metadata,
// supports uneven shards, and the gathered key-mask shards are trimmed to their
// true lengths before concatenation.  "Add fast-ulysses attention backend",
// Summary / Performance: the exchange around the attention module is the part
// whose speed matters (7518 us -> 6762 us per layer on 4 H800s).
//
// These kernels are HBM-bound copies: one warp per output row, 16-byte vector
// loads and stores, each lane moving kUnroll vectors per loop trip with all
// loads issued before the stores, and a grid of a multiple of the SM count.  Algorithmic bytes = one
// read + one write of every valid element (+ one write of every padding
// element in the inverse).
#include "uaa_common.cuh"

namespace uaa {
namespace {

constexpr int kMaxShards = 64;
constexpr int kThreads = 256;
constexpr int kUnroll = 4;

struct Partition {
  int P;
  int cap;
  int offs[kMaxShards + 1];  // prefix sums of the shard lengths
};

__device__ __forceinline__ int find_shard(const Partition& part, int n) {
  int p = 0;
#pragma unroll 1
  while (p + 1 < part.P && n >= part.offs[p + 1]) ++p;
  return p;
}

// One warp copies a run of n 16-byte vectors (or writes n zero vectors when src is
// null), each lane moving up to kUnroll vectors per trip with all loads issued first.
__device__ __forceinline__ void copy_run(const uint4* __restrict__ src, uint4* __restrict__ dst, int n, int lane) {
  for (int v0 = lane; v0 < n; v0 += 32 * kUnroll) {
    uint4 v[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int i = v0 + 32 * u;
      v[u] = make_uint4(0u, 0u, 0u, 0u);
      if (src && i < n) v[u] = __ldcs(src + i);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u)
      if (v0 + 32 * u < n) __stcs(dst + v0 + 32 * u, v[u]);
  }
}

// y[g, b, n, h', :] = x[p, b, s, g*Hg + h', :] with n = offs[p] + s, and 0 for
// the padding heads g*Hg + h' >= H (Hg = ceil(H/P)).
// One warp per output row (g, b, n): the row's Hg*rowvec vectors are one
// contiguous run of the source row as well, so the index arithmetic (two
// divisions and the shard search) is paid once per row, not per vector.
__global__ void __launch_bounds__(kThreads) seq_to_head_kernel(const uint4* __restrict__ x, uint4* __restrict__ y,
                                                               const __grid_constant__ Partition part, int B,
                                                               int H, int Hg, int rowvec, uint32_t rows) {
  const int N = part.offs[part.P];
  const int run = Hg * rowvec;
  const int lane = threadIdx.x & 31;
  const uint32_t warps = gridDim.x * (blockDim.x >> 5);
  for (uint32_t r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const int n = (int)(r % (uint32_t)N);
    const uint32_t gb = r / (uint32_t)N;
    const int b = (int)(gb % (uint32_t)B);
    const int g = (int)(gb / (uint32_t)B);
    const int p = find_shard(part, n);
    const int s = n - part.offs[p];
    const int heads = H - g * Hg < Hg ? H - g * Hg : Hg;  // real heads of this group (may be <= 0)
    const int real = heads > 0 ? heads * rowvec : 0;
    uint4* dst = y + (size_t)r * run;
    const uint4* src = x + (((size_t)p * B + b) * part.cap + s) * (size_t)H * rowvec + (size_t)g * run;
    copy_run(src, dst, real, lane);
    copy_run(nullptr, dst + real, run - real, lane);
  }
}

// x[p, b, s, h, :] = y[h / Hg, b, offs[p] + s, h % Hg, :] for s < L_p, else 0
// (h < H only: the padding heads of the groups are dropped).
// One warp per output row (p, b, s): the row is P contiguous runs, one per head
// group, each a contiguous run of that group's row n = offs[p] + s.
__global__ void __launch_bounds__(kThreads) head_to_seq_kernel(const uint4* __restrict__ y, uint4* __restrict__ x,
                                                               const __grid_constant__ Partition part, int B,
                                                               int H, int Hg, int rowvec, uint32_t rows) {
  const int N = part.offs[part.P];
  const int rowlen = H * rowvec;
  const int lane = threadIdx.x & 31;
  const uint32_t warps = gridDim.x * (blockDim.x >> 5);
  for (uint32_t r = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows; r += warps) {
    const int s = (int)(r % (uint32_t)part.cap);
    const uint32_t pb = r / (uint32_t)part.cap;
    const int b = (int)(pb % (uint32_t)B);
    const int p = (int)(pb / (uint32_t)B);
    uint4* dst = x + (size_t)r * rowlen;
    if (s >= part.offs[p + 1] - part.offs[p]) {  // transport padding
      copy_run(nullptr, dst, rowlen, lane);
      continue;
    }
    const int n = part.offs[p] + s;
#pragma unroll 1
    for (int g = 0; g * Hg < H; ++g) {
      const int heads = H - g * Hg < Hg ? H - g * Hg : Hg;
      const uint4* src = y + (((size_t)g * B + b) * N + n) * (size_t)Hg * rowvec;
      copy_run(src, dst + (size_t)g * Hg * rowvec, heads * rowvec, lane);
    }
  }
}

// mask[b, offs[p] + s] = gathered[p, b, s] for s < L_p (each shard trimmed
// before concatenation).  One thread per output byte.
__global__ void __launch_bounds__(kThreads) assemble_key_mask_kernel(const uint8_t* __restrict__ gathered,
                                                                     uint8_t* __restrict__ mask,
                                                                     const __grid_constant__ Partition part,
                                                                     int B, uint32_t total) {
  const int N = part.offs[part.P];
  for (uint32_t idx = blockIdx.x * blockDim.x + threadIdx.x; idx < total; idx += gridDim.x * blockDim.x) {
    const int n = (int)(idx % (uint32_t)N);
    const int b = (int)(idx / (uint32_t)N);
    const int p = find_shard(part, n);
    const int s = n - part.offs[p];
    mask[idx] = gathered[((size_t)p * B + b) * part.cap + s];
  }
}

// x[z, s, :] = 0 for the padding rows len[p] <= s < cap of every slab z = p*B + b of a
// (nseg*B, cap, H, D) bf16 buffer; one thread per 16-byte vector.
__global__ void __launch_bounds__(kThreads) zero_pad_kernel(uint4* __restrict__ x, const __grid_constant__ SeqDesc d, int B,
                                                            int rowvec, int maxpad, uint64_t total) {
  const uint64_t per_slab = (uint64_t)maxpad * rowvec;
  for (uint64_t idx = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; idx < total;
       idx += (uint64_t)gridDim.x * blockDim.x) {
    const uint64_t z = idx / per_slab;
    const uint64_t i = idx - z * per_slab;
    const int p = (int)(z / (uint64_t)B);
    if (i < (uint64_t)(d.cap - d.len[p]) * rowvec)
      x[(z * d.cap + d.len[p]) * rowvec + i] = make_uint4(0u, 0u, 0u, 0u);
  }
}

int sm_count() {
  // per device: the attribute query is cheap, and a process may drive GPUs of different sizes
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess || n <= 0)
    return 148;
  return n;
}

int grid_for(uint64_t work_items, int items_per_thread) {
  // a multiple of the SM count (8 resident 256-thread CTAs per SM), capped by the work
  const uint64_t needed = (work_items + (uint64_t)kThreads * items_per_thread - 1) / ((uint64_t)kThreads * items_per_thread);
  const uint64_t cap = (uint64_t)sm_count() * 8;
  uint64_t g = needed < cap ? needed : cap;
  return g < 1 ? 1 : (int)g;
}

int build_partition(const char* fn, Partition* part, int P, const int* shard_lens, int cap) {
  if (P < 1 || P > kMaxShards) return set_error(UAA_ERR_INVALID_ARG, "%s: P=%d must be in [1, %d]", fn, P, kMaxShards);
  if (!shard_lens) return set_error(UAA_ERR_INVALID_ARG, "%s: shard_lens is NULL", fn);
  if (cap < 0) return set_error(UAA_ERR_INVALID_ARG, "%s: cap=%d is negative", fn, cap);
  part->P = P;
  part->cap = cap;
  part->offs[0] = 0;
  for (int p = 0; p < P; ++p) {
    const int L = shard_lens[p];
    if (L < 0 || L > cap)
      return set_error(UAA_ERR_INVALID_ARG, "%s: shard_lens[%d]=%d outside [0, cap=%d]", fn, p, L, cap);
    if ((int64_t)part->offs[p] + L > INT32_MAX) return set_error(UAA_ERR_INVALID_ARG, "%s: total length overflows", fn);
    part->offs[p + 1] = part->offs[p] + L;
  }
  return UAA_OK;
}

int check_ptr(const char* fn, const char* name, const void* p, size_t align) {
  if (!p) return set_error(UAA_ERR_INVALID_ARG, "%s: %s is NULL", fn, name);
  if (reinterpret_cast<uintptr_t>(p) % align)
    return set_error(UAA_ERR_INVALID_ARG, "%s: %s is not %zu-byte aligned", fn, name, align);
  return UAA_OK;
}

int relayout_common(const char* fn, const void* src, const void* dst, int P, const int* shard_lens, int cap, int B,
                    int H, int D, int elem_bytes, Partition* part, int* rowvec, int* Hg) {
  int st = build_partition(fn, part, P, shard_lens, cap);
  if (st) return st;
  if (B < 0 || H < 1 || D < 1) return set_error(UAA_ERR_INVALID_ARG, "%s: bad sizes B=%d H=%d D=%d", fn, B, H, D);
  if (elem_bytes != 1 && elem_bytes != 2 && elem_bytes != 4 && elem_bytes != 8)
    return set_error(UAA_ERR_INVALID_ARG, "%s: elem_bytes=%d must be 1, 2, 4 or 8", fn, elem_bytes);
  if (((int64_t)D * elem_bytes) % 16)
    return set_error(UAA_ERR_INVALID_ARG, "%s: D*elem_bytes=%lld is not a multiple of 16", fn,
                     (long long)D * elem_bytes);
  *rowvec = (int)((int64_t)D * elem_bytes / 16);
  *Hg = (H + P - 1) / P;  // P does not have to divide H: the groups are padded with zero heads
  const uint64_t big =
      (uint64_t)P * B * (uint64_t)(cap > part->offs[P] ? cap : part->offs[P]) * ((uint64_t)P * (*Hg)) * (*rowvec);
  if (big >= (1ull << 31)) return set_error(UAA_ERR_UNSUPPORTED, "%s: tensor too large (>= 2^31 16-byte vectors)", fn);
  if (B == 0) return UAA_OK;
  if ((st = check_ptr(fn, "src", src, 16))) return st;
  if ((st = check_ptr(fn, "dst", dst, 16))) return st;
  return UAA_OK;
}

}  // namespace

int zero_pad_rows(void* x, const SeqDesc& d, int B, int H, int D, cudaStream_t stream) {
  int maxpad = 0;
  for (int p = 0; p < d.nseg; ++p) maxpad = d.cap - d.len[p] > maxpad ? d.cap - d.len[p] : maxpad;
  if (maxpad == 0 || B == 0 || H == 0) return UAA_OK;
  const int rowvec = H * D * 2 / 16;
  const uint64_t total = (uint64_t)d.nseg * B * maxpad * rowvec;
  zero_pad_kernel<<<grid_for(total, 1), kThreads, 0, stream>>>(static_cast<uint4*>(x), d, B, rowvec, maxpad, total);
  return check_launch("zero_pad_rows");
}

}  // namespace uaa

using namespace uaa;

extern "C" {

int uaa_seq_to_head(const void* x, void* y, int P, const int* shard_lens, int cap, int B, int H, int D,
                    int elem_bytes, uaa_stream_t stream) {
  Partition part;
  int rowvec = 0, Hg = 0;
  int st = relayout_common("uaa_seq_to_head", x, y, P, shard_lens, cap, B, H, D, elem_bytes, &part, &rowvec, &Hg);
  if (st) return st;
  const uint32_t rows = (uint32_t)((uint64_t)P * B * part.offs[P]);
  if (rows == 0) return UAA_OK;
  seq_to_head_kernel<<<grid_for((uint64_t)rows * 32, 1), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(x), static_cast<uint4*>(y), part, B, H, Hg, rowvec, rows);
  return check_launch("uaa_seq_to_head");
}

int uaa_head_to_seq(const void* y, void* x, int P, const int* shard_lens, int cap, int B, int H, int D,
                    int elem_bytes, uaa_stream_t stream) {
  Partition part;
  int rowvec = 0, Hg = 0;
  int st = relayout_common("uaa_head_to_seq", y, x, P, shard_lens, cap, B, H, D, elem_bytes, &part, &rowvec, &Hg);
  if (st) return st;
  const uint32_t rows = (uint32_t)((uint64_t)P * B * cap);
  if (rows == 0 || H == 0) return UAA_OK;
  head_to_seq_kernel<<<grid_for((uint64_t)rows * 32, 1), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<const uint4*>(y), static_cast<uint4*>(x), part, B, H, Hg, rowvec, rows);
  return check_launch("uaa_head_to_seq");
}

int uaa_assemble_key_mask(const uint8_t* gathered, uint8_t* mask, int P, const int* shard_lens, int cap, int B,
                          uaa_stream_t stream) {
  const char* fn = "uaa_assemble_key_mask";
  Partition part;
  int st = build_partition(fn, &part, P, shard_lens, cap);
  if (st) return st;
  if (B < 0) return set_error(UAA_ERR_INVALID_ARG, "%s: B=%d is negative", fn, B);
  const uint64_t total = (uint64_t)B * part.offs[P];
  if ((uint64_t)P * B * cap >= (1ull << 31) || total >= (1ull << 31))
    return set_error(UAA_ERR_UNSUPPORTED, "%s: mask too large", fn);
  if (total == 0) return UAA_OK;
  if (!gathered || !mask) return set_error(UAA_ERR_INVALID_ARG, "%s: NULL pointer", fn);
  assemble_key_mask_kernel<<<grid_for(total, 1), kThreads, 0, static_cast<cudaStream_t>(stream)>>>(
      gathered, mask, part, B, (uint32_t)total);
  return check_launch(fn);
}

}  // extern "C"
