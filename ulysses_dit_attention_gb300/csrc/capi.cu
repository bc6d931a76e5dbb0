// Host side of the C ABI that is shared by every kernel family: the per-thread
// last-error message, the per-device status word (the target of the kernels'
// bounded-wait watchdog), the wait bound, TMA tensor-map encoding for BSHD
// tensors, and the watchdog self-test kernel.
#include <atomic>
#include <cstdarg>
#include <cstdint>
#include <cstdio>
#include <mutex>

#include "uaa_common.cuh"

namespace uaa {

namespace {

thread_local char g_last_error[512] = "";

// The status words of a device: sticky status bits, epoch of the last call that
// gave up, and (debug builds) the first failed range check and its value; a
// file-scope device variable of this translation unit.  Its device address is
// looked up once per device.
__device__ unsigned int g_status_word[4];

constexpr int kMaxDevices = 64;
std::mutex g_dev_mu;
unsigned int* g_status_addr[kMaxDevices] = {nullptr};

constexpr unsigned long long kDefaultTimeoutNs = 4000ull * 1000ull * 1000ull;
std::atomic<unsigned long long> g_timeout_ns{kDefaultTimeoutNs};
// Call epochs: every get_dev_ctx() (one per C-ABI call) takes the next one; 0 is never used.
std::atomic<unsigned int> g_epoch{0};
// Diagnostic: the ring load that the attention kernels' producers skip (-1: none).
std::atomic<int> g_drop_load{-1};

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;
std::once_flag g_encode_once;

}  // namespace

int set_error(int status, const char* fmt, ...) {
  va_list ap;
  va_start(ap, fmt);
  vsnprintf(g_last_error, sizeof(g_last_error), fmt, ap);
  va_end(ap);
  return status;
}

int check_launch(const char* what) {
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "%s: launch failed: %s", what, cudaGetErrorString(e));
  return UAA_OK;
}

int get_dev_ctx(DevCtx* ctx) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
  if (dev < 0 || dev >= kMaxDevices) return set_error(UAA_ERR_CUDA, "device index %d out of range", dev);
  {
    std::lock_guard<std::mutex> lk(g_dev_mu);
    if (!g_status_addr[dev]) {
      void* p = nullptr;
      e = cudaGetSymbolAddress(&p, g_status_word);
      if (e != cudaSuccess)
        return set_error(UAA_ERR_CUDA, "cudaGetSymbolAddress(status word): %s", cudaGetErrorString(e));
      g_status_addr[dev] = static_cast<unsigned int*>(p);
    }
    ctx->status = g_status_addr[dev];
  }
  ctx->timeout_ns = g_timeout_ns.load();
  // teardown waits only wait for copies and MMAs already issued: never shorter than the default
  ctx->settle_ns = ctx->timeout_ns > kDefaultTimeoutNs ? ctx->timeout_ns : kDefaultTimeoutNs;
  unsigned int ep = ++g_epoch;
  if (ep == 0) ep = ++g_epoch;
  ctx->epoch = ep;
  ctx->drop_load = g_drop_load.load();
  return UAA_OK;
}

// The driver's tensor-map encoder, resolved once through the runtime.
static PFN_cuTensorMapEncodeTiled_v12000 encoder() {
  std::call_once(g_encode_once, [] {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  });
  return g_encode;
}

SeqDesc seq_plain(int S) {
  SeqDesc d{};
  d.nseg = 1;
  d.cap = S;
  d.total = S;
  d.len[0] = S;
  d.off[0] = 0;
  d.tile0[0] = 0;
  d.tile0[1] = (S + 127) / 128;
  return d;
}

int seq_sharded(SeqDesc* d, int P, const int* lens, int cap, const char* fn) {
  if (P < 1 || P > kMaxSeg)
    return set_error(UAA_ERR_UNSUPPORTED, "%s: P=%d shards (the fused path takes 1..%d)", fn, P, kMaxSeg);
  if (!lens) return set_error(UAA_ERR_INVALID_ARG, "%s: shard_lens is NULL", fn);
  if (cap < 1) return set_error(UAA_ERR_INVALID_ARG, "%s: cap=%d", fn, cap);
  *d = SeqDesc{};
  d->nseg = P;
  d->cap = cap;
  long long total = 0, tiles = 0;
  for (int p = 0; p < P; ++p) {
    if (lens[p] < 0 || lens[p] > cap)
      return set_error(UAA_ERR_INVALID_ARG, "%s: shard %d has %d rows (cap %d)", fn, p, lens[p], cap);
    d->len[p] = lens[p];
    d->off[p] = (int)total;
    d->tile0[p] = (int)tiles;
    total += lens[p];
    tiles += (lens[p] + 127) / 128;
  }
  if (total > INT32_MAX / 2) return set_error(UAA_ERR_UNSUPPORTED, "%s: sequence too long", fn);
  d->total = (int)total;
  d->tile0[P] = (int)tiles;
  return UAA_OK;
}

int encode_seq_maps(SegMaps* maps, const void* ptr, const SeqDesc& d, int B, int H, int D, int box_rows) {
  if (!encoder()) return set_error(UAA_ERR_CUDA, "cuTensorMapEncodeTiled is not available from the driver");
  *maps = SegMaps{};
  for (int p = 0; p < d.nseg; ++p) {
    // segment p: rows [0, len) of slabs p*B .. p*B+B-1; an empty segment gets a one-row map
    // that no tile reads
    const char* base = static_cast<const char*>(ptr) + (size_t)p * B * d.cap * H * D * 2;
    const int rows = d.len[p] > 0 ? d.len[p] : 1;
    cuuint64_t dims[4] = {(cuuint64_t)D, (cuuint64_t)H, (cuuint64_t)rows, (cuuint64_t)B};
    cuuint64_t strides[3] = {(cuuint64_t)D * 2, (cuuint64_t)H * D * 2, (cuuint64_t)d.cap * H * D * 2};
    cuuint32_t box[4] = {64, 1, (cuuint32_t)box_rows, 1};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    CUresult r = g_encode(&maps->m[p], CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<char*>(base), dims, strides,
                          box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS)
      return set_error(UAA_ERR_CUDA, "cuTensorMapEncodeTiled failed for segment %d (CUresult %d)", p, (int)r);
  }
  return UAA_OK;
}

// exp2_fma2 (the forward's FMA-pipe exponential) over x[0 .. 2*npairs), pair by pair.
__global__ void exp2_fma2_kernel(const float2* __restrict__ x, float2* __restrict__ y, long long npairs) {
  for (long long i = (long long)blockIdx.x * blockDim.x + threadIdx.x; i < npairs;
       i += (long long)gridDim.x * blockDim.x)
    y[i] = exp2_fma2(x[i]);
}

// One thread waits on an mbarrier that nothing arrives on; the bounded wait
// runs out and records a timeout.  No copy or tensor-core work is issued.
__global__ void watchdog_selftest_kernel(DevCtx ctx) {
  __shared__ __align__(8) uint64_t bar;
  if (threadIdx.x == 0) {
    mbar_init(&bar, 1);
    fence_mbar_init();
    if (!mbar_wait(&bar, 0, ctx.timeout_ns)) atomicOr(ctx.status, kStatusTimeout);
  }
}

}  // namespace uaa

using namespace uaa;

extern "C" {

const char* uaa_last_error(void) { return g_last_error; }

#ifdef UAA_DEBUG
const char* uaa_version(void) { return "uaa 0.1 sm_103a (debug: device range checks)"; }
int uaa_debug_build(void) { return 1; }
#else
const char* uaa_version(void) { return "uaa 0.1 sm_103a"; }
int uaa_debug_build(void) { return 0; }
#endif

void uaa_set_wait_timeout_ms(unsigned int ms) {
  g_timeout_ns.store(ms ? (unsigned long long)ms * 1000ull * 1000ull : kDefaultTimeoutNs);
}

void uaa_debug_drop_load(int n) { g_drop_load.store(n < 0 ? -1 : n); }

int uaa_check_device_status(uaa_stream_t stream) {
  DevCtx ctx;
  int st = get_dev_ctx(&ctx);
  if (st != UAA_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  cudaError_t e = cudaStreamSynchronize(s);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "stream synchronize: %s", cudaGetErrorString(e));
  // [0] the sticky bits; [1] the abort epoch, which needs no clearing (an epoch recurs only
  // after 2^32 calls); [2], [3] the first failed debug check (rewritten by the next first one)
  unsigned int words[4] = {0u, 0u, 0u, 0u};
  e = cudaMemcpy(words, ctx.status, sizeof(words), cudaMemcpyDeviceToHost);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "status read: %s", cudaGetErrorString(e));
  const unsigned int word = words[0];
  if (word) {
    e = cudaMemset(ctx.status, 0, sizeof(unsigned int));
    if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "status clear: %s", cudaGetErrorString(e));
    e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "status clear sync: %s", cudaGetErrorString(e));
  }
  if (word & kStatusTimeout)
    return set_error(UAA_ERR_TIMEOUT, "a bounded device-side wait ran out (status word 0x%x)", word);
  if (word & kStatusBadLaunch)
    return set_error(UAA_ERR_CUDA, "a kernel refused its launch configuration (status word 0x%x)", word);
  if (word & kStatusDebugCheck) {
    static const char* what[4] = {"?", "MMA shared-memory operand outside the CTA's shared memory",
                                  "MMA TMEM address outside the CTA's allocation", "output store past the tensor end"};
    return set_error(UAA_ERR_DEBUG_CHECK, "a device range check failed and its access was skipped: %s (value 0x%x)",
                     what[words[2] < 4 ? words[2] : 0], words[3]);
  }
  return UAA_OK;
}

int uaa_watchdog_selftest(unsigned int timeout_us, uaa_stream_t stream) {
  if (timeout_us < 1 || timeout_us > 1000000)
    return set_error(UAA_ERR_INVALID_ARG, "uaa_watchdog_selftest: timeout_us must be in [1, 1000000]");
  DevCtx ctx;
  int st = get_dev_ctx(&ctx);
  if (st != UAA_OK) return st;
  ctx.timeout_ns = (unsigned long long)timeout_us * 1000ull;
  watchdog_selftest_kernel<<<1, 32, 0, static_cast<cudaStream_t>(stream)>>>(ctx);
  return check_launch("uaa_watchdog_selftest");
}

int uaa_debug_exp2_fma2(const float* x, float* y, long long n, uaa_stream_t stream) {
  if (n < 0 || (n & 1)) return set_error(UAA_ERR_INVALID_ARG, "uaa_debug_exp2_fma2: n must be even and >= 0");
  if (n == 0) return UAA_OK;
  if (!x || !y || (reinterpret_cast<uintptr_t>(x) & 7u) || (reinterpret_cast<uintptr_t>(y) & 7u))
    return set_error(UAA_ERR_INVALID_ARG, "uaa_debug_exp2_fma2: x and y must be 8-byte aligned device arrays");
  int dev = 0, sms = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e == cudaSuccess) e = cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "uaa_debug_exp2_fma2: %s", cudaGetErrorString(e));
  const long long pairs = n / 2, blocks = (pairs + 255) / 256, cap = (long long)sms * 8;
  exp2_fma2_kernel<<<(int)(blocks < cap ? blocks : cap), 256, 0, static_cast<cudaStream_t>(stream)>>>(
      reinterpret_cast<const float2*>(x), reinterpret_cast<float2*>(y), pairs);
  return check_launch("uaa_debug_exp2_fma2");
}

}  // extern "C"
