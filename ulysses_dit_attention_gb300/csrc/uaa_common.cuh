// Shared device/host helpers of the sm_103a kernels: inline-PTX wrappers for
// mbarriers, TMA tensor loads, tcgen05 (TMEM allocation, MMA, commit, TMEM
// loads/stores) and the UMMA shared-memory / instruction descriptors, plus the
// host-side launch context (status word, wait bound, last-error message).
#pragma once

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/uaa.h"

namespace uaa {

// ----------------------------------------------------------------------------
// Status word bits written by kernels (OR-ed into a device word that
// uaa_check_device_status() reads and clears).
// ----------------------------------------------------------------------------
enum : uint32_t {
  kStatusTimeout = 1u,      // a bounded wait ran out
  kStatusBadLaunch = 2u,    // a kernel refused its launch configuration (e.g. misaligned shared memory)
  kStatusDebugCheck = 4u,   // debug builds (UAA_DEBUG): a device-side range check failed, the access was skipped
};
// Debug builds leave the first failed check in status[2] (kDbg* below) and its
// offending value in status[3].
enum : uint32_t {
  kDbgSmemOperand = 1u,  // an MMA shared-memory descriptor starts outside this CTA's dynamic shared memory
  kDbgTmemAddress = 2u,  // an MMA accumulator / TMEM operand lies outside the CTA's TMEM allocation
  kDbgGlobalStore = 3u,  // an output store lies past the end of its tensor
};

// Launch context handed to every kernel.  status[0] holds the sticky status
// bits above (reported and cleared by uaa_check_device_status); status[1] holds
// the epoch of the last call whose kernels gave up.  Every C-ABI call gets a new
// epoch, so a timeout makes the other CTAs and kernels of the same call stop
// waiting, while later calls -- whose epochs differ -- run normally even before
// the status has been read.
struct DevCtx {
  unsigned int* status;           // two words of the current device: status bits, abort epoch
  unsigned long long timeout_ns;  // bound of every wait for another role's progress
  unsigned long long settle_ns;   // bound of the teardown waits for copies / MMAs already in flight
  unsigned int epoch;             // this call's epoch (never 0)
  int drop_load;                  // diagnostic: the ring load each producer skips (-1: none)
};

// Host side: per-device status word address, wait bound, error message.
int get_dev_ctx(DevCtx* ctx);           // returns UAA_OK or UAA_ERR_CUDA (message set)
int set_error(int status, const char* fmt, ...);
int check_launch(const char* what);     // cudaGetLastError -> UAA_ERR_CUDA

// ----------------------------------------------------------------------------
// A sequence made of segments.  Segment p holds len[p] rows at rows [0, len[p])
// of slab p*B + b (batch b) of a (nseg*B, cap, H, D) bf16 buffer, and its rows
// follow those of segments 0..p-1 in the sequence: row s of segment p is
// sequence position off[p] + s.  A plain (B, S, H, D) tensor is one segment
// (len = cap = S).  The sequence-sharded inputs of a Ulysses step are P
// segments: shard p holds the positions [off[p], off[p] + len[p]).
// The attention kernels walk it in 128-row tiles that never straddle two
// segments: tile t belongs to segment p with tile0[p] <= t < tile0[p+1] and
// covers its rows (t - tile0[p])*128 .. +127, the last tile of a segment
// being partial.
// ----------------------------------------------------------------------------
constexpr int kMaxSeg = 8;
// With a key mask of at most this many rows, the forward and the dQ kernel skip
// key tiles without an attended key: the counts of such tiles per mask row are
// tabulated in shared memory when the kernel starts (above this many rows every
// tile is visited and masked keys only get P = 0).
constexpr int kMaxCntRows = 256;
struct SeqDesc {
  int nseg;
  int cap;                 // rows per slab
  int total;               // sequence length: sum of len
  int len[kMaxSeg];
  int off[kMaxSeg];
  int tile0[kMaxSeg + 1];  // first 128-row tile of each segment; tile0[nseg] = number of tiles
};
// One tensor map per segment over its (B, len, H, D) rows, 64-column x
// box_rows boxes, 128-byte swizzle: rows past len[p] read as zeros, so padding
// rows of the slab never enter a tile.
struct SegMaps {
  CUtensorMap m[kMaxSeg];
};
// Host: the plain layout (B, S, H, D) as one segment.
SeqDesc seq_plain(int S);
// Host: P segments of the given lengths in slabs of cap rows; UAA_ERR_* on bad input.
int seq_sharded(SeqDesc* d, int P, const int* lens, int cap, const char* fn);
int encode_seq_maps(SegMaps* maps, const void* ptr, const SeqDesc& d, int B, int H, int D, int box_rows);
// Host: write zeros to the padding rows [len[p], cap) of every slab of a (nseg*B, cap, H, D) bf16 buffer.
int zero_pad_rows(void* x, const SeqDesc& d, int B, int H, int D, cudaStream_t stream);

#if defined(__CUDACC__)

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t lane_id() { return threadIdx.x & 31u; }

// One lane of a converged warp is elected (elect.sync over the full mask): true
// in that lane only; its lane index is written to *lane.  Tensor-core issuers use
// it so that the whole warp computes the (uniform) UMMA descriptors and only the
// issue itself is predicated, rather than running the issue code in a
// lane-divergent branch.
__device__ __forceinline__ bool elect_one_sync(uint32_t* lane) {
  uint32_t l, p;
  asm volatile(
      "{\n\t.reg .pred e;\n\t"
      "elect.sync %0|e, 0xffffffff;\n\t"
      "selp.u32 %1, 1, 0, e;\n\t}"
      : "=r"(l), "=r"(p));
  *lane = l;
  return p != 0;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.release.cta.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)),
               "r"(bytes)
               : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.release.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cta.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of parity `parity` to complete.  Returns false if
// it did not complete within timeout_ns (measured with %globaltimer).
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity, unsigned long long timeout_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (globaltimer_ns() - t0 > timeout_ns) return false;
  }
}

// Bounded wait of a kernel role on barrier phase `parity`.  Returns false --
// and the role then leaves its loops -- when the phase did not complete within
// ctx.timeout_ns (the device status records a timeout and this call's epoch is
// published so that every CTA of the call stops waiting), when another role of
// this CTA has already given up (ctl->abort), or when another CTA of the same
// call has (status[1] == epoch).
template <typename Ctl>
__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const DevCtx& ctx, Ctl* ctl) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i)
      if (mbar_try_wait(bar, parity)) return true;
    if (*reinterpret_cast<volatile int*>(&ctl->abort)) return false;
    if (reinterpret_cast<volatile unsigned int*>(ctx.status)[1] == ctx.epoch) {
      *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
      return false;
    }
    if (globaltimer_ns() - t0 > ctx.timeout_ns) {
      atomicOr(ctx.status, kStatusTimeout);
      atomicExch(ctx.status + 1, ctx.epoch);
      *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
      return false;
    }
  }
}

// Teardown wait for work that is already in flight (a TMA copy into this CTA's
// shared memory, the last MMAs before TMEM is released): it ignores the abort
// flags, which only stop waits for other roles, and has its own, longer bound.
__device__ __forceinline__ void settle(uint64_t* bar, uint32_t parity, const DevCtx& ctx) {
  if (!mbar_wait(bar, parity, ctx.settle_ns)) atomicOr(ctx.status, kStatusTimeout);
}

// ---------------------------------------------------------------- TMA
// 4-D tiled tensor load (coordinates innermost first) completing on `bar`.
__device__ __forceinline__ void tma_load_4d(void* smem_dst, const CUtensorMap* map, uint64_t* bar, int c0, int c1,
                                            int c2, int c3) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(smem_dst)),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(smem_u32(bar)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}

// 4-D tiled tensor reduce-add from shared memory into global memory (bulk-group
// completion; out-of-range rows of the box are not written).
__device__ __forceinline__ void tma_reduce_add_4d(const void* smem_src, const CUtensorMap* map, int c0, int c1,
                                                  int c2, int c3) {
  asm volatile(
      "cp.reduce.async.bulk.tensor.4d.global.shared::cta.add.tile.bulk_group"
      " [%0, {%2, %3, %4, %5}], [%1];" ::"l"(reinterpret_cast<uint64_t>(map)),
      "r"(smem_u32(smem_src)), "r"(c0), "r"(c1), "r"(c2), "r"(c3)
      : "memory");
}
// 1-D bulk copy of `bytes` from global to shared memory completing on `bar`
// (both addresses 16-byte aligned, size a multiple of 16).
__device__ __forceinline__ void bulk_load(void* smem_dst, const void* gsrc, uint32_t bytes, uint64_t* bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                   smem_u32(smem_dst)),
               "l"(gsrc), "r"(bytes), "r"(smem_u32(bar))
               : "memory");
}
__device__ __forceinline__ void bulk_commit_group() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
// Wait until every committed bulk group of this thread has finished reading shared memory.
__device__ __forceinline__ void bulk_wait_read_all() {
  asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory");
}
// Wait until every committed bulk group of this thread has completed.
__device__ __forceinline__ void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }

__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(map)) : "memory");
}

// ---------------------------------------------------------------- named barriers
// Hardware CTA barriers 1..15 (0 is __syncthreads).  Whole, converged warps
// take part; `count` is the number of threads (a multiple of 32) per phase.
// The thread that issues tensor-core MMAs synchronises through these rather
// than through an mbarrier: any load it executes (an mbarrier test included)
// is held behind the MMAs it has queued, and the tensor pipe runs dry while
// it waits.  bar.arrive releases and bar.sync acquires, so tcgen05 work fenced
// with tcgen05.fence::before_thread_sync before the arrive is visible to
// tcgen05 work issued after tcgen05.fence::after_thread_sync behind the sync.
__device__ __forceinline__ void named_sync(uint32_t id, uint32_t count) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
__device__ __forceinline__ void named_arrive(uint32_t id, uint32_t count) {
  asm volatile("bar.arrive %0, %1;" ::"r"(id), "r"(count) : "memory");
}

// ---------------------------------------------------------------- tcgen05
// TMEM allocation: warp-wide; writes the allocated base address to smem.
__device__ __forceinline__ void tmem_alloc(uint32_t* smem_dst, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(smem_dst)),
               "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem], bf16 inputs, fp32 accumulate, one CTA.
__device__ __forceinline__ void mma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                         uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// D[tmem] (+)= A[tmem] * B[smem]: A (M x K, bf16) is read from tensor memory,
// one row per lane, two consecutive K elements per 32-bit column.
__device__ __forceinline__ void mma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                            uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

// ----------------------------------------------------------------------------
// Range checks of debug builds (compiled with -DUAA_DEBUG; a separate library).
// Every MMA's operands are checked before it is issued -- shared-memory
// descriptors must start inside this CTA's dynamic shared memory with room for a
// 1 KB swizzle atom, accumulators and TMEM A operands must lie inside the CTA's
// TMEM columns -- and every output store of the attention kernels against the end
// of its tensor.  A failed check skips the access and sets kStatusDebugCheck (the
// first failure also records what and where, see kDbg*).  Release builds compile
// the checks away: the guard structs are empty and every guard is `true`.
// ----------------------------------------------------------------------------
struct MmaGuard {
#ifdef UAA_DEBUG
  unsigned int* status;
  uint32_t smem_lo, smem_hi;  // [first, last + 1) shared-window byte address of the dynamic shared memory
  uint32_t tcol_lo, tcol_hi;  // allocated TMEM columns
#endif
};

__device__ __forceinline__ void dbg_fail(unsigned int* status, uint32_t what, uint32_t value) {
#ifdef UAA_DEBUG
  if (!(atomicOr(status, kStatusDebugCheck) & kStatusDebugCheck)) {
    atomicExch(status + 2, what);
    atomicExch(status + 3, value);
  }
#else
  (void)status;
  (void)what;
  (void)value;
#endif
}

__device__ __forceinline__ MmaGuard mma_guard(const DevCtx& ctx, uint32_t sbase, uint32_t smem_bytes,
                                              uint32_t tmem, uint32_t tcols) {
  MmaGuard g;
#ifdef UAA_DEBUG
  g.status = ctx.status;
  g.smem_lo = sbase;
  g.smem_hi = sbase + smem_bytes;
  g.tcol_lo = tmem & 0xFFFFu;
  g.tcol_hi = (tmem & 0xFFFFu) + tcols;
#else
  (void)ctx;
  (void)sbase;
  (void)smem_bytes;
  (void)tmem;
  (void)tcols;
#endif
  return g;
}

__device__ __forceinline__ bool guard_smem(const MmaGuard& g, uint64_t desc) {
#ifdef UAA_DEBUG
  const uint32_t a = (uint32_t)(desc & 0x3FFFull) << 4;
  if (a < g.smem_lo || a + 1024u > g.smem_hi) {
    dbg_fail(g.status, kDbgSmemOperand, a);
    return false;
  }
#else
  (void)g;
  (void)desc;
#endif
  return true;
}

// ncols TMEM columns from `taddr` (lane field 0: all 128 lanes)
__device__ __forceinline__ bool guard_tmem(const MmaGuard& g, uint32_t taddr, uint32_t ncols) {
#ifdef UAA_DEBUG
  const uint32_t col = taddr & 0xFFFFu;
  if ((taddr >> 16) != 0u || col < g.tcol_lo || col + ncols > g.tcol_hi) {
    dbg_fail(g.status, kDbgTmemAddress, taddr);
    return false;
  }
#else
  (void)g;
  (void)taddr;
  (void)ncols;
#endif
  return true;
}

// The MMAs with their debug checks: M = 128, N = n accumulator columns.
__device__ __forceinline__ void mma_ss_checked(const MmaGuard& g, uint32_t d_tmem, uint64_t adesc, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate, uint32_t n) {
  if (guard_tmem(g, d_tmem, n) && guard_smem(g, adesc) && guard_smem(g, bdesc))
    mma_bf16(d_tmem, adesc, bdesc, idesc, accumulate);
}
// A in TMEM: 128 lanes x 16 bf16 = 8 packed columns
__device__ __forceinline__ void mma_ts_checked(const MmaGuard& g, uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc,
                                               uint32_t idesc, uint32_t accumulate, uint32_t n) {
  if (guard_tmem(g, d_tmem, n) && guard_tmem(g, a_tmem, 8u) && guard_smem(g, bdesc))
    mma_bf16_ts(d_tmem, a_tmem, bdesc, idesc, accumulate);
}

// An output store of `n` elements at element offset `off` of a tensor of `extent` elements.
__device__ __forceinline__ bool guard_store(const DevCtx& ctx, size_t off, size_t n, size_t extent) {
#ifdef UAA_DEBUG
  if (off + n > extent) {
    dbg_fail(ctx.status, kDbgGlobalStore, (uint32_t)(off > 0xFFFFFFFFull ? 0xFFFFFFFFull : off));
    return false;
  }
#else
  (void)ctx;
  (void)off;
  (void)n;
  (void)extent;
#endif
  return true;
}

// Elements of a (nseg*B, cap, H, D) sequence buffer (plain BSHD: B*S*H*D).
__host__ __device__ __forceinline__ size_t seq_extent(const SeqDesc& sd, int B, int H, int D) {
  return (size_t)sd.nseg * B * sd.cap * H * D;
}

// Arrive (once) on `bar` when every tcgen05 operation issued so far by this thread has completed.
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(
                   smem_u32(bar))
               : "memory");
}

// Load 32 consecutive fp32 columns of this thread's TMEM lane and wait for them.
// The load and the wait sit in one asm statement so no use of the registers can
// be scheduled before the wait.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// Load 2 x 32 fp32 columns (at taddr0 and taddr1) of this thread's TMEM lane with a single wait.
__device__ __forceinline__ void tmem_ld32x2(uint32_t taddr0, uint32_t taddr1, float (&v)[64]) {
  uint32_t r[64];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%64];\n\t"
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,"
      "%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
      : "r"(taddr0), "r"(taddr1)
      : "memory");
#pragma unroll
  for (int i = 0; i < 64; ++i) v[i] = __uint_as_float(r[i]);
}

// Load 16 consecutive fp32 columns of this thread's TMEM lane and wait for them.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
      "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- packed fp32 pairs
// Blackwell executes these as one instruction per pair of fp32 values.
__device__ __forceinline__ float2 fma2(float2 a, float2 b, float2 c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)),
        "l"(*reinterpret_cast<uint64_t*>(&c)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 sub2(float2 a, float2 b) {
  uint64_t d;
  asm("sub.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 mul2(float2 a, float2 b) {
  uint64_t d;
  asm("mul.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}
__device__ __forceinline__ float2 add2(float2 a, float2 b) {
  uint64_t d;
  asm("add.rn.f32x2 %0, %1, %2;"
      : "=l"(d)
      : "l"(*reinterpret_cast<uint64_t*>(&a)), "l"(*reinterpret_cast<uint64_t*>(&b)));
  return *reinterpret_cast<float2*>(&d);
}

// 2^x for a pair of x <= 8 (x may be -inf), on the FMA pipe instead of the
// special-function unit.  x is clamped to -127 and split as x = n + f with
// n = rint(x) (adding 1.5 * 2^23 leaves n in the low mantissa bits) and
// |f| <= 1/2; 2^f is a cubic fitted in relative error on [-1/2, 1/2]
// (coefficients from ulysses_dit_attention_gb300/exp2_fit.py, relative error
// below 8e-5 in float32) and 2^n is built in the exponent field, which gives
// exactly 0 for n = -127 (so for -inf).
__device__ __forceinline__ float2 exp2_fma2(float2 x) {
  constexpr float kShift = 12582912.0f;  // 1.5 * 2^23
  constexpr float c0 = 9.999280572e-01f, c1 = 6.932610273e-01f, c2 = 2.426113784e-01f, c3 = 5.517164618e-02f;
  x = make_float2(fmaxf(x.x, -127.f), fmaxf(x.y, -127.f));
  const float2 t = add2(x, make_float2(kShift, kShift));
  const float2 f = sub2(x, sub2(t, make_float2(kShift, kShift)));
  float2 p = fma2(make_float2(c3, c3), f, make_float2(c2, c2));
  p = fma2(p, f, make_float2(c1, c1));
  p = fma2(p, f, make_float2(c0, c0));
  const float2 sc = make_float2(__uint_as_float((__float_as_uint(t.x) << 23) + 0x3f800000u),
                                __uint_as_float((__float_as_uint(t.y) << 23) + 0x3f800000u));
  return mul2(p, sc);
}

__device__ __forceinline__ float max3(float a, float b, float c) {
  float d;
  asm("max.f32 %0, %1, %2, %3;" : "=f"(d) : "f"(a), "f"(b), "f"(c));
  return d;
}

// Store 32 consecutive 32-bit columns (raw bits) of this thread's TMEM lane, then wait for the store.
__device__ __forceinline__ void tmem_st32_bits(uint32_t taddr, const uint32_t (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(v[0]), "r"(v[1]), "r"(v[2]), "r"(v[3]), "r"(v[4]), "r"(v[5]), "r"(v[6]), "r"(v[7]), "r"(v[8]),
      "r"(v[9]), "r"(v[10]), "r"(v[11]), "r"(v[12]), "r"(v[13]), "r"(v[14]), "r"(v[15]), "r"(v[16]),
      "r"(v[17]), "r"(v[18]), "r"(v[19]), "r"(v[20]), "r"(v[21]), "r"(v[22]), "r"(v[23]), "r"(v[24]),
      "r"(v[25]), "r"(v[26]), "r"(v[27]), "r"(v[28]), "r"(v[29]), "r"(v[30]), "r"(v[31])
      : "memory");
}

// Store 32 consecutive fp32 columns of this thread's TMEM lane, then wait for the store.
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
      "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n\t"
      "tcgen05.wait::st.sync.aligned;" ::"r"(taddr),
      "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
      "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
      "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
      "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
      "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
      "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
      "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
      "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
      "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
      "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
      "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// ---------------------------------------------------------------- descriptors
// UMMA shared-memory matrix descriptor for a 128-byte-swizzled operand:
// start address, leading-dimension byte offset (LBO), stride-dimension byte
// offset (SBO), descriptor version 1 (bits 46-47) and swizzle mode 2 =
// 128-byte swizzle (bits 61-63).  Every swizzle atom (8 rows x 128 B) must
// start on a 1024-byte boundary.
//  * K-major operand (rows = M or N, 64 K-elements per 128-byte row): SBO =
//    1024 (next group of 8 rows); LBO unused; a K step of 16 elements inside
//    the 128-byte row adds 32 bytes to the start address.
//  * MN-major operand (rows = K, 64 MN-elements per 128-byte row): LBO = byte
//    distance between 64-element MN chunks, SBO = 1024 (next 8 K rows); a K
//    step of 16 rows adds 2048 bytes.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr & 0x3FFFFu) >> 4);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Descriptor of the same operand advanced by `byte_off` bytes.  Shared-memory
// addresses stay below 256 KB, so the 14-bit start-address field never carries
// into the neighbouring fields and one 32-bit add on the low word suffices; the
// MMA issuer adds a constant per K step instead of re-encoding the descriptor.
__device__ __forceinline__ uint64_t desc_add(uint64_t d, uint32_t byte_off) {
  const uint32_t lo = static_cast<uint32_t>(d) + (byte_off >> 4);
  return (d & 0xFFFFFFFF00000000ull) | lo;
}

#endif  // __CUDACC__

// Instruction descriptor of tcgen05.mma kind::f16 with bf16 A/B and fp32 D:
// bits 4-5 D format (1 = f32), 7-9 A format (1 = bf16), 10-12 B format
// (1 = bf16), 15 A major (1 = MN-major), 16 B major, 17-22 N>>3, 24-28 M>>4.
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int M, int N, bool a_mn_major, bool b_mn_major) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((a_mn_major ? 1u : 0u) << 15) | ((b_mn_major ? 1u : 0u) << 16) |
         (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

constexpr float kLog2e = 1.4426950408889634f;


#if defined(__CUDACC__)
// Segment of 128-row tile t (tile0[p] <= t < tile0[p+1]); t past the last tile maps to the
// last segment, whose rows there read as zeros.
__device__ __forceinline__ int seq_seg_of_tile(const SeqDesc& d, int t) {
  int p = 0;
#pragma unroll 1
  while (p + 1 < d.nseg && t >= d.tile0[p + 1]) ++p;
  return p;
}
// Position of tile t: its segment, its first row within the segment, and the number of
// valid rows (0 past the end of the sequence).
struct SeqTile {
  int seg, row0, valid;
};
__device__ __forceinline__ SeqTile seq_tile(const SeqDesc& d, int t) {
  SeqTile r;
  r.seg = seq_seg_of_tile(d, t);
  r.row0 = (t - d.tile0[r.seg]) * 128;
  const int left = d.len[r.seg] - r.row0;
  r.valid = left < 0 ? 0 : (left < 128 ? left : 128);
  return r;
}
// seq_tile for loops that visit tiles in increasing order.  The cursor keeps the
// current segment's first tile, end and length in registers and reloads them
// from the descriptor only when a visit crosses into a later segment, so a visit
// reads no memory (with one segment: never after the first).
struct SeqCursor {
  int seg = -1, first = 0, next = 0, len = 0;
};
__device__ __forceinline__ SeqTile seq_tile_at(const SeqDesc& d, int t, SeqCursor& c) {
#pragma unroll 1
  while (t >= c.next && c.seg + 1 < d.nseg) {
    ++c.seg;
    c.first = d.tile0[c.seg];
    c.next = d.tile0[c.seg + 1];
    c.len = d.len[c.seg];
  }
  SeqTile r;
  r.seg = c.seg;
  r.row0 = (t - c.first) * 128;
  const int left = c.len - r.row0;
  r.valid = left < 0 ? 0 : (left < 128 ? left : 128);
  return r;
}
// Element offset of (batch b, segment row s of segment p, head h, column 0) in the slab buffer.
__device__ __forceinline__ size_t seq_elem(const SeqDesc& d, int B, int H, int D, int b, int p, int s, int h) {
  return ((((size_t)p * B + b) * d.cap + s) * H + h) * (size_t)D;
}
#endif

}  // namespace uaa
