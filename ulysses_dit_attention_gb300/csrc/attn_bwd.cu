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
// Three kernels, no atomics and no reductions, so every gradient is
// deterministic:
//  1. bwd_preprocess_kernel: Delta_i = sum_d dO_id * O_id (fp32), which equals
//     sum_j P_ij dP_ij, and -LSE_i*log2(e), both into the workspace as (B, H,
//     tiles*128) rows in query-tile order (rows past the end of a segment:
//     Delta = 0, -LSE*log2e = -inf, so they get P = 0), which the dK/dV
//     producer copies into shared memory with one bulk copy per tile.
//  2. attn_bwd_dkdv_kernel (K/V-tile-major): a persistent CTA takes a 128-key
//     tile of one (batch, head) and loops over all 128-row query tiles:
//        S^T  = K Q^T,  P^T = exp2(S^T*c - lse2)            (M = keys)
//        dP^T = V dO^T, dS^T = P^T (dP^T - Delta)
//        dV  += P^T dO, dK += dS^T Q                        (accumulated in TMEM)
//     P^T and dS^T are written back to TMEM as bf16 and read from there as
//     the A operand of the dV / dK MMAs.
//  3. attn_bwd_dq_kernel (Q-tile-major): a persistent CTA takes a 128-row
//     query tile and loops over the key tiles, recomputing S = Q K^T and
//     dP = dO V^T with Q and dO held in TMEM as A operands (so these MMAs
//     read only K / V from shared memory); dS = P (dP - Delta) goes back to
//     TMEM as bf16 and dQ += dS K accumulates in TMEM; dQ is written once,
//     in bf16.  The extra S / dP recomputation (7 GEMMs instead of 5 for the
//     whole backward) buys a reduction-free, deterministic dQ.
// Keys outside the mask get P = 0, hence dK = dV = 0 exactly; key tiles with
// no attended key are skipped (the dK/dV kernel writes zeros for them; the dQ
// kernel, like the forward, walks a per-mask-row count of attended tiles taken
// when it starts, up to 256 mask rows, and visits every tile above that).
//
// Warp roles: warps 0-7 compute (TMEM lane quadrant = warp % 4, column half =
// warp / 4), warp 8 TMA producer; the dK/dV kernel's tcgen05 issuer is warp 9
// (one elected lane), the dQ kernel's are warps 9 and 10 (lane 0 of each).
// MMAs of one thread execute in order, with one measured exception: an MMA
// that takes its A operand from TMEM, issued directly behind such an MMA of
// another GEMM, gave wrong results (dQ_g then dP_{g+1} in the dQ kernel, with
// or without TMEM columns in common), so that pair is separated by a
// completion wait.  Consecutive MMAs of one GEMM, and a shared-memory-operand
// MMA behind a TMEM-operand one, were exact in every run.
//
// Query and key sequences are segmented (SeqDesc): a plain (B, S, H, D)
// tensor is one segment; the sequence shards of a Ulysses step are P segments,
// read and written in place (one TMA tensor map per segment; 128-row tiles
// never straddle two segments, so the last tile of a segment is partial and
// its missing rows read as zeros, with P = 0 for those keys and queries).
#include <math.h>

#include <mutex>

#include "attn_bwd_shared.cuh"

namespace uaa {

int validate_attn_sizes(const char* fn, int B, int Sq, int Sk, int H, int D, float scale);
int check_dev_ptr(const char* fn, const char* name, const void* p);
int launch_bwd_fused(const void* q, const void* k, const void* v, const void* dout, const uint8_t* mask, int mrows,
                     void* dq, void* dk, void* dv, int B, int Sq, int Sk, int H, int D, float scale,
                     const float* delta, const float* nl2, float* dq_acc, cudaStream_t s, const DevCtx& ctx,
                     int (*mark)(int, cudaStream_t));

namespace {

// The dK/dV kernel: warps 0-7 compute, warp 8 TMA producer, warp 9 the tcgen05
// issuer (the dQ kernel has a second issuer, warp 10: kThreads).
constexpr int kSplitThreads = 320;

// ---------------------------------------------------------------------------
// 1. Delta = rowsum(dO * O) and -LSE*log2e per query row.  Eight lanes per
// (b, position, h) row, 16-byte loads.  Stored per (b, h) in query-tile order:
// row r of 128-row tile t of sequence qd at index t*128 + r of a (B, H, tiles*128)
// array, the rows past each segment's end holding Delta = 0 and -inf.
template <int D>
__global__ void __launch_bounds__(256) bwd_preprocess_kernel(const __nv_bfloat16* __restrict__ o,
                                                             const __nv_bfloat16* __restrict__ dout,
                                                             const float* __restrict__ lse,
                                                             float* __restrict__ delta, float* __restrict__ nl2,
                                                             const __grid_constant__ SeqDesc qd, int B, int H) {
  constexpr int kVecPerRow = D / 8;
  constexpr int kPerLane = kVecPerRow / 8;
  const int S = qd.total;
  const int S_pad = qd.tile0[qd.nseg] * 128;
  const size_t rows = (size_t)B * S * H;
  const size_t tid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
  const size_t nthreads = (size_t)gridDim.x * blockDim.x;
  const int sub = threadIdx.x & 7;
  for (size_t r = tid >> 3; r < ((rows + 3) / 4) * 4; r += nthreads >> 3) {
    // r = (b * S + n) * H + h, n a sequence position: row n - off[p] of segment p
    const int h = (int)(r % H);
    const size_t bn = r / H;
    const int n = (int)(bn % S);
    const int b = (int)(bn / S);
    int p = 0;
    if (r < rows)
      while (p + 1 < qd.nseg && n >= qd.off[p + 1]) ++p;
    const int sp = n - qd.off[p];
    float acc = 0.f;
    if (r < rows) {
      const size_t e0 = seq_elem(qd, B, H, D, b, p, sp, h);
      const uint4* po = reinterpret_cast<const uint4*>(o + e0);
      const uint4* pd = reinterpret_cast<const uint4*>(dout + e0);
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
      const float l = lse[((size_t)b * H + h) * S + n];
      const size_t w = ((size_t)b * H + h) * S_pad + (size_t)(qd.tile0[p] * 128 + sp);
      delta[w] = acc;
      nl2[w] = l == -INFINITY ? -INFINITY : -l * kLog2e;
    }
  }
  // the rows past each segment's end in its last tile, for every (b, h)
  for (size_t i = tid; i < (size_t)B * H * S_pad; i += nthreads) {
    const int row = (int)(i % S_pad);
    const int t = row >> 7;
    int p = 0;
    while (p + 1 < qd.nseg && t >= qd.tile0[p + 1]) ++p;
    if ((t - qd.tile0[p]) * 128 + (row & 127) >= qd.len[p]) {
      delta[i] = 0.f;
      nl2[i] = -INFINITY;
    }
  }
}


// ---------------------------------------------------------------------------
// 2. dK / dV (K/V-tile-major)
template <int D>
struct DkdvLayout {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQStages = 3;                   // Q_i (+ Delta_i): last read by dK_i
  static constexpr int kDStages = 2;                   // dO_i (+ -LSE*log2e): last read by dV_i
  static constexpr int kQ = kV + kTileBytes;
  static constexpr int kDO = kQ + kQStages * kTileBytes;
  static constexpr int kLse = kDO + kDStages * kTileBytes;
  static constexpr int kDelta = kLse + kDStages * kBT * 4;
  static constexpr int kCtl = kDelta + kQStages * kBT * 4;
  static constexpr int kSmem = kCtl + 256;
  static_assert(kSmem <= 232448, "dK/dV shared memory exceeds the per-CTA limit");
};

struct DkdvCtl {
  uint64_t bar_kv_full, bar_kv_empty;
  uint64_t bar_q_full[3], bar_q_empty[3];
  uint64_t bar_do_full[2], bar_do_empty[2];
  uint64_t bar_s_full, bar_dp_full, bar_p_ready, bar_ds_ready;
  uint64_t bar_acc_done, bar_acc_free, bar_final;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DkdvCtl) <= 256, "control block");

template <int D, bool kMask>
__global__ void __launch_bounds__(kSplitThreads, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ SegMaps tmQ, const __grid_constant__ SegMaps tmK,
                         const __grid_constant__ SegMaps tmV, const __grid_constant__ SegMaps tmDO,
                         const __grid_constant__ SeqDesc qd, const __grid_constant__ SeqDesc kd,
                         const float* __restrict__ nl2, const float* __restrict__ delta,
                         const uint8_t* __restrict__ key_mask, int mrows, __nv_bfloat16* __restrict__ dk,
                         __nv_bfloat16* __restrict__ dv, int B, int H, int num_items, int head_inner,
                         float scale, float scale_log2, DevCtx ctx) {
  using L = DkdvLayout<D>;
  constexpr int kChunks = D / 64;
  constexpr uint32_t kIdescKK = idesc_bf16_f32(128, kBT, false, false);  // S^T, dP^T
  constexpr uint32_t kIdescKM = idesc_bf16_f32(128, D, false, true);     // dV, dK (A in TMEM)
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;

  extern __shared__ __align__(1024) uint8_t smem[];
  DkdvCtl* ctl = reinterpret_cast<DkdvCtl*>(smem + L::kCtl);
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
  const int nkt = kd.tile0[kd.nseg];  // key tiles: the work items
  const int nqt = qd.tile0[qd.nseg];  // query tiles: the inner loop
  const int Sk = kd.total;
  const uint8_t* mask = kMask ? key_mask : nullptr;

  if (threadIdx.x == 0) {
    // a Q_i / dO_i stage is read by two GEMMs, each releasing it by a commit
    mbar_init(&ctl->bar_kv_full, 1);
    mbar_init(&ctl->bar_kv_empty, 1);
    for (int s = 0; s < L::kQStages; ++s) {
      mbar_init(&ctl->bar_q_full[s], 1);
      mbar_init(&ctl->bar_q_empty[s], 2);
    }
    for (int s = 0; s < L::kDStages; ++s) {
      mbar_init(&ctl->bar_do_full[s], 1);
      mbar_init(&ctl->bar_do_empty[s], 2);
    }
    mbar_init(&ctl->bar_s_full, 1);
    mbar_init(&ctl->bar_dp_full, 1);
    mbar_init(&ctl->bar_p_ready, kComputeThreads);
    mbar_init(&ctl->bar_ds_ready, kComputeThreads);
    mbar_init(&ctl->bar_acc_done, 1);
    mbar_init(&ctl->bar_acc_free, kComputeThreads);
    mbar_init(&ctl->bar_final, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    for (int p = 0; p < qd.nseg; ++p) {
      tma_prefetch_desc(&tmQ.m[p]);
      tma_prefetch_desc(&tmDO.m[p]);
    }
    for (int p = 0; p < kd.nseg; ++p) {
      tma_prefetch_desc(&tmK.m[p]);
      tma_prefetch_desc(&tmV.m[p]);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const MmaGuard mg = mma_guard(ctx, sbase, L::kSmem, tmem, 512);  // debug builds' operand checks
  const size_t k_extent = seq_extent(kd, B, H, D);

  uint32_t q_armed[3] = {0, 0, 0}, do_armed[2] = {0, 0}, kv_armed = 0;
  bool mma_issued = false;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    uint32_t nq = 0, it = 0;
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
      const Item3 w = head_inner ? decode_item_head_inner(item, nkt, H) : decode_item(item, nkt, H);
      if (kMask && !key_tile_any(mask, kd, w.b % mrows, w.t)) continue;
      if (lane == 0) {
        if (it > 0) ok = wait_or_abort(&ctl->bar_kv_empty, (it - 1) & 1, ctx, ctl);
        if (ok) {
          mbar_arrive_expect_tx(&ctl->bar_kv_full, 2 * L::kTileBytes);
          const SeqTile kt = seq_tile(kd, w.t);
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            tma_load_4d(smem + L::kK + c * kChunkBytes, &tmK.m[kt.seg], &ctl->bar_kv_full, c * 64, w.h, kt.row0, w.b);
            tma_load_4d(smem + L::kV + c * kChunkBytes, &tmV.m[kt.seg], &ctl->bar_kv_full, c * 64, w.h, kt.row0, w.b);
          }
          kv_armed = it + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      const size_t row0 = ((size_t)w.b * H + w.h) * ((size_t)nqt * kBT);
      SeqCursor qseg;  // query segment cursor
      for (int i = 0; ok && i < nqt; ++i, ++nq) {
        const SeqTile qt = seq_tile_at(qd, i, qseg);
        const int qs = nq % L::kQStages;
        const uint32_t qu = nq / L::kQStages;
        const int ds = nq % L::kDStages;
        const uint32_t du = nq / L::kDStages;
        if (lane == 0) {
          // Q_i with its Delta row, then dO_i with its -LSE*log2e row (rows past S
          // were written as Delta = 0 and -inf by the preprocess kernel)
          if (qu > 0) ok = wait_or_abort(&ctl->bar_q_empty[qs], (qu - 1) & 1, ctx, ctl);
          if (ok && (int)nq != ctx.drop_load) {
            mbar_arrive_expect_tx(&ctl->bar_q_full[qs], L::kTileBytes + kBT * 4);
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(smem + L::kQ + qs * L::kTileBytes + c * kChunkBytes, &tmQ.m[qt.seg], &ctl->bar_q_full[qs],
                          c * 64, w.h, qt.row0, w.b);
            bulk_load(sDelta + qs * kBT, delta + row0 + (size_t)i * kBT, kBT * 4, &ctl->bar_q_full[qs]);
            q_armed[qs] = qu + 1;
          }
          if (ok && du > 0) ok = wait_or_abort(&ctl->bar_do_empty[ds], (du - 1) & 1, ctx, ctl);
          if (ok) {
            mbar_arrive_expect_tx(&ctl->bar_do_full[ds], L::kTileBytes + kBT * 4);
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(smem + L::kDO + ds * L::kTileBytes + c * kChunkBytes, &tmDO.m[qt.seg],
                          &ctl->bar_do_full[ds], c * 64, w.h, qt.row0, w.b);
            bulk_load(sLse + ds * kBT, nl2 + row0 + (size_t)i * kBT, kBT * 4, &ctl->bar_do_full[ds]);
            do_armed[ds] = du + 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      ++it;
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer (warp 9)
    // One elected lane issues the four GEMMs of every query tile i in the order
    //   S^T_0 dP^T_0 | dV_0 S^T_1 | dK_0 dP^T_1 | dV_1 S^T_2 | dK_1 dP^T_2 | ...
    // each burst after the compute warps' handshake it depends on: dV_i and
    // S^T_{i+1} after p_ready(i) (P^T_i in TMEM; the compute warps arrive only once
    // Q_{i+1} has landed), dK_i and dP^T_{i+1} after ds_ready(i) (dS^T_i in TMEM,
    // dO_{i+1} landed).  While the issuer waits for one handshake the tensor pipe
    // runs the burst before it (1024 cycles).  The MMAs of one thread execute in
    // order: dV_i reads P^T_i before S^T_{i+1} overwrites those columns, and dK_i
    // reads dS^T_i before dP^T_{i+1} does.  The whole warp runs the schedule and
    // computes the descriptors; the waits, MMAs and commits are the elected
    // lane's, so that the compiler issues each MMA as a warp-uniform instruction.
    uint32_t el_lane;
    const bool el = elect_one_sync(&el_lane);
    bool ok = true;
    uint32_t nq = 0, it = 0;
    const uint32_t sK = sbase + L::kK;
    const uint32_t sV = sbase + L::kV;
    auto sq = [&](uint32_t g) { return sbase + L::kQ + (g % L::kQStages) * L::kTileBytes; };
    auto sdo = [&](uint32_t g) { return sbase + L::kDO + (g % L::kDStages) * L::kTileBytes; };
    // a wait of the elected lane, its outcome broadcast to the warp
    auto wait_el = [&](uint64_t* bar, uint32_t parity) {
      bool w = true;
      if (el) w = wait_or_abort(bar, parity, ctx, ctl);
      return __shfl_sync(0xffffffffu, w ? 1 : 0, el_lane) != 0;
    };
    // S^T_g = K Q_g^T (c = 0) or dP^T_g = V dO_g^T (c = 1); the second commit
    // releases this GEMM's read of the Q_g / dO_g stage
    auto issue_kk = [&](int c, uint32_t g) {
      const uint64_t a0 = sdesc_sw128(c == 0 ? sK : sV, 16, 1024);
      const uint64_t b0 = sdesc_sw128(c == 0 ? sq(g) : sdo(g), 16, 1024);
      const uint32_t d = tmem + (c == 0 ? kColS : kColDP);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
        const uint64_t a = desc_add(a0, off), b = desc_add(b0, off);
        if (el) mma_ss_checked(mg, d, a, b, kIdescKK, kk > 0, kBT);
      }
      if (el) {
        mma_commit(c == 0 ? &ctl->bar_s_full : &ctl->bar_dp_full);
        mma_commit(c == 0 ? &ctl->bar_q_empty[g % L::kQStages] : &ctl->bar_do_empty[g % L::kDStages]);
      }
    };
    // dV += P^T dO_g (c = 0; A = P^T in the S^T columns) or dK += dS^T Q_g (c = 1;
    // A = dS^T in the dP^T columns); the commit releases the dO_g / Q_g stage
    auto issue_acc = [&](int c, uint32_t g, bool first_acc) {
      const uint64_t b0 = sdesc_sw128(c == 0 ? sdo(g) : sq(g), kChunkBytes, 1024);
      const uint32_t d = tmem + (c == 0 ? kColDV : kColDK);
      const uint32_t a = tmem + (c == 0 ? kColS : kColDP);
#pragma unroll
      for (int kk = 0; kk < kBT / 16; ++kk) {
        const uint64_t b = desc_add(b0, kk * 2048);
        if (el) mma_ts_checked(mg, d, a + packed_a_col(kk), b, kIdescKM, (!first_acc || kk > 0) ? 1u : 0u, D);
      }
      if (el) mma_commit(c == 0 ? &ctl->bar_do_empty[g % L::kDStages] : &ctl->bar_q_empty[g % L::kQStages]);
    };
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
      const Item3 w = head_inner ? decode_item_head_inner(item, nkt, H) : decode_item(item, nkt, H);
      if (kMask && !key_tile_any(mask, kd, w.b % mrows, w.t)) continue;
      ok = wait_el(&ctl->bar_kv_full, it & 1);
      if (ok) ok = wait_el(&ctl->bar_q_full[nq % L::kQStages], (nq / L::kQStages) & 1);
      if (ok) ok = wait_el(&ctl->bar_do_full[nq % L::kDStages], (nq / L::kDStages) & 1);
      if (ok) {
        tc_fence_after();
        issue_kk(0, nq);
        issue_kk(1, nq);
        if (el) mma_issued = true;
      }
      for (int i = 0; ok && i < nqt; ++i) {
        const uint32_t g = nq + i;
        const bool more = i + 1 < nqt;
        if (!(ok = wait_el(&ctl->bar_p_ready, g & 1))) break;
        if (i == 0 && it > 0) {
          // the previous item's epilogue must have read dK / dV
          if (!(ok = wait_el(&ctl->bar_acc_free, (it - 1) & 1))) break;
        }
        tc_fence_after();
        issue_acc(0, g, i == 0);
        if (more) issue_kk(0, g + 1);
        if (!(ok = wait_el(&ctl->bar_ds_ready, g & 1))) break;
        tc_fence_after();
        issue_acc(1, g, i == 0);
        if (more) issue_kk(1, g + 1);
      }
      if (el) {
        if (ok) {
          mma_commit(&ctl->bar_acc_done);
          mma_commit(&ctl->bar_kv_empty);
        } else {
          *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
        }
      }
      __syncwarp();
      nq += nqt;
      ++it;
    }
  } else {
    // ------------------------------------------------------------ compute warps 0..7
    const int quad = warp & 3;
    const int hf = warp >> 2;
    const int jrow = quad * 32 + lane;  // key row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    uint32_t nq = 0, it = 0;
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
      const Item3 w = head_inner ? decode_item_head_inner(item, nkt, H) : decode_item(item, nkt, H);
      const SeqTile kt = seq_tile(kd, w.t);
      const bool kexists = jrow < kt.valid;  // key row kt.row0 + jrow of segment kt.seg
      const size_t off = seq_elem(kd, B, H, D, w.b, kt.seg, kexists ? kt.row0 + jrow : 0, w.h) + hf * (D / 2);
      const bool kstore = kexists && guard_store(ctx, off, D / 2, k_extent);  // this thread's half row of dK, dV
      if (kMask && !key_tile_any(mask, kd, w.b % mrows, w.t)) {
        // no attended key in this tile: dK = dV = 0
        if (kstore) {
#pragma unroll
          for (int c = 0; c < D / 16; ++c) {
            *reinterpret_cast<uint4*>(dk + off + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
            *reinterpret_cast<uint4*>(dv + off + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
          }
        }
        continue;
      }
      const bool kvalid =
          kexists && (!kMask || key_mask[(size_t)(w.b % mrows) * Sk + kd.off[kt.seg] + kt.row0 + jrow] != 0);
      for (int i = 0; i < nqt; ++i) {
        const uint32_t g = nq + i;
        const int qs = g % L::kQStages;
        const int ds = g % L::kDStages;
        // -LSE*log2e of Q_i sits with the dO_i stage, Delta_i with the Q_i stage;
        // both have landed before S^T_i completes, so these waits stay off the
        // path from S^T_i to P^T_i
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_do_full[ds], (g / L::kDStages) & 1, ctx, ctl));
        if (!ok) break;
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_q_full[qs], (g / L::kQStages) & 1, ctx, ctl));
        if (!ok) break;
        if (i + 1 < nqt) {
          // Q_{i+1}, read by the S^T MMA that this tile's p_ready releases
          const uint32_t g1 = g + 1;
          ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_q_full[g1 % L::kQStages], (g1 / L::kQStages) & 1,
                                                     ctx, ctl));
          if (!ok) break;
        }
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_s_full, g & 1, ctx, ctl));
        if (!ok) break;
        tc_fence_after();
        float p[64];
        tmem_ld32x2(tl + kColS + 64 * hf, tl + kColS + 64 * hf + 32, p);
        {
          const float2* nl2 = reinterpret_cast<const float2*>(sLse + ds * kBT + 64 * hf);
          const float2 c2 = make_float2(scale_log2, scale_log2);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = fma2(make_float2(p[2 * c], p[2 * c + 1]), c2, nl2[c]);
            p[2 * c] = ex2(x.x);
            p[2 * c + 1] = ex2(x.y);
          }
          if (!kvalid) {
#pragma unroll
            for (int c = 0; c < 64; ++c) p[c] = 0.f;
          }
        }
        // P^T as bf16 over the first 32 columns of this half's S^T region
        store_packed64(tl + kColS + 64 * hf, p);
        tc_fence_before();
        mbar_arrive(&ctl->bar_p_ready);
        if (i + 1 < nqt) {
          // dO_{i+1}, read by the dP^T MMA that this tile's ds_ready releases
          const uint32_t g1 = g + 1;
          ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_do_full[g1 % L::kDStages], (g1 / L::kDStages) & 1,
                                                     ctx, ctl));
          if (!ok) break;
        }
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_dp_full, g & 1, ctx, ctl));
        if (!ok) break;
        tc_fence_after();
        float dp[64];
        tmem_ld32x2(tl + kColDP + 64 * hf, tl + kColDP + 64 * hf + 32, dp);
        {
          const float2* dl = reinterpret_cast<const float2*>(sDelta + qs * kBT + 64 * hf);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 d =
                mul2(make_float2(p[2 * c], p[2 * c + 1]), sub2(make_float2(dp[2 * c], dp[2 * c + 1]), dl[c]));
            dp[2 * c] = d.x;
            dp[2 * c + 1] = d.y;
          }
        }
        store_packed64(tl + kColDP + 64 * hf, dp);
        tc_fence_before();
        mbar_arrive(&ctl->bar_ds_ready);
      }
      if (!ok) break;
      // epilogue: dV, and dK = scale * (dS^T Q)
      ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_acc_done, it & 1, ctx, ctl));
      if (!ok) break;
      tc_fence_after();
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        float gg[32];
        tmem_ld32(tl + kColDV + hf * (D / 2) + 32 * c, gg);
        if (kstore) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 v;
            v.x = pack_bf16(gg[8 * t + 0], gg[8 * t + 1]);
            v.y = pack_bf16(gg[8 * t + 2], gg[8 * t + 3]);
            v.z = pack_bf16(gg[8 * t + 4], gg[8 * t + 5]);
            v.w = pack_bf16(gg[8 * t + 6], gg[8 * t + 7]);
            *reinterpret_cast<uint4*>(dv + off + 32 * c + 8 * t) = v;
          }
        }
        tmem_ld32(tl + kColDK + hf * (D / 2) + 32 * c, gg);
        if (kstore) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 v;
            v.x = pack_bf16(gg[8 * t + 0] * scale, gg[8 * t + 1] * scale);
            v.y = pack_bf16(gg[8 * t + 2] * scale, gg[8 * t + 3] * scale);
            v.z = pack_bf16(gg[8 * t + 4] * scale, gg[8 * t + 5] * scale);
            v.w = pack_bf16(gg[8 * t + 6] * scale, gg[8 * t + 7] * scale);
            *reinterpret_cast<uint4*>(dk + off + 32 * c + 8 * t) = v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar_acc_free);
      nq += nqt;
      ++it;
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp && mma_issued) {
    // every MMA has completed before TMEM is released (mma_issued: the issuing lane)
    mma_commit(&ctl->bar_final);
    settle(&ctl->bar_final, 0, ctx);
  }
  if (warp == kProducerWarp && lane == 0) {
    if (kv_armed) settle(&ctl->bar_kv_full, (kv_armed - 1) & 1, ctx);
    for (int s = 0; s < 3; ++s)
      if (q_armed[s]) settle(&ctl->bar_q_full[s], (q_armed[s] - 1) & 1, ctx);
    for (int s = 0; s < 2; ++s)
      if (do_armed[s]) settle(&ctl->bar_do_full[s], (do_armed[s] - 1) & 1, ctx);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

// ---------------------------------------------------------------------------
// 3. dQ (Q-tile-major)
template <int D>
struct DqLayout {
  // K and V tiles in rings of their own: a K slot is freed only by dQ (late in a key
  // tile's processing), a V slot already by dP, so V gets fewer slots and K more
  static constexpr int kKRing = (D == 128) ? 4 : 7;
  static constexpr int kVRing = (D == 128) ? 3 : 6;
  static constexpr int kRing = kKRing + kVRing;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kRingOff = 0;  // K slots, then V slots (Q and dO live in TMEM)
  static constexpr int kCtl = kRingOff + kRing * kTileBytes;
  static constexpr int kWords = kCtl + 512;              // mask bits of the key tile in each K slot
  static constexpr int kCnt = kWords + kKRing * 16;      // attended key tiles per mask row
  static constexpr int kSmem = kCnt + kMaxCntRows * 4;
  static_assert(kSmem <= 232448, "dQ shared memory exceeds the per-CTA limit");
};

struct DqCtl {
  uint64_t bar_qdo_ready;
  uint64_t bar_kv_full[16], bar_kv_empty[16];
  uint64_t bar_s_full, bar_s_read, bar_dp_full, bar_ds_ready;
  uint64_t bar_dq_done, bar_dq_free, bar_final[2], bar_dq_step;
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(DqCtl) <= 512, "control block");

// kSeg: the key or query sequence has more than one segment (the fused Ulysses
// step); with one segment the per-tile addressing reduces to row 128j of map 0.
template <int D, bool kMask, bool kSeg>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_dq_kernel(const __grid_constant__ SegMaps tmK, const __grid_constant__ SegMaps tmV,
                       const __grid_constant__ SeqDesc qd, const __grid_constant__ SeqDesc kd,
                       const float* __restrict__ nl2g, const float* __restrict__ delta,
                       const uint8_t* __restrict__ key_mask, int mrows, const __nv_bfloat16* __restrict__ qg,
                       const __nv_bfloat16* __restrict__ dog, __nv_bfloat16* __restrict__ dq, int B, int H,
                       int num_items, float scale, float scale_log2, DevCtx ctx) {
  using L = DqLayout<D>;
  constexpr int kChunks = D / 64;
  constexpr int R = L::kRing;
  constexpr int KR = L::kKRing, VR = L::kVRing;
  // slot and use of key tile g's K and V
  auto kslot = [](uint32_t g) { return (int)(g % KR); };
  auto vslot = [](uint32_t g) { return KR + (int)(g % VR); };
  auto kpar = [](uint32_t g) { return (g / KR) & 1u; };
  auto vpar = [](uint32_t g) { return (g / VR) & 1u; };
  constexpr uint32_t kIdescKK = idesc_bf16_f32(128, kBT, false, false);  // S, dP
  constexpr uint32_t kIdescKM = idesc_bf16_f32(128, D, false, true);     // dQ (A in TMEM)
  // TMEM: S, dP (then dS), the dQ accumulator, and Q / dO as A operands of S / dP
  constexpr uint32_t kColS = 0, kColDP = 128, kColDQ = 256, kColQ = 384, kColDO = 448;

  extern __shared__ __align__(1024) uint8_t smem[];
  DqCtl* ctl = reinterpret_cast<DqCtl*>(smem + L::kCtl);
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(ctx.status, kStatusBadLaunch);
    return;
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nkt = kd.tile0[kd.nseg];  // key tiles: the inner loop
  const int nqt = qd.tile0[qd.nseg];  // query tiles: the work items
  const uint8_t* mask = kMask ? key_mask : nullptr;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->bar_qdo_ready, kComputeThreads);
    for (int s = 0; s < R; ++s) {
      mbar_init(&ctl->bar_kv_full[s], 1);
      mbar_init(&ctl->bar_kv_empty[s], s < KR ? 2 : 1);  // K: S and dQ read it; V: dP only
    }
    mbar_init(&ctl->bar_s_full, 1);
    // the compute warps plus the other issuer's hand-over (see the issuers)
    mbar_init(&ctl->bar_s_read, kComputeThreads + 1);
    mbar_init(&ctl->bar_dp_full, 1);
    mbar_init(&ctl->bar_ds_ready, kComputeThreads + 1);
    mbar_init(&ctl->bar_dq_done, 1);
    mbar_init(&ctl->bar_dq_free, kComputeThreads);
    mbar_init(&ctl->bar_dq_step, 1);
    mbar_init(&ctl->bar_final[0], 1);
    mbar_init(&ctl->bar_final[1], 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    for (int p = 0; p < kd.nseg; ++p) {
      tma_prefetch_desc(&tmK.m[p]);
      tma_prefetch_desc(&tmV.m[p]);
    }
  }
  if (warp == kMmaWarp) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  // Key tiles with at least one attended key, per mask row (batch b uses row b % mrows).
  // Every role takes an item's tile count from this table, which no one writes after the
  // start, and only the producer reads the mask itself: it hands each tile's bits to the
  // compute warps with the tile's K slot (`kwords`), so no per-tile mask read sits on the
  // issuers' or the compute warps' path.
  int* tile_cnt = reinterpret_cast<int*>(smem + L::kCnt);
  uint32_t(*kwords)[4] = reinterpret_cast<uint32_t(*)[4]>(smem + L::kWords);
  const bool skip = kMask && mrows <= kMaxCntRows;
  if (skip) {
    for (int r = threadIdx.x; r < mrows; r += kThreads) tile_cnt[r] = 0;
    __syncthreads();
    // one warp per (row, tile) pair, four tiles in flight per warp
    const int pairs = mrows * nkt;
    for (int p0 = warp * 4; p0 < pairs; p0 += (kThreads / 32) * 4) {
      bool any[4];
#pragma unroll
      for (int u = 0; u < 4; ++u) {
        const int pr = p0 + u;
        bool hit = false;
        if (pr < pairs) {
          const int r = pr / nkt, j = pr - r * nkt;
          const SeqTile kt = seq_tile(kd, j);
          const uint8_t* row = mask + (size_t)r * kd.total + kd.off[kt.seg] + kt.row0;
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int c = 32 * t + lane;
            hit |= c < kt.valid && row[c] != 0;
          }
        }
        any[u] = hit;
      }
#pragma unroll
      for (int u = 0; u < 4; ++u)
        if (__any_sync(0xffffffffu, any[u]) && lane == 0 && p0 + u < pairs) atomicAdd(&tile_cnt[(p0 + u) / nkt], 1);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;
  const MmaGuard mg = mma_guard(ctx, sbase, L::kSmem, tmem, 512);  // debug builds' operand checks
  const size_t q_extent = seq_extent(qd, B, H, D);
  // key tiles an item of batch b walks
  auto item_tiles = [&](int b) { return skip ? tile_cnt[b % mrows] : nkt; };

  uint32_t kv_armed[16] = {};
  bool mma_issued = false;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    uint32_t n = 0, it = 0, gp = 0;  // n: loads, gp: key tiles loaded
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x, ++it) {
      const Item3 w = decode_item(item, nqt, H);
      if (item_tiles(w.b) == 0) continue;  // no attended key: no load, dQ = 0
      SeqCursor kseg;  // key segment cursor (tiles are visited in order)
      for (int j = 0; ok && j < nkt; ++j) {
        uint32_t words[4] = {0u, 0u, 0u, 0u};
        if (kMask) {
          key_tile_bits(mask, kd, w.b % mrows, j, words);
          // the same test as the tile-count table: the other roles expect exactly those tiles
          if (skip && (words[0] | words[1] | words[2] | words[3]) == 0) continue;
        }
#pragma unroll
        for (int kind = 0; kind < 2; ++kind, ++n) {  // 0 = K_j, 1 = V_j
          const int slot = kind == 0 ? kslot(gp) : vslot(gp);
          const uint32_t use = kind == 0 ? gp / KR : gp / VR;
          if (lane == 0 && use > 0) ok = wait_or_abort(&ctl->bar_kv_empty[slot], (use - 1) & 1, ctx, ctl);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (kMask && kind == 0 && lane == 0) {
            // read by the compute warps between this tile's kv_full and its ds_ready, which
            // comes before the dQ MMA that frees the slot
#pragma unroll
            for (int t = 0; t < 4; ++t) kwords[slot][t] = words[t];
          }
          if (lane == 0 && (int)n != ctx.drop_load) {
            mbar_arrive_expect_tx(&ctl->bar_kv_full[slot], L::kTileBytes);
            int ms = 0, row0 = j * kBT;
            if constexpr (kSeg) {
              const SeqTile kt = seq_tile_at(kd, j, kseg);
              ms = kt.seg;
              row0 = kt.row0;
            }
            const CUtensorMap* map = kind == 0 ? &tmK.m[ms] : &tmV.m[ms];
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(smem + L::kRingOff + slot * L::kTileBytes + c * kChunkBytes, map,
                          &ctl->bar_kv_full[slot], c * 64, w.h, row0, w.b);
            kv_armed[slot] = use + 1;
          }
        }
        ++gp;
      }
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp1) {
    // ------------------------------------------------------------ MMA issuers (lane 0 of warps 9 and 10)
    // Two chains, each issued by its own thread, per processed key tile g:
    //   warp 9  (chain s): S_0 | S_1 | S_2 | ...            (S_{g+1} after s_read(g))
    //   warp 10 (chain d): dP_0 | dQ_0 dP_1 | dQ_1 dP_2 | ... (after ds_ready(g))
    // The threads take turns burst by burst, each waiting while the other's
    // burst runs.  The turn is handed over through the handshake barriers
    // themselves: chain d arrives on s_read(g) once it has issued all but four
    // MMAs of the burst holding dP_g, chain s on ds_ready(g) once it has done so
    // for S_{g+1} (after the last key tile, once s_read(last) has completed), so
    // each thread's one wait per burst covers both the compute warps' handshake
    // and its turn.  The tensor pipe queues only about one MMA, and a single
    // issuing thread that stopped to wait between GEMMs would leave it idle for
    // a few hundred cycles per wait.  In chain d, dQ_g and dP_{g+1} both take A
    // from TMEM, and dP_{g+1} is issued only once dQ_g has completed (see the
    // top of this file).
    const int c = warp - kMmaWarp;  // 0: chain s, 1: chain d
    bool ok = true;
    uint32_t g = 0, it = 0;  // g: processed key tiles across items
    uint32_t dq_step = 0;    // chain d: dQ completions waited for
    auto slot_addr = [&](int slot) { return sbase + L::kRingOff + slot * L::kTileBytes; };
    // hand the turn to the other chain (see above)
    auto pass_turn = [&]() { mbar_arrive(c == 0 ? &ctl->bar_ds_ready : &ctl->bar_s_read); };
    // S_gg = Q K^T (A = Q in TMEM); releases (this thread's share of) the slots of K_gg and V_gg
    auto issue_s = [&](uint32_t gg, bool pass) {
      const uint64_t b0 = sdesc_sw128(slot_addr(kslot(gg)), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
        mma_ts_checked(mg, tmem + kColS, tmem + kColQ + kk * 8, desc_add(b0, off), kIdescKK, kk > 0, kBT);
        if (pass && kk == (D / 16 > 4 ? D / 16 - 5 : 0)) pass_turn();
      }
      mma_commit(&ctl->bar_s_full);
      mma_commit(&ctl->bar_kv_empty[kslot(gg)]);
    };
    // dP_gg = dO V^T (A = dO in TMEM); V_gg is read only by this GEMM.  dP is on the
    // critical path (dP -> dS -> dQ -> next dP), so the turn passes only after its
    // last MMA: S MMAs issued earlier would be interleaved with it and delay it.
    auto issue_dp = [&](uint32_t gg, bool pass) {
      const uint64_t b0 = sdesc_sw128(slot_addr(vslot(gg)), 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
        mma_ts_checked(mg, tmem + kColDP, tmem + kColDO + kk * 8, desc_add(b0, off), kIdescKK, kk > 0, kBT);
      }
      if (pass) pass_turn();
      mma_commit(&ctl->bar_dp_full);
      mma_commit(&ctl->bar_kv_empty[vslot(gg)]);
    };
    // dQ += dS K_gg (A = dS in the dP columns)
    auto issue_dq = [&](uint32_t gg, bool first, bool pass) {
      const uint64_t b0 = sdesc_sw128(slot_addr(kslot(gg)), kChunkBytes, 1024);
#pragma unroll
      for (int kk = 0; kk < kBT / 16; ++kk) {
        mma_ts_checked(mg, tmem + kColDQ, tmem + kColDP + packed_a_col(kk), desc_add(b0, kk * 2048), kIdescKM,
                       (!first || kk > 0) ? 1u : 0u, D);
        if (pass && kk == kBT / 16 - 5) pass_turn();
      }
      mma_commit(&ctl->bar_kv_empty[kslot(gg)]);
    };
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x, ++it) {
      const Item3 w = decode_item(item, nqt, H);
      const int ntl = item_tiles(w.b);  // key tiles of this item
      if (ntl == 0) {
        // No attended key: no MMA, and the compute warps write dQ = 0 once dq_done
        // of the item arrives.  They still store Q and dO and arrive on qdo_ready:
        // both chains wait for that phase too, or a later item's parity wait could
        // be satisfied by this phase still being open.
        if (lane == 0) ok = wait_or_abort(&ctl->bar_qdo_ready, it & 1, ctx, ctl);
        ok = __shfl_sync(0xffffffffu, ok, 0);
        if (!ok) break;
        if (lane == 0 && c == 1) mma_commit(&ctl->bar_dq_done);
        __syncwarp();
        continue;
      }
      if (lane == 0) {
        // Q and dO of this item were stored into TMEM by the compute warps.  Past the
        // first key tile the compute warps arrive on s_read / ds_ready only after they
        // have seen K / V of the next tile land, so no other wait is needed.
        ok = wait_or_abort(&ctl->bar_qdo_ready, it & 1, ctx, ctl);
        if (ok) {
          // K_g for chain s, V_g for chain d
          ok = c == 0 ? wait_or_abort(&ctl->bar_kv_full[kslot(g)], kpar(g), ctx, ctl)
                      : wait_or_abort(&ctl->bar_kv_full[vslot(g)], vpar(g), ctx, ctl);
        }
        if (ok) {
          tc_fence_after();
          // chain d's first burst (dP of the item's first key tile) releases chain s's S of the next tile
          if (c == 0) issue_s(g, false);
          else issue_dp(g, true);
          mma_issued = true;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      for (int i = 0; ok && i < ntl; ++i) {
        const bool more = i + 1 < ntl;  // another key tile in this item
        const bool first = i == 0;
        if (lane == 0) {
          if (c == 0) {
            // S of the next key tile once this one's S was read into registers (after the
            // last tile: only the hand-over, which must follow s_read of that tile)
            ok = wait_or_abort(&ctl->bar_s_read, g & 1, ctx, ctl);
            if (ok) {
              tc_fence_after();
              if (more) issue_s(g + 1, true);
              else pass_turn();
            }
          } else {
            ok = wait_or_abort(&ctl->bar_ds_ready, g & 1, ctx, ctl);
            if (ok && first && it > 0) ok = wait_or_abort(&ctl->bar_dq_free, (it - 1) & 1, ctx, ctl);
            if (ok) {
              tc_fence_after();
              issue_dq(g, first, false);
              if (more) {
                // dP_{g+1} issued directly behind dQ_g (both with A in TMEM) gave
                // wrong results, also with dS moved out of the dP columns: dQ_g must
                // complete first.
                mma_commit(&ctl->bar_dq_step);
                ok = wait_or_abort(&ctl->bar_dq_step, dq_step & 1, ctx, ctl);
                ++dq_step;
                if (ok) {
                  tc_fence_after();
                  issue_dp(g + 1, true);
                }
              }
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
        ++g;
      }
      if (!ok) break;
      if (lane == 0 && c == 1) mma_commit(&ctl->bar_dq_done);
      __syncwarp();
    }
    if (!ok && lane == 0) *reinterpret_cast<volatile int*>(&ctl->abort) = 1;  // the other issuer waits for our hand-over
  } else {
    // ------------------------------------------------------------ compute warps 0..7
    const int quad = warp & 3;
    const int hf = warp >> 2;
    const int row = quad * 32 + lane;  // query row = TMEM lane
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    bool ok = true;
    uint32_t g = 0, it = 0;
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x, ++it) {
      const Item3 w = decode_item(item, nqt, H);
      const SeqTile qt = seq_tile(qd, w.t);
      const bool qvalid = row < qt.valid;  // query row qt.row0 + row of segment qt.seg
      const size_t qoff = seq_elem(qd, B, H, D, w.b, qt.seg, qvalid ? qt.row0 + row : 0, w.h);
      {
        // the previous item's MMAs have all completed (its dq_done was waited on)
        const __nv_bfloat16* src = (hf == 0 ? qg : dog) + qoff;
#pragma unroll
        for (int c = 0; c < D / 64; ++c) {
          uint32_t wv[32];
#pragma unroll
          for (int t = 0; t < 8; ++t) {
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (qvalid) v = __ldg(reinterpret_cast<const uint4*>(src) + 8 * c + t);
            wv[4 * t + 0] = v.x;
            wv[4 * t + 1] = v.y;
            wv[4 * t + 2] = v.z;
            wv[4 * t + 3] = v.w;
          }
          tmem_st32_bits(tl + (hf == 0 ? kColQ : kColDO) + 32 * c, wv);
        }
        tc_fence_before();
        mbar_arrive(&ctl->bar_qdo_ready);
      }
      // rows past the segment read the padding (-inf, 0)
      const size_t prow = ((size_t)w.b * H + w.h) * ((size_t)nqt * kBT) + (size_t)w.t * kBT + row;
      const float nl2 = nl2g[prow];
      const float dl = delta[prow];
      int ntiles = 0;
      const int ntl = item_tiles(w.b);  // key tiles of this item
      SeqCursor kseg;  // key segment cursor
      for (int j = 0; j < ntl; ++j) {  // j: the key tile itself when there is no mask
        uint32_t words[4];
        if (kMask) {
          // the tile's mask bits, left by the producer with its K slot; the first tile
          // of an item waits for that slot's load here (later tiles did below)
          if (j == 0) {
            ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_kv_full[kslot(g)], kpar(g), ctx, ctl));
            if (!ok) break;
          }
#pragma unroll
          for (int t = 0; t < 4; ++t) words[t] = kwords[kslot(g)][t];
        }
        // is there a next key tile?  Its K and V are read by the MMAs this tile's
        // s_read and ds_ready release; they normally land long before, and
        // waiting for them here keeps these waits off the issuing thread.
        const bool has_next = j + 1 < ntl;
        if (has_next) {
          bool okw = wait_or_abort(&ctl->bar_kv_full[kslot(g + 1)], kpar(g + 1), ctx, ctl);
          if (okw) okw = wait_or_abort(&ctl->bar_kv_full[vslot(g + 1)], vpar(g + 1), ctx, ctl);
          ok = __all_sync(0xffffffffu, okw);
          if (!ok) break;
        }
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_s_full, g & 1, ctx, ctl));
        if (!ok) break;
        tc_fence_after();
        float p[64];
        tmem_ld32x2(tl + kColS + 64 * hf, tl + kColS + 64 * hf + 32, p);
        tc_fence_before();
        mbar_arrive(&ctl->bar_s_read);
        {
          const float2 c2 = make_float2(scale_log2, scale_log2);
          const float2 n2 = make_float2(nl2, nl2);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = fma2(make_float2(p[2 * c], p[2 * c + 1]), c2, n2);
            p[2 * c] = ex2(x.x);
            p[2 * c + 1] = ex2(x.y);
          }
          if (kMask) {
            const uint32_t w0 = words[2 * hf], w1 = words[2 * hf + 1];
            if ((w0 & w1) != 0xffffffffu) {  // only tiles with masked (or missing) keys need it
#pragma unroll
              for (int c = 0; c < 32; ++c) {
                if (!((w0 >> c) & 1u)) p[c] = 0.f;
                if (!((w1 >> c) & 1u)) p[32 + c] = 0.f;
              }
            }
          } else {
            // the last tile of a key segment is partial: its rows past the segment read as zeros
            const int lim = (kSeg ? seq_tile_at(kd, j, kseg).valid
                                  : ((j + 1) * kBT > kd.total ? kd.total - j * kBT : kBT)) - 64 * hf;
            if (lim < 64) {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (c >= lim) p[c] = 0.f;
            }
          }
        }
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_dp_full, g & 1, ctx, ctl));
        if (!ok) break;
        tc_fence_after();
        float dp[64];
        tmem_ld32x2(tl + kColDP + 64 * hf, tl + kColDP + 64 * hf + 32, dp);
        {
          const float2 d2 = make_float2(dl, dl);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 d =
                mul2(make_float2(p[2 * c], p[2 * c + 1]), sub2(make_float2(dp[2 * c], dp[2 * c + 1]), d2));
            dp[2 * c] = d.x;
            dp[2 * c + 1] = d.y;
          }
        }
        store_packed64(tl + kColDP + 64 * hf, dp);
        tc_fence_before();
        mbar_arrive(&ctl->bar_ds_ready);
        ++g;
        ++ntiles;
      }
      if (!ok) break;
      // epilogue: dQ = scale * (dS K)
      ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_dq_done, it & 1, ctx, ctl));
      if (!ok) break;
      tc_fence_after();
      __nv_bfloat16* drow = dq + qoff + hf * (D / 2);
      const bool qstore = qvalid && guard_store(ctx, qoff + hf * (D / 2), D / 2, q_extent);  // this thread's half row
#pragma unroll 1
      for (int c = 0; c < D / 64; ++c) {
        float gg[32];
        tmem_ld32(tl + kColDQ + hf * (D / 2) + 32 * c, gg);
        if (ntiles == 0) {
#pragma unroll
          for (int t = 0; t < 32; ++t) gg[t] = 0.f;
        }
        if (qstore) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            uint4 v;
            v.x = pack_bf16(gg[8 * t + 0] * scale, gg[8 * t + 1] * scale);
            v.y = pack_bf16(gg[8 * t + 2] * scale, gg[8 * t + 3] * scale);
            v.z = pack_bf16(gg[8 * t + 4] * scale, gg[8 * t + 5] * scale);
            v.w = pack_bf16(gg[8 * t + 6] * scale, gg[8 * t + 7] * scale);
            *reinterpret_cast<uint4*>(drow + 32 * c + 8 * t) = v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar_dq_free);
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before();
  __syncthreads();
  if ((warp == kMmaWarp || warp == kMmaWarp1) && lane == 0 && mma_issued) {
    mma_commit(&ctl->bar_final[warp - kMmaWarp]);
    settle(&ctl->bar_final[warp - kMmaWarp], 0, ctx);
  }
  if (warp == kProducerWarp && lane == 0) {
    for (int s = 0; s < R; ++s)
      if (kv_armed[s]) settle(&ctl->bar_kv_full[s], (kv_armed[s] - 1) & 1, ctx);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess || n <= 0)
    return 148;
  return n;
}

int grid_cap(size_t work, int per_block) {
  const size_t need = (work + per_block - 1) / per_block;
  const size_t cap = (size_t)sm_count() * 8;
  return (int)(need < 1 ? 1 : (need < cap ? need : cap));
}

// Optional profiling events of the calling thread (uaa_set_bwd_profile_events).
thread_local cudaEvent_t t_prof_events[3] = {nullptr, nullptr, nullptr};

int record_prof(int i, cudaStream_t stream) {
  if (!t_prof_events[i]) return UAA_OK;
  cudaError_t e = cudaEventRecord(t_prof_events[i], stream);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "uaa_attn_bwd: profiling event: %s", cudaGetErrorString(e));
  return UAA_OK;
}

template <int D, bool kMask>
int launch_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
               const uint8_t* mask, int mrows, void* dq, void* dk, void* dv, int B, const SeqDesc& qd,
               const SeqDesc& kd, int H, float scale, float* delta, bool fused, cudaStream_t stream,
               const DevCtx& ctx) {
  const size_t rows = (size_t)B * qd.total * H;
  const int nqt = qd.tile0[qd.nseg], nkt = kd.tile0[kd.nseg];
  float* nl2 = delta + (size_t)B * H * nqt * kBT;
  bwd_preprocess_kernel<D><<<grid_cap(rows * 8, 256), 256, 0, stream>>>(
      static_cast<const __nv_bfloat16*>(out), static_cast<const __nv_bfloat16*>(dout), lse, delta, nl2, qd, B, H);
  int st = check_launch("uaa_attn_bwd (preprocess)");
  if (st) return st;
  if (fused) {
    // one K/V-major pass (dQ by reductions into the fp32 accumulator after the two row vectors)
    float* dq_acc = nl2 + (size_t)B * H * nqt * kBT;
    return launch_bwd_fused(q, k, v, dout, mask, mrows, dq, dk, dv, B, qd.total, kd.total, H, D, scale, delta, nl2,
                            dq_acc, stream, ctx, record_prof);
  }
  SegMaps mq, mk, mv, mdo;
  if ((st = encode_seq_maps(&mq, q, qd, B, H, D, 128))) return st;
  if ((st = encode_seq_maps(&mk, k, kd, B, H, D, 128))) return st;
  if ((st = encode_seq_maps(&mv, v, kd, B, H, D, 128))) return st;
  if ((st = encode_seq_maps(&mdo, dout, qd, B, H, D, 128))) return st;
  // dK/dV items are key tiles, dQ items are query tiles
  const long long items_k = (long long)nkt * H * B;
  const long long items_q = (long long)nqt * H * B;
  if (items_k > INT32_MAX || items_q > INT32_MAX)
    return set_error(UAA_ERR_UNSUPPORTED, "uaa_attn_bwd: too many work items");
  const int grid_k = (int)(items_k < sm_count() ? items_k : sm_count());
  const int grid_q = (int)(items_q < sm_count() ? items_q : sm_count());
  if ((st = record_prof(0, stream))) return st;
  if (items_k > 0) {
    auto kern = attn_bwd_dkdv_kernel<D, kMask>;
    const int smem = DkdvLayout<D>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "uaa_attn_bwd: smem attribute: %s", cudaGetErrorString(e));
    // With a key mask, order the items head-innermost (the empty key tiles spread evenly
    // over the CTAs) when one batch's Q and dO for all heads fit in half of L2
    const int head_inner = (mask != nullptr && 4LL * H * qd.total * D <= (64LL << 20)) ? 1 : 0;
    kern<<<grid_k, kSplitThreads, smem, stream>>>(mq, mk, mv, mdo, qd, kd, nl2, delta, mask, mrows,
                                             static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), B, H,
                                             (int)items_k, head_inner, scale, scale * kLog2e, ctx);
    if ((st = check_launch("uaa_attn_bwd (dK/dV)"))) return st;
  }
  if ((st = record_prof(1, stream))) return st;
  if (items_q > 0) {
    auto kern = (qd.nseg > 1 || kd.nseg > 1) ? attn_bwd_dq_kernel<D, kMask, true> : attn_bwd_dq_kernel<D, kMask, false>;
    const int smem = DqLayout<D>::kSmem;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "uaa_attn_bwd: smem attribute: %s", cudaGetErrorString(e));
    kern<<<grid_q, kThreads, smem, stream>>>(mk, mv, qd, kd, nl2, delta, mask, mrows,
                                             static_cast<const __nv_bfloat16*>(q),
                                             static_cast<const __nv_bfloat16*>(dout), static_cast<__nv_bfloat16*>(dq),
                                             B, H, (int)items_q, scale, scale * kLog2e, ctx);
    if ((st = check_launch("uaa_attn_bwd (dQ)"))) return st;
  }
  return record_prof(2, stream);
}

// mrows: rows of key_mask; batch b uses row b % mrows
int bwd_dispatch(const void* q, const void* k, const void* v, const void* out, const void* dout, const float* lse,
                 const uint8_t* key_mask, int mrows, void* dq, void* dk, void* dv, int B, const SeqDesc& qd,
                 const SeqDesc& kd, int H, int D, float scale, float* delta, cudaStream_t s, const DevCtx& ctx,
                 bool fused = false) {
#define UAA_BWD(DD, MM)                                                                                        \
  launch_bwd<DD, MM>(q, k, v, out, dout, lse, key_mask, mrows, dq, dk, dv, B, qd, kd, H, scale, delta, fused, s, \
                     ctx)
  if (D == 64) return key_mask ? UAA_BWD(64, true) : UAA_BWD(64, false);
  return key_mask ? UAA_BWD(128, true) : UAA_BWD(128, false);
#undef UAA_BWD
}

}  // namespace
}  // namespace uaa

using namespace uaa;

extern "C" void uaa_set_bwd_profile_events(void* before_dkdv, void* after_dkdv, void* after_dq) {
  t_prof_events[0] = static_cast<cudaEvent_t>(before_dkdv);
  t_prof_events[1] = static_cast<cudaEvent_t>(after_dkdv);
  t_prof_events[2] = static_cast<cudaEvent_t>(after_dq);
}

extern "C" size_t uaa_attn_bwd_workspace_bytes(int B, int S, int H, int D) {
  if (B < 0 || S < 0 || H < 0 || (D != 64 && D != 128)) return 0;
  // Delta and -LSE*log2e, each (B, H, S_pad) fp32, S_pad = S rounded up to 128
  return (((size_t)B * H * padded_rows(S) * 8) + 255) & ~(size_t)255;
}

extern "C" int uaa_attn_bwd_cross(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                  const float* lse, const uint8_t* key_mask, void* dq, void* dk, void* dv, int B,
                                  int Sq, int Sk, int H, int D, float scale, void* workspace, size_t workspace_bytes,
                                  uaa_stream_t stream) {
  const char* fn = "uaa_attn_bwd";
  int st = validate_attn_sizes(fn, B, Sq, Sk, H, D, scale);
  if (st) return st;
  if ((uint64_t)B * H == 0 || (uint64_t)Sq + Sk == 0) return UAA_OK;
  if (Sq == 0) return set_error(UAA_ERR_INVALID_ARG, "%s: keys without queries (Sq = 0)", fn);
  if ((st = check_dev_ptr(fn, "q", q)) || (st = check_dev_ptr(fn, "k", k)) || (st = check_dev_ptr(fn, "v", v)) ||
      (st = check_dev_ptr(fn, "out", out)) || (st = check_dev_ptr(fn, "dout", dout)) ||
      (st = check_dev_ptr(fn, "dq", dq)) || (st = check_dev_ptr(fn, "dk", dk)) || (st = check_dev_ptr(fn, "dv", dv)))
    return st;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: lse is NULL or not 4-byte aligned", fn);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace is NULL or not 256-byte aligned", fn);
  const size_t need = uaa_attn_bwd_workspace_bytes(B, Sq, H, D);
  if (workspace_bytes < need)
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace has %zu bytes, %zu needed", fn, workspace_bytes, need);
  DevCtx ctx;
  if ((st = get_dev_ctx(&ctx))) return st;
  return bwd_dispatch(q, k, v, out, dout, lse, key_mask, B, dq, dk, dv, B, seq_plain(Sq), seq_plain(Sk), H, D,
                      scale, static_cast<float*>(workspace), static_cast<cudaStream_t>(stream), ctx);
}

extern "C" size_t uaa_ulysses_attn_bwd_workspace_bytes(int P, const int* shard_lens, int cap, int B, int H, int D) {
  SeqDesc sd;
  if (B < 0 || H < 0 || (D != 64 && D != 128)) return 0;
  if (seq_sharded(&sd, P, shard_lens, cap, "uaa_ulysses_attn_bwd_workspace_bytes")) return 0;
  // Delta and -LSE*log2e, each (B, H, tiles * 128) fp32 in query-tile order
  return (((size_t)B * H * sd.tile0[sd.nseg] * kBT * 8) + 255) & ~(size_t)255;
}

extern "C" int uaa_ulysses_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                    const float* lse, const uint8_t* key_mask, void* dq, void* dk, void* dv, int P,
                                    const int* shard_lens, int cap, int B, int H, int D, float scale, void* workspace,
                                    size_t workspace_bytes, uaa_stream_t stream) {
  const char* fn = "uaa_ulysses_attn_bwd";
  SeqDesc sd;
  int st = seq_sharded(&sd, P, shard_lens, cap, fn);
  if (st) return st;
  if ((st = validate_attn_sizes(fn, B, sd.total, sd.total, H, D, scale))) return st;
  if ((uint64_t)B * H == 0) return UAA_OK;
  if ((st = check_dev_ptr(fn, "q", q)) || (st = check_dev_ptr(fn, "k", k)) || (st = check_dev_ptr(fn, "v", v)) ||
      (st = check_dev_ptr(fn, "out", out)) || (st = check_dev_ptr(fn, "dout", dout)) ||
      (st = check_dev_ptr(fn, "dq", dq)) || (st = check_dev_ptr(fn, "dk", dk)) || (st = check_dev_ptr(fn, "dv", dv)))
    return st;
  if ((uint64_t)P * B * cap * H * D * 4 >= (1ull << 40))
    return set_error(UAA_ERR_UNSUPPORTED, "%s: tensor larger than the TMA stride range", fn);
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // padding rows of the gradient shards are zero, as after the head->seq exchange
  if ((st = zero_pad_rows(dq, sd, B, H, D, s)) || (st = zero_pad_rows(dk, sd, B, H, D, s)) ||
      (st = zero_pad_rows(dv, sd, B, H, D, s)))
    return st;
  if (sd.total == 0) return UAA_OK;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: lse is NULL or not 4-byte aligned", fn);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace is NULL or not 256-byte aligned", fn);
  const size_t need = uaa_ulysses_attn_bwd_workspace_bytes(P, shard_lens, cap, B, H, D);
  if (workspace_bytes < need)
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace has %zu bytes, %zu needed", fn, workspace_bytes, need);
  DevCtx ctx;
  if ((st = get_dev_ctx(&ctx))) return st;
  return bwd_dispatch(q, k, v, out, dout, lse, key_mask, B, dq, dk, dv, B, sd, sd, H, D, scale,
                      static_cast<float*>(workspace), s, ctx);
}

extern "C" int uaa_attn_bwd(const void* q, const void* k, const void* v, const void* out, const void* dout,
                            const float* lse, const uint8_t* key_mask, void* dq, void* dk, void* dv, int B, int S,
                            int H, int D, float scale, void* workspace, size_t workspace_bytes,
                            uaa_stream_t stream) {
  return uaa_attn_bwd_cross(q, k, v, out, dout, lse, key_mask, dq, dk, dv, B, S, S, H, D, scale, workspace,
                            workspace_bytes, stream);
}

extern "C" size_t uaa_attn_bwd_fused_workspace_bytes(int B, int S, int H, int D) {
  if (B < 0 || S < 0 || H < 0 || (D != 64 && D != 128)) return 0;
  // Delta and -LSE*log2e (B, H, S_pad) fp32, then the fp32 dQ accumulator (B, H, S_pad, D)
  const size_t rows = (size_t)B * H * padded_rows(S);
  return ((rows * 8 + rows * D * 4) + 255) & ~(size_t)255;
}

extern "C" int uaa_attn_bwd_fused(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                  const float* lse, const uint8_t* key_mask, void* dq, void* dk, void* dv, int B,
                                  int S, int H, int D, float scale, void* workspace, size_t workspace_bytes,
                                  uaa_stream_t stream) {
  const char* fn = "uaa_attn_bwd_fused";
  int st = validate_attn_sizes(fn, B, S, S, H, D, scale);
  if (st) return st;
  if ((uint64_t)B * H * S == 0) return UAA_OK;
  if ((st = check_dev_ptr(fn, "q", q)) || (st = check_dev_ptr(fn, "k", k)) || (st = check_dev_ptr(fn, "v", v)) ||
      (st = check_dev_ptr(fn, "out", out)) || (st = check_dev_ptr(fn, "dout", dout)) ||
      (st = check_dev_ptr(fn, "dq", dq)) || (st = check_dev_ptr(fn, "dk", dk)) || (st = check_dev_ptr(fn, "dv", dv)))
    return st;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: lse is NULL or not 4-byte aligned", fn);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace is NULL or not 256-byte aligned", fn);
  const size_t need = uaa_attn_bwd_fused_workspace_bytes(B, S, H, D);
  if (workspace_bytes < need)
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace has %zu bytes, %zu needed", fn, workspace_bytes, need);
  DevCtx ctx;
  if ((st = get_dev_ctx(&ctx))) return st;
  return bwd_dispatch(q, k, v, out, dout, lse, key_mask, B, dq, dk, dv, B, seq_plain(S), seq_plain(S), H, D, scale,
                      static_cast<float*>(workspace), static_cast<cudaStream_t>(stream), ctx, true);
}

extern "C" int uaa_attn_bwd_groups(const void* q, const void* k, const void* v, const void* out, const void* dout,
                                   const float* lse, const uint8_t* key_mask, void* dq, void* dk, void* dv, int G,
                                   int B, int S, int H, int D, float scale, void* workspace, size_t workspace_bytes,
                                   uaa_stream_t stream) {
  const char* fn = "uaa_attn_bwd_groups";
  if (G < 1 || B < 0) return set_error(UAA_ERR_INVALID_ARG, "%s: G=%d, B=%d", fn, G, B);
  if ((long long)G * B > 65535) return set_error(UAA_ERR_UNSUPPORTED, "%s: G*B must be <= 65535", fn);
  const int GB = G * B;
  int st = validate_attn_sizes(fn, GB, S, S, H, D, scale);
  if (st) return st;
  if ((uint64_t)GB * S * H == 0) return UAA_OK;
  if ((st = check_dev_ptr(fn, "q", q)) || (st = check_dev_ptr(fn, "k", k)) || (st = check_dev_ptr(fn, "v", v)) ||
      (st = check_dev_ptr(fn, "out", out)) || (st = check_dev_ptr(fn, "dout", dout)) ||
      (st = check_dev_ptr(fn, "dq", dq)) || (st = check_dev_ptr(fn, "dk", dk)) || (st = check_dev_ptr(fn, "dv", dv)))
    return st;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: lse is NULL or not 4-byte aligned", fn);
  if (!workspace || (reinterpret_cast<uintptr_t>(workspace) & 255u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace is NULL or not 256-byte aligned", fn);
  const size_t need = uaa_attn_bwd_workspace_bytes(GB, S, H, D);
  if (workspace_bytes < need)
    return set_error(UAA_ERR_INVALID_ARG, "%s: workspace has %zu bytes, %zu needed", fn, workspace_bytes, need);
  DevCtx ctx;
  if ((st = get_dev_ctx(&ctx))) return st;
  return bwd_dispatch(q, k, v, out, dout, lse, key_mask, B, dq, dk, dv, GB, seq_plain(S), seq_plain(S), H, D, scale,
                      static_cast<float*>(workspace), static_cast<cudaStream_t>(stream), ctx);
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
// Nothing in the array needs to start at zero: every call rewrites the Delta
// and -LSE*log2e vectors it holds (padding rows included) before reading them.
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
  int st = validate_attn_sizes(fn, B, S, S, H, D, scale);
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
