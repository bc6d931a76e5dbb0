// Attention backward in one K/V-tile-major pass on sm_103a: dK and dV
// accumulate in TMEM as in the split path, and each query tile's dQ
// contribution dS K is formed by a fifth GEMM and added into an fp32 dQ
// accumulator in global memory with vector reductions (red.global.add.v4.f32).
//
// "Fix double transpose of K/V in templated attention backward", description:
// the backward op takes Q, K, V in one layout, dO and the saved LSE and returns
// dQ, dK, dV.  The pages leave open how dQ is formed; this pass does the five
// GEMMs of the textbook gradient once each (the split path recomputes S and dP
// in a separate Q-major pass, seven GEMMs in all), at the price of dQ
// reductions whose order varies from run to run: dQ is then not bit-for-bit
// reproducible (dK and dV are).
//
// Per work item (128 keys of one (batch, head)) and query tile i:
//   S^T_i  = K Q_i^T                    (SS MMA -> TMEM columns [0,128))
//   dP^T_i = V dO_i^T                   (SS MMA -> TMEM columns [128,256))
//   P^T = exp2(S^T*c - lse2), dS^T = P^T (dP^T - Delta)          (compute warps)
//   dV += P^T dO_i                      (TS MMA, P^T packed bf16 in the S columns)
//   dK += dS^T Q_i                      (TS MMA, dS^T packed bf16 in the dP columns)
//   dQ_i = dS_i K                       (SS MMA: dS from shared memory, MN-major)
// dS^T rows are also written to shared memory by the compute warps (thread =
// key row, 64 query values = one 128-byte swizzled row), which is the MN-major
// A operand of the dQ GEMM.  With D = 128 the 512 TMEM columns hold S^T, dP^T,
// dV and dK, so dQ_i is accumulated in the dP^T columns once dK_i has read
// dS^T_i there, and dP^T_{i+1} waits until the compute warps have drained dQ_i;
// with D = 64 dQ has columns of its own.
//
// Roles: warps 0-7 compute (TMEM lane quadrant = warp % 4, column half =
// warp / 4), warp 8 TMA producer, warp 9 issuer A (dV_i, S^T_{i+1}: released by
// the P^T hand-over), warp 10 issuer B (dK_i, dQ_i: released by the dS
// hand-over; dP^T_{i+1}: released by the dQ drain).  The compute warps order
// their work dS_i, P_{i+1}, drain of dQ_i, so S^T_{i+1} and the softmax of the
// next tile overlap dK_i and dQ_i.  Each item walks the query tiles starting at
// its own key-tile index, so the CTAs of one head add into different dQ rows.
#include <math.h>

#include "attn_bwd_shared.cuh"

namespace uaa {
namespace {

template <int D>
struct FusedLayout {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kStages = (D == 128) ? 2 : 4;  // Q_i / dO_i stages
  static constexpr int kK = 0;
  static constexpr int kV = kK + kTileBytes;
  static constexpr int kQ = kV + kTileBytes;
  static constexpr int kDO = kQ + kStages * kTileBytes;
  static constexpr int kDS = kDO + kStages * kTileBytes;  // dS (128 keys x 128 queries bf16)
  static constexpr int kLse = kDS + 128 * 128 * 2;
  static constexpr int kDelta = kLse + kStages * kBT * 4;
  static constexpr int kCtl = kDelta + kStages * kBT * 4;
  static constexpr int kSmem = kCtl + 256;
  static_assert(kSmem <= 232448, "fused backward shared memory exceeds the per-CTA limit");
  static_assert(kDS % 1024 == 0, "swizzled operands need 1024-byte alignment");
};

struct FusedCtl {
  uint64_t bar_kv_full, bar_kv_empty;
  uint64_t bar_q_full[4], bar_q_empty[4];
  uint64_t bar_do_full[4], bar_do_empty[4];
  uint64_t bar_s_full, bar_dp_full, bar_p_ready, bar_ds_ready, bar_dq_full, bar_dq_free;
  uint64_t bar_acc_done, bar_acc_free, bar_final[2];
  uint32_t tmem_base;
  int abort;
};
static_assert(sizeof(FusedCtl) <= 256, "control block");

// Query tile of step i of an item whose key tile is j: the walk starts at tile j % nqt.
__device__ __forceinline__ int fused_qtile(int i, int j, int nqt) {
  int t = i + j % nqt;
  return t >= nqt ? t - nqt : t;
}

template <int D, bool kMask>
__global__ void __launch_bounds__(kThreads, 1)
    attn_bwd_fused_kernel(const __grid_constant__ SegMaps tmQ, const __grid_constant__ SegMaps tmK,
                          const __grid_constant__ SegMaps tmV, const __grid_constant__ SegMaps tmDO,
                          const __grid_constant__ SeqDesc qd, const __grid_constant__ SeqDesc kd,
                          const float* __restrict__ nl2, const float* __restrict__ delta,
                          const uint8_t* __restrict__ key_mask, int mrows, float* __restrict__ dq_acc,
                          __nv_bfloat16* __restrict__ dk, __nv_bfloat16* __restrict__ dv, int B, int H,
                          int num_items, float scale, float scale_log2, DevCtx ctx) {
  using L = FusedLayout<D>;
  constexpr int kChunks = D / 64;
  constexpr int NS = L::kStages;
  constexpr bool kSharedDq = (D == 128);  // dQ_i lives in the dP^T columns
  constexpr uint32_t kIdescKK = idesc_bf16_f32(128, kBT, false, false);  // S^T, dP^T
  constexpr uint32_t kIdescKM = idesc_bf16_f32(128, D, false, true);     // dV, dK (A in TMEM)
  constexpr bool kTransDq = (D == 128);   // dQ^T (M = D = 128) rather than dQ (M = queries)
  constexpr uint32_t kIdescQ = idesc_bf16_f32(128, kTransDq ? kBT : D, true, true);  // both operands MN-major
  constexpr uint32_t kColS = 0, kColDP = 128, kColDV = 256, kColDK = 256 + D;
  constexpr uint32_t kColDQ = kSharedDq ? kColDP : 256 + 2 * D;

  extern __shared__ __align__(1024) uint8_t smem[];
  FusedCtl* ctl = reinterpret_cast<FusedCtl*>(smem + L::kCtl);
  float* sLse = reinterpret_cast<float*>(smem + L::kLse);
  float* sDelta = reinterpret_cast<float*>(smem + L::kDelta);
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    if (threadIdx.x == 0) atomicOr(ctx.status, kStatusBadLaunch);
    return;
  }
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int Sq = qd.total, Sk = kd.total;  // plain sequences (one segment each)
  const int nkt = (Sk + kBT - 1) / kBT;  // key tiles: the work items
  const int nqt = (Sq + kBT - 1) / kBT;  // query tiles: the inner loop
  const uint8_t* mask = kMask ? key_mask : nullptr;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->bar_kv_full, 1);
    mbar_init(&ctl->bar_kv_empty, 2);  // both issuers read K (and V)
    for (int s = 0; s < NS; ++s) {
      mbar_init(&ctl->bar_q_full[s], 1);
      mbar_init(&ctl->bar_q_empty[s], 2);  // S^T (issuer A), dK (issuer B)
      mbar_init(&ctl->bar_do_full[s], 1);
      mbar_init(&ctl->bar_do_empty[s], 2);  // dP^T (issuer B), dV (issuer A)
    }
    mbar_init(&ctl->bar_s_full, 1);
    mbar_init(&ctl->bar_dp_full, 1);
    mbar_init(&ctl->bar_p_ready, kComputeThreads);
    mbar_init(&ctl->bar_ds_ready, kComputeThreads);
    mbar_init(&ctl->bar_dq_full, 1);
    mbar_init(&ctl->bar_dq_free, kComputeThreads);
    mbar_init(&ctl->bar_acc_done, 2);
    mbar_init(&ctl->bar_acc_free, kComputeThreads);
    mbar_init(&ctl->bar_final[0], 1);
    mbar_init(&ctl->bar_final[1], 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    tma_prefetch_desc(&tmQ.m[0]);
    tma_prefetch_desc(&tmDO.m[0]);
    tma_prefetch_desc(&tmK.m[0]);
    tma_prefetch_desc(&tmV.m[0]);
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
  const size_t k_extent = (size_t)B * Sk * H * D, acc_extent = (size_t)B * H * nqt * kBT * D;

  uint32_t q_armed[4] = {0, 0, 0, 0}, do_armed[4] = {0, 0, 0, 0}, kv_armed = 0;
  bool mma_issued = false;

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    uint32_t nq = 0, it = 0;
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
      const Item3 w = decode_item(item, nkt, H);
      if (kMask && !key_tile_any(mask, kd, w.b % mrows, w.t)) continue;
      if (lane == 0) {
        if (it > 0) ok = wait_or_abort(&ctl->bar_kv_empty, (it - 1) & 1, ctx, ctl);
        if (ok) {
          mbar_arrive_expect_tx(&ctl->bar_kv_full, 2 * L::kTileBytes);
#pragma unroll
          for (int c = 0; c < kChunks; ++c) {
            tma_load_4d(smem + L::kK + c * kChunkBytes, &tmK.m[0], &ctl->bar_kv_full, c * 64, w.h, w.t * kBT, w.b);
            tma_load_4d(smem + L::kV + c * kChunkBytes, &tmV.m[0], &ctl->bar_kv_full, c * 64, w.h, w.t * kBT, w.b);
          }
          kv_armed = it + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      const size_t row0 = ((size_t)w.b * H + w.h) * ((size_t)nqt * kBT);
      for (int i = 0; ok && i < nqt; ++i, ++nq) {
        const int qt = fused_qtile(i, w.t, nqt);
        const int s = nq % NS;
        const uint32_t u = nq / NS;
        if (lane == 0) {
          // Q_i with its Delta row, then dO_i with its -LSE*log2e row
          if (u > 0) ok = wait_or_abort(&ctl->bar_q_empty[s], (u - 1) & 1, ctx, ctl);
          if (ok && (int)nq != ctx.drop_load) {
            mbar_arrive_expect_tx(&ctl->bar_q_full[s], L::kTileBytes + kBT * 4);
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(smem + L::kQ + s * L::kTileBytes + c * kChunkBytes, &tmQ.m[0], &ctl->bar_q_full[s],
                          c * 64, w.h, qt * kBT, w.b);
            bulk_load(sDelta + s * kBT, delta + row0 + (size_t)qt * kBT, kBT * 4, &ctl->bar_q_full[s]);
            q_armed[s] = u + 1;
          }
          if (ok && u > 0) ok = wait_or_abort(&ctl->bar_do_empty[s], (u - 1) & 1, ctx, ctl);
          if (ok) {
            mbar_arrive_expect_tx(&ctl->bar_do_full[s], L::kTileBytes + kBT * 4);
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(smem + L::kDO + s * L::kTileBytes + c * kChunkBytes, &tmDO.m[0], &ctl->bar_do_full[s],
                          c * 64, w.h, qt * kBT, w.b);
            bulk_load(sLse + s * kBT, nl2 + row0 + (size_t)qt * kBT, kBT * 4, &ctl->bar_do_full[s]);
            do_armed[s] = u + 1;
          }
        }
        ok = __shfl_sync(0xffffffffu, ok, 0);
      }
      ++it;
    }
  } else if (warp == kMmaWarp || warp == kMmaWarp1) {
    // ------------------------------------------------------------ MMA issuers (lane 0 of warps 9 and 10)
    // A (warp 9):  S^T_0 | dV_0 S^T_1 | dV_1 S^T_2 | ...        (each burst after p_ready)
    // B (warp 10): dP^T_0 | dK_0 dQ_0 | dP^T_1 | dK_1 dQ_1 | ... (dK/dQ after ds_ready, dP^T after dq_free
    //              with D = 128, where dQ_i occupies the dP^T columns)
    // MMAs of one thread execute in order: dV_i reads P^T_i (S columns) before
    // S^T_{i+1} overwrites them, and dK_i reads dS^T_i (dP columns) before dQ_i
    // (D = 128) overwrites them.
    const bool isA = warp == kMmaWarp;
    bool ok = true;
    uint32_t nq = 0, it = 0;
    const uint32_t sK = sbase + L::kK;
    const uint32_t sV = sbase + L::kV;
    const uint32_t sDS = sbase + L::kDS;
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
      const Item3 w = decode_item(item, nkt, H);
      if (kMask && !key_tile_any(mask, kd, w.b % mrows, w.t)) continue;
      if (lane == 0) {
        auto sq = [&](uint32_t g) { return sbase + L::kQ + (g % NS) * L::kTileBytes; };
        auto sdo = [&](uint32_t g) { return sbase + L::kDO + (g % NS) * L::kTileBytes; };
        // S^T_g = K Q_g^T (A) or dP^T_g = V dO_g^T (B)
        auto issue_first = [&](uint32_t g) {
          const uint64_t a0 = sdesc_sw128(isA ? sK : sV, 16, 1024);
          const uint64_t b0 = sdesc_sw128(isA ? sq(g) : sdo(g), 16, 1024);
          const uint32_t d = tmem + (isA ? kColS : kColDP);
#pragma unroll
          for (int kk = 0; kk < D / 16; ++kk) {
            const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
            mma_ss_checked(mg, d, desc_add(a0, off), desc_add(b0, off), kIdescKK, kk > 0, kBT);
          }
          mma_commit(isA ? &ctl->bar_s_full : &ctl->bar_dp_full);
          mma_commit(isA ? &ctl->bar_q_empty[g % NS] : &ctl->bar_do_empty[g % NS]);
        };
        // dV += P^T dO_g (A) or dK += dS^T Q_g (B)
        auto issue_acc = [&](uint32_t g, bool first_acc) {
          const uint64_t b0 = sdesc_sw128(isA ? sdo(g) : sq(g), kChunkBytes, 1024);
          const uint32_t d = tmem + (isA ? kColDV : kColDK);
          const uint32_t a = tmem + (isA ? kColS : kColDP);
#pragma unroll
          for (int kk = 0; kk < kBT / 16; ++kk)
            mma_ts_checked(mg, d, a + packed_a_col(kk), desc_add(b0, kk * 2048), kIdescKM,
                           (!first_acc || kk > 0) ? 1u : 0u, D);
          mma_commit(isA ? &ctl->bar_do_empty[g % NS] : &ctl->bar_q_empty[g % NS]);
        };
        // D = 128: dQ_g^T = K^T dS_g^T, so that a TMEM lane holds one dQ column d for the
        // tile's 128 queries and a warp's 32 lanes add 32 consecutive columns of a query row
        // (128 contiguous bytes per reduction instruction).  A = K^T (D x keys, MN-major: the
        // K tile's 64-column chunks 16 KB apart), B = dS^T (queries x keys, MN-major: the dS
        // tile's 64-query chunks 16 KB apart); a K step of 16 keys = 16 rows = 2048 bytes.
        // D = 64: dQ_g = dS_g K (A = dS, B = K, the same two descriptors swapped).
        auto issue_dq = [&]() {
          const uint64_t ds0 = sdesc_sw128(sDS, 128 * 128, 1024);
          const uint64_t k0 = sdesc_sw128(sK, kChunkBytes, 1024);
          const uint64_t a0 = kTransDq ? k0 : ds0, b0 = kTransDq ? ds0 : k0;
#pragma unroll
          for (int kk = 0; kk < kBT / 16; ++kk)
            mma_ss_checked(mg, tmem + kColDQ, desc_add(a0, kk * 2048), desc_add(b0, kk * 2048), kIdescQ, kk > 0,
                           kTransDq ? kBT : D);
          mma_commit(&ctl->bar_dq_full);
        };
        ok = wait_or_abort(&ctl->bar_kv_full, it & 1, ctx, ctl);
        if (ok) {
          if (isA) {
            ok = wait_or_abort(&ctl->bar_q_full[nq % NS], (nq / NS) & 1, ctx, ctl);
          } else {
            ok = wait_or_abort(&ctl->bar_do_full[nq % NS], (nq / NS) & 1, ctx, ctl);
            // D = 128: the previous item's last dQ (in the dP columns) has been drained
            if (ok && kSharedDq && nq > 0) ok = wait_or_abort(&ctl->bar_dq_free, (nq - 1) & 1, ctx, ctl);
          }
        }
        if (ok) {
          tc_fence_after();
          issue_first(nq);
          mma_issued = true;
        }
        for (int i = 0; ok && i < nqt; ++i) {
          const uint32_t g = nq + i;
          const bool more = i + 1 < nqt;
          if (isA) {
            if (!(ok = wait_or_abort(&ctl->bar_p_ready, g & 1, ctx, ctl))) break;
            if (i == 0 && it > 0 && !(ok = wait_or_abort(&ctl->bar_acc_free, (it - 1) & 1, ctx, ctl))) break;
            tc_fence_after();
            issue_acc(g, i == 0);
            if (more) {
              // Q_{g+1} has normally landed long ago (its stage was freed by tile g-1)
              const uint32_t g1 = g + 1;
              if (!(ok = wait_or_abort(&ctl->bar_q_full[g1 % NS], (g1 / NS) & 1, ctx, ctl))) break;
              issue_first(g1);
            }
          } else {
            if (!(ok = wait_or_abort(&ctl->bar_ds_ready, g & 1, ctx, ctl))) break;
            if (i == 0 && it > 0 && !(ok = wait_or_abort(&ctl->bar_acc_free, (it - 1) & 1, ctx, ctl))) break;
            // D = 64: dQ_{g-1} (own columns) has been drained before dQ_g overwrites it
            if (!kSharedDq && g > 0 && !(ok = wait_or_abort(&ctl->bar_dq_free, (g - 1) & 1, ctx, ctl))) break;
            tc_fence_after();
            issue_acc(g, i == 0);
            issue_dq();
            if (more) {
              // D = 128: dP^T_{g+1} overwrites the dP columns that hold dQ_g
              const uint32_t g1 = g + 1;
              if (kSharedDq && !(ok = wait_or_abort(&ctl->bar_dq_free, g & 1, ctx, ctl))) break;
              if (!(ok = wait_or_abort(&ctl->bar_do_full[g1 % NS], (g1 / NS) & 1, ctx, ctl))) break;
              tc_fence_after();
              issue_first(g1);
            }
          }
        }
        if (ok) {
          mma_commit(&ctl->bar_acc_done);
          mma_commit(&ctl->bar_kv_empty);
        } else {
          *reinterpret_cast<volatile int*>(&ctl->abort) = 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      nq += nqt;
      ++it;
    }
  } else {
    // ------------------------------------------------------------ compute warps 0..7
    const int quad = warp & 3;
    const int hf = warp >> 2;
    const int jrow = quad * 32 + lane;  // key row (TMEM lane) of S^T, dP^T, dV, dK; query row of dQ
    const uint32_t tl = tmem + ((uint32_t)(quad * 32) << 16);
    // this thread's row of the dS tile: chunk hf (queries 64*hf ..), row jrow, 16-byte units swizzled
    uint8_t* ds_row = smem + L::kDS + hf * (128 * 128) + jrow * 128;
    bool ok = true;
    uint32_t nq = 0, it = 0;
    const float2 c2 = make_float2(scale_log2, scale_log2);
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
      const Item3 w = decode_item(item, nkt, H);
      const int kvalid_rows = Sk - w.t * kBT < kBT ? Sk - w.t * kBT : kBT;
      const bool kexists = jrow < kvalid_rows;
      const size_t off = (((size_t)w.b * Sk + (kexists ? w.t * kBT + jrow : 0)) * H + w.h) * D + hf * (D / 2);
      const bool kstore = kexists && guard_store(ctx, off, D / 2, k_extent);  // this thread's half row of dK, dV
      if (kMask && !key_tile_any(mask, kd, w.b % mrows, w.t)) {
        // no attended key in this tile: dK = dV = 0, and no dQ contribution
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
          kexists && (!kMask || key_mask[(size_t)(w.b % mrows) * Sk + w.t * kBT + jrow] != 0);
      float p[64];  // P^T of the current query tile (this thread's key row, 64 queries)
      // P^T_g from S^T_g; then arrive on p_ready (which releases dV_g and S^T_{g+1})
      auto make_p = [&](uint32_t g) -> bool {
        const int s = g % NS;
        // -LSE*log2e of the tile's queries arrives with dO_g
        if (!__all_sync(0xffffffffu, wait_or_abort(&ctl->bar_do_full[s], (g / NS) & 1, ctx, ctl))) return false;
        if (!__all_sync(0xffffffffu, wait_or_abort(&ctl->bar_s_full, g & 1, ctx, ctl))) return false;
        tc_fence_after();
        tmem_ld32x2(tl + kColS + 64 * hf, tl + kColS + 64 * hf + 32, p);
        const float2* n2 = reinterpret_cast<const float2*>(sLse + s * kBT + 64 * hf);
#pragma unroll
        for (int c = 0; c < 32; ++c) {
          const float2 x = fma2(make_float2(p[2 * c], p[2 * c + 1]), c2, n2[c]);
          p[2 * c] = ex2(x.x);
          p[2 * c + 1] = ex2(x.y);
        }
        if (!kvalid) {
#pragma unroll
          for (int c = 0; c < 64; ++c) p[c] = 0.f;
        }
        store_packed64(tl + kColS + 64 * hf, p);
        tc_fence_before();
        mbar_arrive(&ctl->bar_p_ready);
        return true;
      };
      if (!(ok = make_p(nq))) break;
      for (int i = 0; i < nqt; ++i) {
        const uint32_t g = nq + i;
        const int qt = fused_qtile(i, w.t, nqt);
        const bool more = i + 1 < nqt;
        // ---- dS_g = P (dP - Delta): TMEM (A operand of dK_g) and shared memory (A of dQ_g);
        // Delta of the tile's queries arrives with Q_g
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_q_full[g % NS], (g / NS) & 1, ctx, ctl));
        if (!ok) break;
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_dp_full, g & 1, ctx, ctl));
        if (!ok) break;
        tc_fence_after();
        {
          float dp[64];
          tmem_ld32x2(tl + kColDP + 64 * hf, tl + kColDP + 64 * hf + 32, dp);
          const float2* dl = reinterpret_cast<const float2*>(sDelta + (g % NS) * kBT + 64 * hf);
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 d =
                mul2(make_float2(p[2 * c], p[2 * c + 1]), sub2(make_float2(dp[2 * c], dp[2 * c + 1]), dl[c]));
            dp[2 * c] = d.x;
            dp[2 * c + 1] = d.y;
          }
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) pk[c] = pack_bf16(dp[2 * c], dp[2 * c + 1]);
          tmem_st32_bits(tl + kColDP + 64 * hf, pk);
          // the row of 64 queries in the 128-byte-swizzled layout: 16-byte unit u at u ^ (row & 7)
#pragma unroll
          for (int u = 0; u < 8; ++u)
            *reinterpret_cast<uint4*>(ds_row + ((u ^ (jrow & 7)) << 4)) =
                make_uint4(pk[4 * u], pk[4 * u + 1], pk[4 * u + 2], pk[4 * u + 3]);
        }
        fence_proxy_async_smem();  // the generic-proxy stores to dS must be visible to the MMA
        tc_fence_before();
        mbar_arrive(&ctl->bar_ds_ready);
        // ---- P of the next query tile (S^T_{g+1} was issued right after dV_g)
        if (more && !(ok = make_p(g + 1))) break;
        // ---- dQ_g: add this thread's query row (half of its D columns) into the accumulator
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_dq_full, g & 1, ctx, ctl));
        if (!ok) break;
        tc_fence_after();
        {
          float acc[D / 2];
          if constexpr (D == 128)
            tmem_ld32x2(tl + kColDQ + 64 * hf, tl + kColDQ + 64 * hf + 32, *reinterpret_cast<float(*)[64]>(acc));
          else
            tmem_ld32(tl + kColDQ + 32 * hf, *reinterpret_cast<float(*)[32]>(acc));
          tc_fence_before();
          mbar_arrive(&ctl->bar_dq_free);
          float* acc_bh = dq_acc + ((size_t)w.b * H + w.h) * ((size_t)nqt * kBT) * D;
          if constexpr (kTransDq) {
            // lane = column d = jrow, acc[c] = dQ[query 64*hf + c][d]: the warp adds 32 consecutive
            // columns of one query row per instruction
            const int q0 = qt * kBT + 64 * hf;
            const size_t a0 = ((size_t)w.b * H + w.h) * ((size_t)nqt * kBT) * D + (size_t)q0 * D + jrow;
            if (guard_store(ctx, a0, (size_t)63 * D + 1, acc_extent)) {
#pragma unroll
              for (int c = 0; c < 64; ++c)
                if (q0 + c < Sq) atomicAdd(acc_bh + (size_t)(q0 + c) * D + jrow, acc[c]);
            }
          } else {
            const int qrow = qt * kBT + jrow;  // query row of this thread in dQ_g
            if (qrow < Sq &&
                guard_store(ctx, ((size_t)w.b * H + w.h) * ((size_t)nqt * kBT) * D + (size_t)qrow * D + hf * (D / 2),
                            D / 2, acc_extent)) {
              float* dst = acc_bh + (size_t)qrow * D + hf * (D / 2);
#pragma unroll
              for (int c = 0; c < D / 8; ++c)
                asm volatile("red.global.add.v4.f32 [%0], {%1, %2, %3, %4};" ::"l"(dst + 4 * c), "f"(acc[4 * c]),
                             "f"(acc[4 * c + 1]), "f"(acc[4 * c + 2]), "f"(acc[4 * c + 3])
                             : "memory");
            }
          }
        }
      }
      if (!ok) break;
      // ---- epilogue: dV, and dK = scale * (dS^T Q)
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
  if ((warp == kMmaWarp || warp == kMmaWarp1) && lane == 0 && mma_issued) {
    mma_commit(&ctl->bar_final[warp - kMmaWarp]);
    settle(&ctl->bar_final[warp - kMmaWarp], 0, ctx);
  }
  if (warp == kProducerWarp && lane == 0) {
    if (kv_armed) settle(&ctl->bar_kv_full, (kv_armed - 1) & 1, ctx);
    for (int s = 0; s < NS; ++s) {
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

// dq[b, s, h, :] = bf16(scale * acc[b, h, s, :]) for s < Sq; one thread per 8 columns.
template <int D>
__global__ void __launch_bounds__(256) dq_convert_kernel(const float* __restrict__ acc, __nv_bfloat16* __restrict__ dq,
                                                         int B, int Sq, int H, int Spad, float scale) {
  constexpr int kVec = D / 8;
  const size_t total = (size_t)B * Sq * H * kVec;
  for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
    const int v = (int)(i % kVec);
    size_t r = i / kVec;
    const int h = (int)(r % H);
    r /= H;
    const int s = (int)(r % Sq);
    const int b = (int)(r / Sq);
    const float4* src = reinterpret_cast<const float4*>(acc + (((size_t)b * H + h) * Spad + s) * D + 8 * v);
    const float4 a = __ldcs(src), c = __ldcs(src + 1);
    uint4 o;
    o.x = pack_bf16(a.x * scale, a.y * scale);
    o.y = pack_bf16(a.z * scale, a.w * scale);
    o.z = pack_bf16(c.x * scale, c.y * scale);
    o.w = pack_bf16(c.z * scale, c.w * scale);
    *reinterpret_cast<uint4*>(dq + i * 8) = o;
  }
}

int sm_count_fused() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) !=
                                                cudaSuccess || n <= 0)
    return 148;
  return n;
}

template <int D, bool kMask>
int launch_fused(const void* q, const void* k, const void* v, const void* dout, const uint8_t* mask, int mrows,
                 void* dq, void* dk, void* dv, int B, int Sq, int Sk, int H, float scale, const float* delta,
                 const float* nl2, float* dq_acc, cudaStream_t stream, const DevCtx& ctx,
                 int (*mark)(int, cudaStream_t)) {
  const SeqDesc qd = seq_plain(Sq), kd = seq_plain(Sk);
  SegMaps mq, mk, mv, mdo;
  int st;
  if ((st = encode_seq_maps(&mq, q, qd, B, H, D, 128))) return st;
  if ((st = encode_seq_maps(&mk, k, kd, B, H, D, 128))) return st;
  if ((st = encode_seq_maps(&mv, v, kd, B, H, D, 128))) return st;
  if ((st = encode_seq_maps(&mdo, dout, qd, B, H, D, 128))) return st;
  const int nqt = (Sq + kBT - 1) / kBT, nkt = (Sk + kBT - 1) / kBT;
  const size_t acc_bytes = (size_t)B * H * nqt * kBT * D * sizeof(float);
  cudaError_t e = cudaMemsetAsync(dq_acc, 0, acc_bytes, stream);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "uaa_attn_bwd: dQ accumulator clear: %s", cudaGetErrorString(e));
  const long long items = (long long)nkt * H * B;
  if (items > INT32_MAX) return set_error(UAA_ERR_UNSUPPORTED, "uaa_attn_bwd: too many work items");
  const int sms = sm_count_fused();
  if ((st = mark(0, stream))) return st;
  if (items > 0) {
    auto kern = attn_bwd_fused_kernel<D, kMask>;
    const int smem = FusedLayout<D>::kSmem;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
    if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "uaa_attn_bwd: smem attribute: %s", cudaGetErrorString(e));
    const int grid = (int)(items < sms ? items : sms);
    kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, mdo, qd, kd, nl2, delta, mask, mrows, dq_acc,
                                           static_cast<__nv_bfloat16*>(dk), static_cast<__nv_bfloat16*>(dv), B, H,
                                           (int)items, scale, scale * kLog2e, ctx);
    if ((st = check_launch("uaa_attn_bwd (fused)"))) return st;
  }
  if ((st = mark(1, stream))) return st;
  const size_t vecs = (size_t)B * Sq * H * (D / 8);
  const size_t blocks = (vecs + 255) / 256;
  const int cgrid = (int)(blocks < (size_t)sms * 8 ? blocks : (size_t)sms * 8);
  dq_convert_kernel<D><<<cgrid < 1 ? 1 : cgrid, 256, 0, stream>>>(dq_acc, static_cast<__nv_bfloat16*>(dq), B, Sq, H,
                                                                  nqt * kBT, scale);
  if ((st = check_launch("uaa_attn_bwd (dQ convert)"))) return st;
  return mark(2, stream);
}

}  // namespace

// Fused backward after the preprocess kernel (Delta and -LSE*log2e in the workspace); mark(i)
// is called on the stream before the kernel (0), after it (1) and after the dQ conversion (2).
int launch_bwd_fused(const void* q, const void* k, const void* v, const void* dout, const uint8_t* mask, int mrows,
                     void* dq, void* dk, void* dv, int B, int Sq, int Sk, int H, int D, float scale,
                     const float* delta, const float* nl2, float* dq_acc, cudaStream_t s, const DevCtx& ctx,
                     int (*mark)(int, cudaStream_t)) {
#define UAA_FUSED(DD, MM) \
  launch_fused<DD, MM>(q, k, v, dout, mask, mrows, dq, dk, dv, B, Sq, Sk, H, scale, delta, nl2, dq_acc, s, ctx, mark)
  if (D == 64) return mask ? UAA_FUSED(64, true) : UAA_FUSED(64, false);
  return mask ? UAA_FUSED(128, true) : UAA_FUSED(128, false);
#undef UAA_FUSED
}

}  // namespace uaa
