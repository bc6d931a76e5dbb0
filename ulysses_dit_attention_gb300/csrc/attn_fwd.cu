// Attention forward on sm_103a: O = softmax(scale * Q K^T + bias) V and the
// log-sum-exp, for non-causal multi-head attention in BSHD layout.
//
// "Fix double transpose of K/V in templated attention backward", description:
// the forward op returns out in BSHD; follow-up item 1: the LSE must always be
// produced for the backward (it is written unconditionally here); follow-up
// item 2: a bool mask enters as an additive -inf/0 bias.  "[attention] Add
// Ulysses Anything backward", Unsupported cases: the key-padding mask is
// head-broadcast (B, 1, 1, S).
//
// Design: a persistent grid (one CTA per SM) walks work items; an item is a
// pair of 128-row query tiles (256 rows) of one (batch, head).
//   warp 8     TMA producer: the item's two Q tiles, then K_j, V_j tiles of
//              128 keys through a 5-stage ring (128-byte swizzled, 64 columns
//              per box); with a mask it also packs each tile's 128 mask bits
//              into shared memory.
//   warp 9     tcgen05 issuer (lane 0), ping-pong over the two tiles:
//                S0_0 S1_0 | PV0_0 S0_1 | PV1_0 S1_1 | PV0_1 S0_2 | ...
//              so while one softmax warpgroup works on its tile the tensor
//              core runs the other tile's MMAs.  PV reads P from TMEM (A
//              operand in tensor memory) and V from shared memory.  The
//              softmax warpgroups hand P over through hardware named
//              barriers, not mbarriers: a load by the issuing thread waits
//              behind the MMAs it has queued, which would drain the tensor
//              pipe at every hand-over.
//   warps 0-3  softmax of query tile 0, warps 4-7 softmax of tile 1: thread r
//              owns query row r (TMEM lane r), so the row max and row sum are
//              thread-local; online softmax in base 2 with a lazily updated
//              offset (O is rescaled in TMEM only when the row max grew by
//              more than 2^8); P is packed to bf16 pairs and stored over the
//              first 64 columns of the tile's S buffer with tcgen05.st; the
//              epilogue writes O / l in bf16 and LSE = offset*ln2 + ln l.
// The S_t of the next key tile is issued after PV_t of the current one: the
// MMAs of one thread execute in issue order, so PV_t has read P_t before S_t
// overwrites those columns.
// TMEM columns: [0,128) S/P of tile 0, [128,256) S/P of tile 1, [256,256+D)
// O of tile 0, [256+D,256+2D) O of tile 1.
// Query and key sequences are segmented (SeqDesc): a plain (B, S, H, D)
// tensor is one segment; the sequence shards of a Ulysses step are P segments,
// read and written in place (one TMA tensor map per segment; 128-row tiles
// never straddle two segments; keys past a segment's end are masked, query
// rows past it are not written).
#include <math.h>

#include "uaa_common.cuh"

namespace uaa {
namespace {

constexpr int kBN = 128;  // keys per K/V tile
constexpr int kChunkBytes = 128 * 128;  // 128 rows x 128 bytes (one swizzle column block)
constexpr int kThreads = 320;
constexpr int kProducerWarp = 8;
constexpr int kMmaWarp = 9;
constexpr float kRescaleThreshold = 8.0f;
// One column pair of P in kExpFmaEvery takes its exponentials from exp2_fma2
// (FMA pipe) instead of ex2 (special-function unit): with two 128-row query
// tiles per CTA, the 2 x 128 x 128 exponentials of a key-tile step take as
// many special-function cycles as the step's four GEMMs take tensor cycles.
constexpr int kExpFmaEvery = 8;
// named barrier kBarP + t: "P_t is in TMEM" (the 128 threads of softmax warpgroup t
// arrive, the issuer warp syncs)
constexpr uint32_t kBarP = 1;
constexpr uint32_t kBarPCount = 128 + 32;  // log2 units: rescale O only when the max grows by > 2^8
template <int D>
struct FwdLayout {
  static constexpr int kRing = 5;
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kQ = 0;                                  // two Q tiles
  static constexpr int kRingOff = kQ + 2 * kTileBytes;          // K/V ring
  static constexpr int kCtl = kRingOff + kRing * kTileBytes;
  static constexpr int kCnt = kCtl + 512;                       // attended key tiles per mask row
  static constexpr int kSmem = kCnt + kMaxCntRows * 4;
  static_assert(kSmem <= 232448, "forward shared memory exceeds the per-CTA limit");
  static_assert(kRing <= 5, "control block holds five ring slots");
};

struct FwdCtl {
  uint64_t bar_q_full;
  uint64_t bar_q_empty;
  uint64_t bar_kv_full[5];
  uint64_t bar_kv_empty[5];
  uint64_t bar_s_full[2];
  uint64_t bar_pv_done[2];
  uint64_t bar_o_free;
  uint64_t bar_final;
  uint32_t tmem_base;
  int abort;
  uint32_t mask_words[5][4];  // per ring slot (filled with the V tile)
};
static_assert(sizeof(FwdCtl) <= 512, "control block");

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}


struct Item {
  int qp, h, b;
};

__device__ __forceinline__ Item decode_item(int item, int nqp, int H) {
  Item it;
  it.qp = item % nqp;
  const int bh = item / nqp;
  it.h = bh % H;
  it.b = bh / H;
  return it;
}

// kSeg: the key or query sequence has more than one segment (the fused Ulysses
// step); with one segment the per-tile addressing reduces to row 128j of map 0.
template <int D, bool kMask, bool kSeg>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ SegMaps tmQ, const __grid_constant__ SegMaps tmK,
                    const __grid_constant__ SegMaps tmV, const __grid_constant__ SeqDesc qd,
                    const __grid_constant__ SeqDesc kd,
                    const uint8_t* __restrict__ key_mask, int mrows, __nv_bfloat16* __restrict__ out,
                    float* __restrict__ lse, int B, int H, int num_items, float scale_log2, DevCtx ctx) {
  using L = FwdLayout<D>;
  constexpr int kChunks = D / 64;
  constexpr int R = L::kRing;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, kBN, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);
  constexpr float kLn2 = 0.6931471805599453f;

  extern __shared__ __align__(1024) uint8_t smem[];
  FwdCtl* ctl = reinterpret_cast<FwdCtl*>(smem + L::kCtl);
  const uint32_t sbase = smem_u32(smem);
  if (sbase & 1023u) {
    // the swizzled operand tiles need 1024-byte alignment; never expected to trigger
    if (threadIdx.x == 0) atomicOr(ctx.status, kStatusBadLaunch);
    return;
  }

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int nqp = (qd.tile0[qd.nseg] + 1) / 2;  // query tile pairs (an item)
  const int nkt = kd.tile0[kd.nseg];             // key tiles
  const int Sk = kd.total;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->bar_q_full, 1);
    mbar_init(&ctl->bar_q_empty, 1);
    for (int s = 0; s < R; ++s) {
      mbar_init(&ctl->bar_kv_full[s], 1);
      mbar_init(&ctl->bar_kv_empty[s], 1);
    }
    for (int w = 0; w < 2; ++w) {
      mbar_init(&ctl->bar_s_full[w], 1);
      mbar_init(&ctl->bar_pv_done[w], 1);
    }
    mbar_init(&ctl->bar_o_free, 256);
    mbar_init(&ctl->bar_final, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == kProducerWarp && lane == 0) {
    for (int p = 0; p < qd.nseg; ++p) tma_prefetch_desc(&tmQ.m[p]);
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
  // Every role takes its per-item tile count from this table, which no one writes after
  // the start, so producer, issuer and softmax walk the same schedule -- after a failure
  // too (the forward's named barriers rely on it).
  int* tile_cnt = reinterpret_cast<int*>(smem + L::kCnt);
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
          const uint8_t* row = key_mask + (size_t)r * Sk + kd.off[kt.seg] + kt.row0;
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
  const size_t o_extent = seq_extent(qd, B, H, D), lse_extent = (size_t)B * H * qd.total;
  // key tiles an item of batch b walks
  auto item_tiles = [&](int b) { return skip ? tile_cnt[b % mrows] : nkt; };

  // Teardown bookkeeping of the producer: uses armed per barrier.
  uint32_t kv_armed[5] = {0, 0, 0, 0, 0};
  uint32_t q_armed = 0;
  bool mma_issued = false;  // set in the issuing lane once it has issued an MMA

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    uint32_t n = 0;   // K/V ring counter across items
    uint32_t ne = 0;  // items with at least one attended key tile (the Q buffer's uses)
    for (int item = blockIdx.x; ok && item < num_items; item += gridDim.x) {
      const Item w = decode_item(item, nqp, H);
      if (item_tiles(w.b) == 0) continue;  // no attended key: the softmax warps write O = 0
      const int mb = w.b % mrows;
      if (lane == 0) {
        if (ne > 0) ok = wait_or_abort(&ctl->bar_q_empty, (ne - 1) & 1, ctx, ctl);
        if (ok) {
          mbar_arrive_expect_tx(&ctl->bar_q_full, 2 * L::kTileBytes);
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            // a tile past the last one reads as zeros (rows past its segment) and is never written
            const SeqTile qt = seq_tile(qd, 2 * w.qp + t);
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(smem + L::kQ + t * L::kTileBytes + c * kChunkBytes, &tmQ.m[qt.seg], &ctl->bar_q_full,
                          c * 64, w.h, qt.row0, w.b);
          }
          q_armed = ne + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      ++ne;
      SeqCursor kseg;  // key segment cursor (tiles are visited in order)
      for (int j = 0; ok && j < nkt; ++j) {
        SeqTile kt;
        if constexpr (kSeg) {
          kt = seq_tile_at(kd, j, kseg);
        } else {
          kt.seg = 0;
          kt.row0 = j * kBN;
          kt.valid = Sk - kt.row0 < kBN ? Sk - kt.row0 : kBN;
        }
        // bit c of word t: key c' = 32t + c of the tile (sequence position off + row0 + c')
        // exists and is attended
        uint32_t words[4] = {0u, 0u, 0u, 0u};
        if (kMask) {
#pragma unroll
          for (int t = 0; t < 4; ++t) {
            const int c = 32 * t + lane;
            const bool valid = c < kt.valid && key_mask[(size_t)mb * Sk + kd.off[kt.seg] + kt.row0 + c] != 0;
            words[t] = __ballot_sync(0xffffffffu, valid);
          }
          // the same test as the tile-count table: the softmax and issuer expect exactly those tiles
          if (skip && (words[0] | words[1] | words[2] | words[3]) == 0) continue;
        }
#pragma unroll
        for (int kind = 0; kind < 2; ++kind, ++n) {  // 0 = K_j, 1 = V_j
          const int slot = n % R;
          const uint32_t use = n / R;
          if (lane == 0 && use > 0) ok = wait_or_abort(&ctl->bar_kv_empty[slot], (use - 1) & 1, ctx, ctl);
          ok = __shfl_sync(0xffffffffu, ok, 0);
          if (!ok) break;
          if (kMask && kind == 1 && lane == 0) {
#pragma unroll
            for (int t = 0; t < 4; ++t) ctl->mask_words[slot][t] = words[t];
          }
          if (lane == 0 && (int)n != ctx.drop_load) {
            mbar_arrive_expect_tx(&ctl->bar_kv_full[slot], L::kTileBytes);
            const int ms = kSeg ? kt.seg : 0;
            const CUtensorMap* map = kind == 0 ? &tmK.m[ms] : &tmV.m[ms];
#pragma unroll
            for (int c = 0; c < kChunks; ++c)
              tma_load_4d(smem + L::kRingOff + slot * L::kTileBytes + c * kChunkBytes, map,
                          &ctl->bar_kv_full[slot], c * 64, w.h, kt.row0, w.b);
            kv_armed[slot] = use + 1;
          }
        }
      }
    }
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ MMA issuer
    // The whole warp runs the schedule (named barriers take whole warps) and
    // computes every UMMA descriptor; one elected lane waits and issues.  Keeping
    // the descriptor arithmetic warp-uniform, outside any lane-divergent branch,
    // keeps each issue short: written as a one-lane branch, an MMA issue took
    // ~80 cycles beside busy softmax warps, more than the 64 the MMA runs.
    // Within an item this warp executes no memory instruction: it learns that
    // P_t is in TMEM from named barrier kBarP + t, which the softmax warpgroup of
    // tile t arrives on.
    uint32_t el_lane;
    const bool el = elect_one_sync(&el_lane);
    bool ok = true;
    uint32_t g = 0;   // global tile counter across items (phase index of s/pv barriers)
    uint32_t ne = 0;  // items with at least one attended key tile (phases of q_full, o_free)
    auto ring_addr = [&](uint32_t n) { return sbase + L::kRingOff + (n % R) * L::kTileBytes; };
    auto issue_s = [&](int t, uint32_t nk) {
      const uint32_t sQ = sbase + L::kQ + t * L::kTileBytes;
      const uint32_t sK = ring_addr(nk);
      const uint32_t d = tmem + (uint32_t)(t * kBN);
      const uint64_t dq0 = sdesc_sw128(sQ, 16, 1024), dk0 = sdesc_sw128(sK, 16, 1024);
#pragma unroll
      for (int kk = 0; kk < D / 16; ++kk) {
        const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
        const uint64_t a = desc_add(dq0, off), b = desc_add(dk0, off);
        if (el) mma_ss_checked(mg, d, a, b, kIdescS, kk > 0, kBN);
      }
      if (el) mma_commit(&ctl->bar_s_full[t]);
    };
    auto issue_pv = [&](int t, uint32_t nv, bool acc) {
      const uint32_t aP = tmem + (uint32_t)(t * kBN);  // P_t: 128 rows x 128 keys bf16 = 64 columns
      const uint32_t sV = ring_addr(nv);
      const uint32_t d = tmem + 256 + (uint32_t)(t * D);
      const uint64_t dv0 = sdesc_sw128(sV, kChunkBytes, 1024);
#pragma unroll
      for (int kk = 0; kk < kBN / 16; ++kk) {
        const uint64_t b = desc_add(dv0, kk * 2048);
        if (el) mma_ts_checked(mg, d, aP + kk * 8, b, kIdescPV, (acc || kk > 0) ? 1u : 0u, D);
      }
      if (el) mma_commit(&ctl->bar_pv_done[t]);
    };
    for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
      // an item without an attended key tile takes no MMA and no barrier
      const int nt = item_tiles(decode_item(item, nqp, H).b);
      if (nt == 0) continue;
      // After a failure anywhere in the CTA this warp stops issuing but still
      // meets the softmax warpgroups at every named barrier of the schedule.
      if (ok && *reinterpret_cast<volatile int*>(&ctl->abort)) ok = false;
      const uint32_t nk = 2 * g;  // K_0 of this item
      if (ok) {
        bool w = true;
        if (el) {
          w = wait_or_abort(&ctl->bar_q_full, ne & 1, ctx, ctl);
          if (w) w = wait_or_abort(&ctl->bar_kv_full[nk % R], (nk / R) & 1, ctx, ctl);
        }
        ok = __shfl_sync(0xffffffffu, w, el_lane);
        if (ok) {
          tc_fence_after();
          issue_s(0, nk);
          issue_s(1, nk);
          if (el) {
            mma_commit(&ctl->bar_kv_empty[nk % R]);
            mma_issued = true;
          }
        }
      }
      for (int j = 0; j < nt; ++j) {
        const uint32_t gj = g + j;
        const uint32_t nv = 2 * gj + 1;
        const bool more = j + 1 < nt;
        const uint32_t nk1 = 2 * (gj + 1);
        // tile 0: PV0_j, then S0_{j+1}.  V_j and K_{j+1} have landed: the softmax
        // warpgroups wait for them before they arrive.
        named_sync(kBarP + 0, kBarPCount);
        if (ok && j == 0 && ne > 0) {
          // the previous item's epilogue must have read O before PV0_0 overwrites it
          bool w = true;
          if (el) w = wait_or_abort(&ctl->bar_o_free, (ne - 1) & 1, ctx, ctl);
          ok = __shfl_sync(0xffffffffu, w, el_lane);
        }
        if (ok) {
          tc_fence_after();
          issue_pv(0, nv, j > 0);
          if (more) issue_s(0, nk1);
        }
        __syncwarp();
        // tile 1: PV1_j, then S1_{j+1}
        named_sync(kBarP + 1, kBarPCount);
        if (ok) {
          tc_fence_after();
          issue_pv(1, nv, j > 0);
          if (el) mma_commit(&ctl->bar_kv_empty[nv % R]);
          if (more) {
            issue_s(1, nk1);
            if (el) mma_commit(&ctl->bar_kv_empty[nk1 % R]);
          }
        }
        __syncwarp();
      }
      // both Q tiles are free once this item's MMAs are done
      if (ok && el) mma_commit(&ctl->bar_q_empty);
      __syncwarp();
      g += nt;
      ++ne;
    }
  } else {
    // ------------------------------------------------------------ softmax warpgroups
    const int t = warp >> 2;                 // query tile of this warpgroup
    const int row = (warp & 3) * 32 + lane;  // TMEM lane = query row within the tile
    const uint32_t tl = tmem + ((uint32_t)((warp & 3) * 32) << 16);
    const uint32_t colS = (uint32_t)(t * kBN);
    const uint32_t colO = 256 + (uint32_t)(t * D);
    bool ok = true;
    uint32_t g = 0;
    for (int item = blockIdx.x; item < num_items; item += gridDim.x) {
      const Item w = decode_item(item, nqp, H);
      const int nt = item_tiles(w.b);
      if (nt == 0) {
        // no attended key for this batch: O = 0 and LSE = -inf, without MMAs or barriers
        const SeqTile qt = seq_tile(qd, 2 * w.qp + t);
        if (row < qt.valid) {
          const int qs = qt.row0 + row;
          const size_t oo = seq_elem(qd, B, H, D, w.b, qt.seg, qs, w.h);
          if (guard_store(ctx, oo, D, o_extent)) {
            __nv_bfloat16* orow = out + oo;
#pragma unroll
            for (int c = 0; c < D / 8; ++c) *reinterpret_cast<uint4*>(orow + 8 * c) = make_uint4(0u, 0u, 0u, 0u);
          }
          const size_t lo = ((size_t)w.b * H + w.h) * qd.total + qd.off[qt.seg] + qs;
          if (guard_store(ctx, lo, 1, lse_extent)) lse[lo] = -INFINITY;
        }
        continue;
      }
      float mu = -INFINITY;  // log2-domain offset in use (scaled max, possibly stale by < 2^8)
      float l_run = 0.f;
      SeqCursor kseg;  // key segment cursor
      for (int j = 0; j < nt; ++j) {
        const uint32_t gj = g + j;
        if (ok) {
          // V_j and K_{j+1}, read by the MMAs that this step's arrival releases,
          // have normally landed long before S_j completes: waiting here keeps
          // these waits off both the issuing thread and the S -> P path
          const uint32_t nv = 2 * gj + 1, nk1 = nv + 1;
          bool okw = wait_or_abort(&ctl->bar_kv_full[nv % R], (nv / R) & 1, ctx, ctl);
          if (okw && j + 1 < nt) okw = wait_or_abort(&ctl->bar_kv_full[nk1 % R], (nk1 / R) & 1, ctx, ctl);
          if (okw) okw = wait_or_abort(&ctl->bar_s_full[t], gj & 1, ctx, ctl);
          ok = __all_sync(0xffffffffu, okw);
        }
        if (!ok) {
          // after a failure: keep meeting the issuer at every step of the schedule;
          // a rendezvous, so this warp never runs a phase ahead of it
          named_sync(kBarP + t, kBarPCount);
          continue;
        }
        tc_fence_after();
        float s[kBN];
        tmem_ld32x2(tl + colS, tl + colS + 32, *reinterpret_cast<float(*)[64]>(&s[0]));
        tmem_ld32x2(tl + colS + 64, tl + colS + 96, *reinterpret_cast<float(*)[64]>(&s[64]));
        if (kMask) {
          // the producer wrote V_j's mask words before arming kv_full, which this
          // warp has already waited on
          const uint32_t nv = 2 * gj + 1;
          uint32_t mw[4];
#pragma unroll
          for (int q = 0; q < 4; ++q) mw[q] = ctl->mask_words[nv % R][q];
          // a tile whose keys are all attended (most tiles of a key-padding mask) needs no bias
          if ((mw[0] & mw[1] & mw[2] & mw[3]) != 0xffffffffu) {
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (!((mw[c >> 5] >> (c & 31)) & 1u)) s[c] = -INFINITY;
          }
        } else {
          // the last tile of a segment is partial: its rows past the segment read as zeros
          const int lim = kSeg ? seq_tile_at(kd, j, kseg).valid : ((j + 1) * kBN > Sk ? Sk - j * kBN : kBN);
          if (lim < kBN) {
#pragma unroll
            for (int c = 0; c < kBN; ++c)
              if (c >= lim) s[c] = -INFINITY;
          }
        }
        // row max over the tile: eight independent chains (the max sits on the
        // critical path between S_t and PV_t), then a short tree
        float m8[8];
#pragma unroll
        for (int q = 0; q < 8; ++q) m8[q] = fmaxf(s[q], s[q + 8]);
#pragma unroll
        for (int c = 16; c < kBN; c += 16)
#pragma unroll
          for (int q = 0; q < 8; ++q) m8[q] = max3(m8[q], s[c + q], s[c + q + 8]);
        const float mt = fmaxf(max3(m8[0], m8[1], m8[2]), max3(max3(m8[3], m8[4], m8[5]), m8[6], m8[7]));
        const float mt2 = mt * scale_log2;  // -inf if every key of the tile is masked
        float alpha = 1.f;
        if (mt2 > mu + kRescaleThreshold) {
          alpha = ex2(mu - mt2);  // 0 when mu = -inf
          mu = mt2;
        }
        const float mu_use = (mu == -INFINITY) ? 0.f : mu;
        // PV_{j-1} of this tile, which reads the P columns about to be overwritten
        // and accumulates the O about to be rescaled, has completed: it was
        // issued before S_j, and the commit behind s_full covers every earlier
        // MMA of the issuing thread.
        const float2 c2 = make_float2(scale_log2, scale_log2);
        const float2 nm2 = make_float2(-mu_use, -mu_use);
        float2 rs2 = make_float2(0.f, 0.f);
#pragma unroll
        for (int hh = 0; hh < 2; ++hh) {
          uint32_t pk[32];
#pragma unroll
          for (int c = 0; c < 32; ++c) {
            const float2 x = fma2(make_float2(s[64 * hh + 2 * c], s[64 * hh + 2 * c + 1]), c2, nm2);
            const float2 e =
                (c % kExpFmaEvery == kExpFmaEvery - 1) ? exp2_fma2(x) : make_float2(ex2(x.x), ex2(x.y));
            rs2 = add2(rs2, e);
            pk[c] = pack_bf16(e.x, e.y);
          }
          // P (bf16 pairs) over the first 64 columns of this tile's S buffer
          tmem_st32_bits(tl + colS + 32 * hh, pk);
        }
        l_run = l_run * alpha + (rs2.x + rs2.y);
        if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
          for (int c = 0; c < D / 32; ++c) {
            float o[32];
            tmem_ld32(tl + colO + 32 * c, o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] *= alpha;
            tmem_st32(tl + colO + 32 * c, o);
          }
        }
        tc_fence_before();
        named_arrive(kBarP + t, kBarPCount);
      }
      if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_pv_done[t], (g + nt - 1) & 1, ctx, ctl));
      if (!ok) {
        g += nt;
        continue;
      }
      tc_fence_after();
      const SeqTile qt = seq_tile(qd, 2 * w.qp + t);
      const bool qvalid = row < qt.valid;
      const int qs = qt.row0 + row;  // row within the query segment
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      const size_t oo = seq_elem(qd, B, H, D, w.b, qt.seg, qvalid ? qs : 0, w.h);
      const bool ostore = qvalid && guard_store(ctx, oo, D, o_extent);
      __nv_bfloat16* orow = out + oo;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tl + colO + 32 * c, o);
        if (ostore) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            uint4 v;
            v.x = pack_bf16(o[8 * i + 0] * inv, o[8 * i + 1] * inv);
            v.y = pack_bf16(o[8 * i + 2] * inv, o[8 * i + 3] * inv);
            v.z = pack_bf16(o[8 * i + 4] * inv, o[8 * i + 5] * inv);
            v.w = pack_bf16(o[8 * i + 6] * inv, o[8 * i + 7] * inv);
            *reinterpret_cast<uint4*>(orow + 32 * c + 8 * i) = v;
          }
        }
      }
      tc_fence_before();
      mbar_arrive(&ctl->bar_o_free);
      if (qvalid) {
        const size_t lo = ((size_t)w.b * H + w.h) * qd.total + qd.off[qt.seg] + qs;
        if (guard_store(ctx, lo, 1, lse_extent)) lse[lo] = l_run > 0.f ? mu * kLn2 + logf(l_run) : -INFINITY;
      }
      g += nt;
    }
  }

  // ------------------------------------------------------------ teardown
  // Waits here ignore the abort flag (they must see in-flight work land) but
  // stay bounded.
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp && mma_issued) {
    // every MMA has completed before TMEM is released
    mma_commit(&ctl->bar_final);
    settle(&ctl->bar_final, 0, ctx);
  }
  if (warp == kProducerWarp && lane == 0) {
    // no TMA write may still be in flight into this CTA's shared memory
    if (q_armed) settle(&ctl->bar_q_full, (q_armed - 1) & 1, ctx);
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

template <int D, bool kMask, bool kSeg>
int launch_fwd(const void* q, const void* k, const void* v, const uint8_t* mask, int mrows, void* out, float* lse,
               int B, const SeqDesc& qd, const SeqDesc& kd, int H, float scale, cudaStream_t stream,
               const DevCtx& ctx) {
  SegMaps mq, mk, mv;
  int st;
  if ((st = encode_seq_maps(&mq, q, qd, B, H, D, 128))) return st;
  if ((st = encode_seq_maps(&mk, k, kd, B, H, D, 128))) return st;
  if ((st = encode_seq_maps(&mv, v, kd, B, H, D, 128))) return st;
  auto kern = attn_fwd_kernel<D, kMask, kSeg>;
  const int smem = FwdLayout<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "uaa_attn_fwd: smem attribute: %s", cudaGetErrorString(e));
  const long long nqp = (qd.tile0[qd.nseg] + 1) / 2;
  const long long items = nqp * H * B;
  if (items > INT32_MAX) return set_error(UAA_ERR_UNSUPPORTED, "uaa_attn_fwd: too many work items");
  const int grid = (int)(items < sm_count() ? items : sm_count());
  kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, qd, kd, mask, mrows, static_cast<__nv_bfloat16*>(out), lse, B,
                                         H, (int)items, scale * kLog2e, ctx);
  return check_launch("uaa_attn_fwd");
}

// mrows: rows of key_mask; batch b uses row b % mrows (mrows = B, or the B batches shared by
// the G head groups of a Ulysses step launched as one batch of G*B)
int fwd_dispatch(const void* q, const void* k, const void* v, const uint8_t* key_mask, int mrows, void* out,
                 float* lse, int B, const SeqDesc& qd, const SeqDesc& kd, int H, int D, float scale, cudaStream_t s,
                 const DevCtx& ctx) {
  const bool seg = qd.nseg > 1 || kd.nseg > 1;
#define UAA_FWD(DD, MM, SS) launch_fwd<DD, MM, SS>(q, k, v, key_mask, mrows, out, lse, B, qd, kd, H, scale, s, ctx)
  if (D == 64) {
    if (seg) return key_mask ? UAA_FWD(64, true, true) : UAA_FWD(64, false, true);
    return key_mask ? UAA_FWD(64, true, false) : UAA_FWD(64, false, false);
  }
  if (seg) return key_mask ? UAA_FWD(128, true, true) : UAA_FWD(128, false, true);
  return key_mask ? UAA_FWD(128, true, false) : UAA_FWD(128, false, false);
#undef UAA_FWD
}

}  // namespace

int validate_attn_sizes(const char* fn, int B, int Sq, int Sk, int H, int D, float scale) {
  if (B < 0 || Sq < 0 || Sk < 0 || H < 0)
    return set_error(UAA_ERR_INVALID_ARG, "%s: negative size B=%d Sq=%d Sk=%d H=%d", fn, B, Sq, Sk, H);
  if (Sq > 0 && Sk == 0) return set_error(UAA_ERR_INVALID_ARG, "%s: queries without keys (Sk = 0)", fn);
  if (D != 64 && D != 128) return set_error(UAA_ERR_UNSUPPORTED, "%s: D=%d (only 64 and 128 are built)", fn, D);
  if (!(scale > 0.f) || !isfinite(scale))
    return set_error(UAA_ERR_INVALID_ARG, "%s: scale must be positive and finite", fn);
  if (B > 65535 || H > 65535) return set_error(UAA_ERR_UNSUPPORTED, "%s: B and H must be <= 65535", fn);
  const uint64_t S = (uint64_t)(Sq > Sk ? Sq : Sk);
  if ((uint64_t)B * S * H * D * 4 >= (1ull << 40))
    return set_error(UAA_ERR_UNSUPPORTED, "%s: tensor larger than the TMA stride range", fn);
  return UAA_OK;
}

int check_dev_ptr(const char* fn, const char* name, const void* p) {
  if (!p) return set_error(UAA_ERR_INVALID_ARG, "%s: %s is NULL", fn, name);
  if (reinterpret_cast<uintptr_t>(p) & 15u)
    return set_error(UAA_ERR_INVALID_ARG, "%s: %s is not 16-byte aligned", fn, name);
  return UAA_OK;
}

}  // namespace uaa

using namespace uaa;

extern "C" int uaa_attn_fwd_cross(const void* q, const void* k, const void* v, const uint8_t* key_mask, void* out,
                                  float* lse, int B, int Sq, int Sk, int H, int D, float scale, uaa_stream_t stream) {
  const char* fn = "uaa_attn_fwd";
  int st = validate_attn_sizes(fn, B, Sq, Sk, H, D, scale);
  if (st) return st;
  if ((uint64_t)B * Sq * H == 0) return UAA_OK;
  if ((st = check_dev_ptr(fn, "q", q)) || (st = check_dev_ptr(fn, "k", k)) || (st = check_dev_ptr(fn, "v", v)) ||
      (st = check_dev_ptr(fn, "out", out)))
    return st;
  if (!lse) return set_error(UAA_ERR_INVALID_ARG, "%s: lse is NULL", fn);
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return set_error(UAA_ERR_INVALID_ARG, "%s: lse is not 4-byte aligned", fn);
  DevCtx ctx;
  if ((st = get_dev_ctx(&ctx))) return st;
  return fwd_dispatch(q, k, v, key_mask, B, out, lse, B, seq_plain(Sq), seq_plain(Sk), H, D, scale,
                      static_cast<cudaStream_t>(stream), ctx);
}

extern "C" int uaa_attn_fwd(const void* q, const void* k, const void* v, const uint8_t* key_mask, void* out,
                            float* lse, int B, int S, int H, int D, float scale, uaa_stream_t stream) {
  return uaa_attn_fwd_cross(q, k, v, key_mask, out, lse, B, S, S, H, D, scale, stream);
}

extern "C" int uaa_attn_fwd_groups(const void* q, const void* k, const void* v, const uint8_t* key_mask, void* out,
                                   float* lse, int G, int B, int S, int H, int D, float scale, uaa_stream_t stream) {
  const char* fn = "uaa_attn_fwd_groups";
  if (G < 1 || B < 0) return set_error(UAA_ERR_INVALID_ARG, "%s: G=%d, B=%d", fn, G, B);
  if ((long long)G * B > 65535) return set_error(UAA_ERR_UNSUPPORTED, "%s: G*B must be <= 65535", fn);
  int st = validate_attn_sizes(fn, G * B, S, S, H, D, scale);
  if (st) return st;
  if ((uint64_t)B * S * H == 0) return UAA_OK;
  if ((st = check_dev_ptr(fn, "q", q)) || (st = check_dev_ptr(fn, "k", k)) || (st = check_dev_ptr(fn, "v", v)) ||
      (st = check_dev_ptr(fn, "out", out)))
    return st;
  if (!lse || (reinterpret_cast<uintptr_t>(lse) & 3u))
    return set_error(UAA_ERR_INVALID_ARG, "%s: lse is NULL or not 4-byte aligned", fn);
  DevCtx ctx;
  if ((st = get_dev_ctx(&ctx))) return st;
  return fwd_dispatch(q, k, v, key_mask, B, out, lse, G * B, seq_plain(S), seq_plain(S), H, D, scale,
                      static_cast<cudaStream_t>(stream), ctx);
}

extern "C" int uaa_ulysses_attn_fwd(const void* q, const void* k, const void* v, const uint8_t* key_mask, void* out,
                                    float* lse, int P, const int* shard_lens, int cap, int B, int H, int D, float scale,
                                    uaa_stream_t stream) {
  const char* fn = "uaa_ulysses_attn_fwd";
  SeqDesc sd;
  int st = seq_sharded(&sd, P, shard_lens, cap, fn);
  if (st) return st;
  if ((st = validate_attn_sizes(fn, B, sd.total, sd.total, H, D, scale))) return st;
  if ((uint64_t)B * H == 0) return UAA_OK;
  if ((st = check_dev_ptr(fn, "q", q)) || (st = check_dev_ptr(fn, "k", k)) || (st = check_dev_ptr(fn, "v", v)) ||
      (st = check_dev_ptr(fn, "out", out)))
    return st;
  if (sd.total > 0 && !lse) return set_error(UAA_ERR_INVALID_ARG, "%s: lse is NULL", fn);
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return set_error(UAA_ERR_INVALID_ARG, "%s: lse is not 4-byte aligned", fn);
  if ((uint64_t)P * B * cap * H * D * 4 >= (1ull << 40))
    return set_error(UAA_ERR_UNSUPPORTED, "%s: tensor larger than the TMA stride range", fn);
  DevCtx ctx;
  if ((st = get_dev_ctx(&ctx))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  // padding rows of the output shards are zero, as after the head->seq exchange
  if ((st = zero_pad_rows(out, sd, B, H, D, s))) return st;
  if (sd.total == 0) return UAA_OK;
  return fwd_dispatch(q, k, v, key_mask, B, out, lse, B, sd, sd, H, D, scale, s, ctx);
}
