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
// Design (one CTA = one 128-row query tile of one (batch, head)):
//   warp 4     TMA producer: Q once, then K/V tiles of 128 keys into a
//              2-stage ring (128-byte swizzled, 64 columns per box); with a
//              mask it also packs the tile's 128 mask bits into shared memory.
//   warp 5     tcgen05 issuer (one thread): S_j = Q K_j^T into one of two
//              TMEM S buffers (S_{j+1} is issued before P_j is ready, so the
//              tensor core overlaps the softmax), then O += P_j V_j into a
//              TMEM O accumulator; completion is signalled with tcgen05.commit.
//   warps 0-3  softmax: thread r owns query row r (TMEM lane r), so the row
//              max and row sum are thread-local; online softmax in base 2,
//              P_j written as bf16 to shared memory (K-major, swizzled) as the
//              A operand of the PV MMA; O rescaled in TMEM when the running
//              max moves; epilogue O / l -> bf16, LSE = m*scale + ln l.
// TMEM columns: [0,128) S buffer 0, [128,256) S buffer 1, [256,256+D) O.
#include <math.h>

#include "uaa_common.cuh"

namespace uaa {
namespace {

constexpr int kBM = 128;  // query rows per CTA (TMEM lanes)
constexpr int kBN = 128;  // keys per K/V tile
constexpr int kKStages = 2;
constexpr int kVStages = 2;
constexpr int kChunkBytes = 128 * 128;  // 128 rows x 128 bytes (one swizzle column block)
constexpr int kThreads = 192;

template <int D>
struct FwdLayout {
  static constexpr int kTileBytes = 128 * D * 2;
  static constexpr int kQ = 0;
  static constexpr int kK = kQ + kTileBytes;
  static constexpr int kV = kK + kKStages * kTileBytes;
  static constexpr int kP = kV + kVStages * kTileBytes;
  static constexpr int kCtl = kP + kBM * kBN * 2;
  static constexpr int kBytes = kCtl + 256;
  // keep one CTA per SM (the 512 TMEM columns are allocated whole)
  static constexpr int kSmem = (kBytes + 1024 > 120 * 1024) ? kBytes + 1024 : 120 * 1024;
};

struct FwdCtl {
  uint64_t bar_q;
  uint64_t bar_k_full[kKStages];
  uint64_t bar_k_empty[kKStages];
  uint64_t bar_v_full[kVStages];
  uint64_t bar_v_empty[kVStages];
  uint64_t bar_s_full[2];
  uint64_t bar_p_full;
  uint64_t bar_o_full;
  uint64_t bar_final;
  uint32_t tmem_base;
  int abort;
  uint32_t mask_words[kVStages][4];
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ uint32_t pack_bf16(float a, float b) {
  __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
  return *reinterpret_cast<uint32_t*>(&v);
}

__device__ __forceinline__ bool wait_or_abort(uint64_t* bar, uint32_t parity, const DevCtx& ctx, FwdCtl* ctl) {
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

// Bounded wait used during teardown: does not give up on the abort flag.
__device__ __forceinline__ void settle(uint64_t* bar, uint32_t parity, const DevCtx& ctx) {
  if (!mbar_wait(bar, parity, ctx.timeout_ns)) atomicOr(ctx.status, kStatusTimeout);
}

template <int D, bool kMask>
__global__ void __launch_bounds__(kThreads, 1)
    attn_fwd_kernel(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                    const __grid_constant__ CUtensorMap tmV, const uint8_t* __restrict__ key_mask,
                    __nv_bfloat16* __restrict__ out, float* __restrict__ lse, int S, int H, float scale,
                    float scale_log2, DevCtx ctx) {
  using L = FwdLayout<D>;
  constexpr int kChunks = D / 64;
  constexpr uint32_t kIdescS = idesc_bf16_f32(128, kBN, false, false);
  constexpr uint32_t kIdescPV = idesc_bf16_f32(128, D, false, true);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  FwdCtl* ctl = reinterpret_cast<FwdCtl*>(smem + L::kCtl);
  const uint32_t sbase = smem_u32(smem);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int qt = blockIdx.x;
  const int h = blockIdx.y;
  const int b = blockIdx.z;
  const int q0 = qt * kBM;
  const int nkt = (S + kBN - 1) / kBN;

  if (threadIdx.x == 0) {
    mbar_init(&ctl->bar_q, 1);
    for (int s = 0; s < kKStages; ++s) {
      mbar_init(&ctl->bar_k_full[s], 1);
      mbar_init(&ctl->bar_k_empty[s], 1);
    }
    for (int s = 0; s < kVStages; ++s) {
      mbar_init(&ctl->bar_v_full[s], 1);
      mbar_init(&ctl->bar_v_empty[s], 1);
    }
    mbar_init(&ctl->bar_s_full[0], 1);
    mbar_init(&ctl->bar_s_full[1], 1);
    mbar_init(&ctl->bar_p_full, 4 * 32);
    mbar_init(&ctl->bar_o_full, 1);
    mbar_init(&ctl->bar_final, 1);
    ctl->abort = 0;
    fence_mbar_init();
  }
  if (warp == 4 && lane == 0) {
    tma_prefetch_desc(&tmQ);
    tma_prefetch_desc(&tmK);
    tma_prefetch_desc(&tmV);
  }
  if (warp == 5) {
    tmem_alloc(&ctl->tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = ctl->tmem_base;

  // Teardown bookkeeping of the producer: uses armed per stage.
  uint32_t k_armed[kKStages] = {0, 0};
  uint32_t v_armed[kVStages] = {0, 0};
  bool q_armed = false;
  bool mma_issued = false;

  if (warp == 4) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    if (lane == 0) {
      mbar_arrive_expect_tx(&ctl->bar_q, L::kTileBytes);
#pragma unroll
      for (int c = 0; c < kChunks; ++c) tma_load_4d(smem + L::kQ + c * kChunkBytes, &tmQ, &ctl->bar_q, c * 64, h, q0, b);
      q_armed = true;
    }
    for (int j = 0; j < nkt; ++j) {
      const int ks = j % kKStages;
      const uint32_t ku = j / kKStages;
      if (lane == 0) {
        if (ku > 0) ok = wait_or_abort(&ctl->bar_k_empty[ks], (ku - 1) & 1, ctx, ctl);
        if (ok) {
          mbar_arrive_expect_tx(&ctl->bar_k_full[ks], L::kTileBytes);
#pragma unroll
          for (int c = 0; c < kChunks; ++c)
            tma_load_4d(smem + L::kK + ks * L::kTileBytes + c * kChunkBytes, &tmK, &ctl->bar_k_full[ks], c * 64, h,
                        j * kBN, b);
          k_armed[ks] = ku + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      const int vs = j % kVStages;
      const uint32_t vu = j / kVStages;
      if (lane == 0 && vu > 0) ok = wait_or_abort(&ctl->bar_v_empty[vs], (vu - 1) & 1, ctx, ctl);
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      if (kMask) {
        // bit c of word t = key j*128 + 32t + c is attended
        uint32_t words[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) {
          const int key = j * kBN + 32 * t + lane;
          const bool valid = key < S && key_mask[(size_t)b * S + key] != 0;
          words[t] = __ballot_sync(0xffffffffu, valid);
        }
        if (lane == 0) {
#pragma unroll
          for (int t = 0; t < 4; ++t) ctl->mask_words[vs][t] = words[t];
        }
        __syncwarp();
      }
      if (lane == 0) {
        mbar_arrive_expect_tx(&ctl->bar_v_full[vs], L::kTileBytes);
#pragma unroll
        for (int c = 0; c < kChunks; ++c)
          tma_load_4d(smem + L::kV + vs * L::kTileBytes + c * kChunkBytes, &tmV, &ctl->bar_v_full[vs], c * 64, h,
                      j * kBN, b);
        v_armed[vs] = vu + 1;
      }
    }
  } else if (warp == 5) {
    // ------------------------------------------------------------ MMA issuer
    if (lane == 0) {
      bool ok = wait_or_abort(&ctl->bar_q, 0, ctx, ctl);
      tc_fence_after();
      const uint32_t sQ = sbase + L::kQ;
      const uint32_t sP = sbase + L::kP;
      auto issue_s = [&](int j) -> bool {
        const int ks = j % kKStages;
        const uint32_t ku = j / kKStages;
        if (!wait_or_abort(&ctl->bar_k_full[ks], ku & 1, ctx, ctl)) return false;
        tc_fence_after();
        const uint32_t sK = sbase + L::kK + ks * L::kTileBytes;
        const uint32_t d = tmem + (uint32_t)((j & 1) * kBN);
#pragma unroll
        for (int kk = 0; kk < D / 16; ++kk) {
          const uint32_t off = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          mma_bf16(d, sdesc_sw128(sQ + off, 16, 1024), sdesc_sw128(sK + off, 16, 1024), kIdescS, kk > 0);
        }
        mma_commit(&ctl->bar_k_empty[ks]);
        mma_commit(&ctl->bar_s_full[j & 1]);
        mma_issued = true;
        return true;
      };
      if (ok) ok = issue_s(0);
      for (int j = 0; ok && j < nkt; ++j) {
        if (j + 1 < nkt && !(ok = issue_s(j + 1))) break;
        if (!(ok = wait_or_abort(&ctl->bar_p_full, j & 1, ctx, ctl))) break;
        tc_fence_after();
        const int vs = j % kVStages;
        if (!(ok = wait_or_abort(&ctl->bar_v_full[vs], (j / kVStages) & 1, ctx, ctl))) break;
        tc_fence_after();
        const uint32_t sV = sbase + L::kV + vs * L::kTileBytes;
#pragma unroll
        for (int kk = 0; kk < kBN / 16; ++kk) {
          const uint32_t aoff = (kk >> 2) * kChunkBytes + (kk & 3) * 32;
          mma_bf16(tmem + 256, sdesc_sw128(sP + aoff, 16, 1024), sdesc_sw128(sV + kk * 2048, kChunkBytes, 1024),
                   kIdescPV, (j > 0 || kk > 0) ? 1u : 0u);
        }
        mma_commit(&ctl->bar_v_empty[vs]);
        mma_commit(&ctl->bar_o_full);
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps 0..3
    const int row = warp * 32 + lane;
    const uint32_t tl = tmem + ((uint32_t)(warp * 32) << 16);
    uint8_t* sP = smem + L::kP;
    float m_run = -INFINITY;
    float l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < nkt; ++j) {
      const int sb = j & 1;
      ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_s_full[sb], (j >> 1) & 1, ctx, ctl));
      if (!ok) break;
      tc_fence_after();
      float s[kBN];
#pragma unroll
      for (int c = 0; c < kBN / 32; ++c)
        tmem_ld32(tl + sb * kBN + 32 * c, *reinterpret_cast<float(*)[32]>(&s[32 * c]));
      if (kMask) {
        const int vs = j % kVStages;
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_v_full[vs], (j / kVStages) & 1, ctx, ctl));
        if (!ok) break;
        uint32_t w[4];
#pragma unroll
        for (int t = 0; t < 4; ++t) w[t] = ctl->mask_words[vs][t];
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (!((w[c >> 5] >> (c & 31)) & 1u)) s[c] = -INFINITY;
      } else if ((j + 1) * kBN > S) {
        const int lim = S - j * kBN;
#pragma unroll
        for (int c = 0; c < kBN; ++c)
          if (c >= lim) s[c] = -INFINITY;
      }
      float mt = s[0];
#pragma unroll
      for (int c = 1; c < kBN; ++c) mt = fmaxf(mt, s[c]);
      const float m_new = fmaxf(m_run, mt);
      const float m_use = (m_new == -INFINITY) ? 0.f : m_new * scale_log2;
      const float alpha = ex2(m_run * scale_log2 - m_use);
      float rs = 0.f;
#pragma unroll
      for (int c = 0; c < kBN; ++c) {
        s[c] = ex2(fmaf(s[c], scale_log2, -m_use));
        rs += s[c];
      }
      l_run = l_run * alpha + rs;
      m_run = m_new;
      if (j > 0) {
        // PV_{j-1} must be done before P is overwritten and O is rescaled
        ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_o_full, (j - 1) & 1, ctx, ctl));
        if (!ok) break;
        tc_fence_after();
      }
#pragma unroll
      for (int ch = 0; ch < kBN / 64; ++ch) {
#pragma unroll
        for (int pc = 0; pc < 8; ++pc) {
          const float* src = &s[ch * 64 + pc * 8];
          uint4 v;
          v.x = pack_bf16(src[0], src[1]);
          v.y = pack_bf16(src[2], src[3]);
          v.z = pack_bf16(src[4], src[5]);
          v.w = pack_bf16(src[6], src[7]);
          *reinterpret_cast<uint4*>(sP + ch * kChunkBytes + row * 128 + ((pc ^ (row & 7)) << 4)) = v;
        }
      }
      if (j > 0 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll 1
        for (int c = 0; c < D / 32; ++c) {
          float o[32];
          tmem_ld32(tl + 256 + 32 * c, o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] *= alpha;
          tmem_st32(tl + 256 + 32 * c, o);
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&ctl->bar_p_full);
    }
    if (ok) ok = __all_sync(0xffffffffu, wait_or_abort(&ctl->bar_o_full, (nkt - 1) & 1, ctx, ctl));
    if (ok) {
      tc_fence_after();
      const int q = q0 + row;
      const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
      __nv_bfloat16* orow = out + (((size_t)b * S + q) * H + h) * D;
#pragma unroll 1
      for (int c = 0; c < D / 32; ++c) {
        float o[32];
        tmem_ld32(tl + 256 + 32 * c, o);
        if (q < S) {
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
      if (q < S) lse[((size_t)b * H + h) * S + q] = l_run > 0.f ? m_run * scale + logf(l_run) : -INFINITY;
    }
  }

  // ------------------------------------------------------------ teardown
  // Waits here ignore the abort flag (they must see in-flight work land) but
  // stay bounded.
  tc_fence_before();
  __syncthreads();
  if (warp == 5 && lane == 0 && mma_issued) {
    // every MMA has completed before TMEM is released
    mma_commit(&ctl->bar_final);
    settle(&ctl->bar_final, 0, ctx);
  }
  if (warp == 4 && lane == 0) {
    // no TMA write may still be in flight into this CTA's shared memory
    if (q_armed) settle(&ctl->bar_q, 0, ctx);
    for (int s = 0; s < kKStages; ++s)
      if (k_armed[s]) settle(&ctl->bar_k_full[s], (k_armed[s] - 1) & 1, ctx);
    for (int s = 0; s < kVStages; ++s)
      if (v_armed[s]) settle(&ctl->bar_v_full[s], (v_armed[s] - 1) & 1, ctx);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 5) {
    tc_fence_after();
    tmem_dealloc(tmem, 512);
  }
}

template <int D, bool kMask>
int launch_fwd(const void* q, const void* k, const void* v, const uint8_t* mask, void* out, float* lse, int B,
               int S, int H, float scale, cudaStream_t stream, const DevCtx& ctx) {
  CUtensorMap mq, mk, mv;
  int st;
  if ((st = encode_bshd_map(&mq, q, B, S, H, D, 128))) return st;
  if ((st = encode_bshd_map(&mk, k, B, S, H, D, 128))) return st;
  if ((st = encode_bshd_map(&mv, v, B, S, H, D, 128))) return st;
  auto kern = attn_fwd_kernel<D, kMask>;
  const int smem = FwdLayout<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return set_error(UAA_ERR_CUDA, "uaa_attn_fwd: smem attribute: %s", cudaGetErrorString(e));
  dim3 grid((S + kBM - 1) / kBM, H, B);
  kern<<<grid, kThreads, smem, stream>>>(mq, mk, mv, mask, static_cast<__nv_bfloat16*>(out), lse, S, H, scale,
                                         scale * kLog2e, ctx);
  return check_launch("uaa_attn_fwd");
}

}  // namespace

int validate_attn_sizes(const char* fn, int B, int S, int H, int D, float scale) {
  if (B < 0 || S < 0 || H < 0) return set_error(UAA_ERR_INVALID_ARG, "%s: negative size B=%d S=%d H=%d", fn, B, S, H);
  if (D != 64 && D != 128) return set_error(UAA_ERR_UNSUPPORTED, "%s: D=%d (only 64 and 128 are built)", fn, D);
  if (!(scale > 0.f) || !isfinite(scale))
    return set_error(UAA_ERR_INVALID_ARG, "%s: scale must be positive and finite", fn);
  if (B > 65535 || H > 65535) return set_error(UAA_ERR_UNSUPPORTED, "%s: B and H must be <= 65535", fn);
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

extern "C" int uaa_attn_fwd(const void* q, const void* k, const void* v, const uint8_t* key_mask, void* out,
                            float* lse, int B, int S, int H, int D, float scale, uaa_stream_t stream) {
  const char* fn = "uaa_attn_fwd";
  int st = validate_attn_sizes(fn, B, S, H, D, scale);
  if (st) return st;
  if ((uint64_t)B * S * H == 0) return UAA_OK;
  if ((st = check_dev_ptr(fn, "q", q)) || (st = check_dev_ptr(fn, "k", k)) || (st = check_dev_ptr(fn, "v", v)) ||
      (st = check_dev_ptr(fn, "out", out)))
    return st;
  if (!lse) return set_error(UAA_ERR_INVALID_ARG, "%s: lse is NULL", fn);
  if (reinterpret_cast<uintptr_t>(lse) & 3u) return set_error(UAA_ERR_INVALID_ARG, "%s: lse is not 4-byte aligned", fn);
  DevCtx ctx;
  if ((st = get_dev_ctx(&ctx))) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (D == 64)
    return key_mask ? launch_fwd<64, true>(q, k, v, key_mask, out, lse, B, S, H, scale, s, ctx)
                    : launch_fwd<64, false>(q, k, v, key_mask, out, lse, B, S, H, scale, s, ctx);
  return key_mask ? launch_fwd<128, true>(q, k, v, key_mask, out, lse, B, S, H, scale, s, ctx)
                  : launch_fwd<128, false>(q, k, v, key_mask, out, lse, B, S, H, scale, s, ctx);
}
