/*
 * uaa.h -- C ABI of the GB300 (sm_103a) Ulysses DiT attention library.
 *
 * The library implements the data-parallel hot path discussed in three
 * pull-request pages:
 *   - "[attention] Add Ulysses Anything backward" (diffusers PR 14834),
 *     cited below as "UAA-bwd";
 *   - "Add fast-ulysses attention backend" (LightX2V PR 1234), "fast-ulysses";
 *   - "Fix double transpose of K/V in templated attention backward"
 *     (diffusers PR 14341), "double-transpose".
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Attention tensors are BSHD: (B, S, H, D) contiguous, bf16, row stride
 *    H*D elements.  The forward op returns its output in BSHD and the backward
 *    consumes Q, K, V in that same layout ("double-transpose", description).
 *  - D must be 64 or 128.  Non-causal, no dropout ("double-transpose",
 *    Not verified: non-causal, no dropout).
 *  - lse is fp32 (B, H, S): the natural log of sum_j exp(scale*q.k_j + bias_j).
 *  - key_mask is an optional uint8 (B, S) array, nonzero = attend.  It is the
 *    head-broadcast (B, 1, 1, S) key-padding mask ("UAA-bwd", Unsupported cases,
 *    per-head masks) and acts as an additive 0 / -inf bias
 *    ("double-transpose", follow-up item 2).  A query row whose keys are all
 *    masked gets O = 0, LSE = -inf and no gradient.  Key tiles (128 keys)
 *    without an attended key cost no tensor work as long as the mask has at
 *    most 256 rows (each kernel tabulates the rows' attended tiles when it
 *    starts); with more rows the forward and the dQ pass compute every tile,
 *    masked keys at P = 0 (same results).
 *  - All pointers marked "device" are device memory owned by the caller; the
 *    library never allocates or frees device memory.  Host arrays
 *    (shard_lens) are read during the call only.
 *  - Work is enqueued on `stream` and is asynchronous; nothing synchronises
 *    the stream except uaa_check_device_status().
 *  - Every entry point validates its arguments on the host first.  A negative
 *    status from validation means nothing was launched.  The message for the
 *    last non-OK status of the calling thread is in uaa_last_error().
 *  - Device-side waits (mbarrier / TMA / tensor-core completion) are bounded.
 *    A wait that runs out records UAA_ERR_TIMEOUT in a device status word and
 *    the kernel returns; uaa_check_device_status() reports and clears it.  The
 *    give-up is scoped to the call whose wait ran out: its other CTAs and
 *    kernels stop waiting too (their outputs are then incomplete), while later
 *    calls run normally even before the status has been read.  The calls
 *    themselves cannot see a timeout of their own kernels (they return before
 *    the kernels run): only uaa_check_device_status() reports it.
 *
 * Pointer alignment: every device pointer must be 16-byte aligned (the TMA
 * loads and the 16-byte vector copies need it).
 */
#ifndef UAA_H_
#define UAA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* CUDA stream handle (cudaStream_t / CUstream); 0 = the legacy default stream. */
typedef void* uaa_stream_t;

typedef enum {
  UAA_OK = 0,
  UAA_ERR_INVALID_ARG = -1,   /* bad pointer, size, shape or alignment */
  UAA_ERR_UNSUPPORTED = -2,   /* valid request outside what is built (e.g. D not 64/128) */
  UAA_ERR_PER_HEAD_MASK = -3, /* a (B, H>1, 1, S) mask: Ulysses cannot shard it ("UAA-bwd",
                                 What does this PR do: fail fast on per-head masks) */
  UAA_ERR_CUDA = -4,          /* a CUDA runtime / driver call failed */
  UAA_ERR_TIMEOUT = -5,       /* a bounded device-side wait ran out (reported by
                                 uaa_check_device_status) */
  UAA_ERR_DEBUG_CHECK = -6    /* debug builds only: a device-side range check failed
                                 and its access was skipped (uaa_check_device_status) */
} uaa_status;

/* Attention forward.
 * "double-transpose", description: the forward op returns out in BSHD and the
 * backward needs the log-sum-exp; its follow-up item 1 shows what goes wrong
 * when the LSE is not computed, so this call ALWAYS writes lse (no flag).
 *   q, k, v  : device, bf16 (B, S, H, D)
 *   key_mask : device, uint8 (B, S) or NULL (no mask)
 *   out      : device, bf16 (B, S, H, D)
 *   lse      : device, fp32 (B, H, S)
 *   scale    : softmax scale applied to q.k (the usual value is 1/sqrt(D))
 * Returns UAA_OK or a negative uaa_status. */
int uaa_attn_fwd(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                 void* out, float* lse, int B, int S, int H, int D, float scale,
                 uaa_stream_t stream);

/* Attention forward with separate query and key lengths (cross-attention, or a
 * query block against a key set of another length).  "UAA-bwd", What does
 * this PR do: the query and key partition metadata are saved separately, so
 * the query and key sequences can be sharded -- and be as long -- differently.
 *   q        : device, bf16 (B, Sq, H, D)
 *   k, v     : device, bf16 (B, Sk, H, D)
 *   key_mask : device, uint8 (B, Sk) or NULL
 *   out      : device, bf16 (B, Sq, H, D); lse : device, fp32 (B, H, Sq)
 * Sk must be positive when Sq is.  uaa_attn_fwd(..., S, ...) is this call with
 * Sq = Sk = S.  Returns UAA_OK or a negative uaa_status. */
int uaa_attn_fwd_cross(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                       void* out, float* lse, int B, int Sq, int Sk, int H, int D, float scale,
                       uaa_stream_t stream);

/* Bytes of device workspace uaa_attn_bwd needs for (B, S, H, D): two fp32
 * (B, H, S_pad) vectors, S_pad = S rounded up to a multiple of 128 -- the row
 * dot Delta = rowsum(dO * O) and -LSE * log2(e) -- rounded up to 256 bytes.
 * Returns 0 for invalid sizes. */
size_t uaa_attn_bwd_workspace_bytes(int B, int S, int H, int D);

/* Attention backward: dQ, dK, dV from dO, O and LSE.
 * "double-transpose", description: the backward op receives Q, K, V in one
 * layout (no second transpose of K/V), dO in BSHD and the saved LSE.
 * The result is deterministic (no atomics): two calls on the same inputs give
 * identical bits.
 *   q, k, v, out, dout : device, bf16 (B, S, H, D)
 *   lse                : device, fp32 (B, H, S), as written by uaa_attn_fwd
 *   key_mask           : device, uint8 (B, S) or NULL; must be the mask the
 *                        forward used.  Masked keys get dK = dV = 0 exactly.
 *   dq, dk, dv         : device, bf16 (B, S, H, D), written (not accumulated)
 *   workspace          : device, at least uaa_attn_bwd_workspace_bytes() bytes,
 *                        256-byte aligned; contents on entry are ignored
 * Returns UAA_OK or a negative uaa_status. */
int uaa_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                 const void* dout, const float* lse, const uint8_t* key_mask,
                 void* dq, void* dk, void* dv, int B, int S, int H, int D, float scale,
                 void* workspace, size_t workspace_bytes, uaa_stream_t stream);

/* Attention backward with separate query and key lengths (the backward of
 * uaa_attn_fwd_cross; "UAA-bwd", What does this PR do: dQ follows the query
 * partition, dK/dV the key partition).
 *   q, out, dout, dq : device, bf16 (B, Sq, H, D); lse : fp32 (B, H, Sq)
 *   k, v, dk, dv     : device, bf16 (B, Sk, H, D); key_mask : uint8 (B, Sk) or NULL
 *   workspace        : at least uaa_attn_bwd_workspace_bytes(B, Sq, H, D) bytes
 * Sq and Sk must both be positive (or B*H = 0).  uaa_attn_bwd(..., S, ...) is
 * this call with Sq = Sk = S.  Returns UAA_OK or a negative uaa_status. */
int uaa_attn_bwd_cross(const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, const uint8_t* key_mask,
                       void* dq, void* dk, void* dv, int B, int Sq, int Sk, int H, int D,
                       float scale, void* workspace, size_t workspace_bytes, uaa_stream_t stream);

/* Workspace of uaa_attn_bwd_fused: the two fp32 row vectors of
 * uaa_attn_bwd_workspace_bytes() followed by an fp32 (B, H, S_pad, D) dQ
 * accumulator (S_pad = S rounded up to 128), rounded up to 256 bytes.
 * Returns 0 for invalid sizes. */
size_t uaa_attn_bwd_fused_workspace_bytes(int B, int S, int H, int D);

/* Attention backward in one K/V-tile-major pass: same arguments and results
 * as uaa_attn_bwd, but each (query tile, key tile) pair's dQ contribution dS K
 * is a fifth GEMM of the same kernel, added into an fp32 dQ accumulator with
 * vector reductions (red.global.add) and converted to bf16 at the end -- the
 * five GEMMs of the gradient are each done once, where uaa_attn_bwd recomputes
 * S and dP in a separate dQ pass (seven GEMMs).  The order of the dQ additions
 * varies from run to run, so dQ is not bit-for-bit reproducible (dK and dV
 * are); use uaa_attn_bwd where reproducible gradients are required.
 * "double-transpose", description (the backward op contract); the pages leave
 * open how dQ is formed.
 *   workspace : at least uaa_attn_bwd_fused_workspace_bytes(B, S, H, D) bytes,
 *               256-byte aligned; contents on entry are ignored
 * Returns UAA_OK or a negative uaa_status. */
int uaa_attn_bwd_fused(const void* q, const void* k, const void* v, const void* out,
                       const void* dout, const float* lse, const uint8_t* key_mask,
                       void* dq, void* dk, void* dv, int B, int S, int H, int D, float scale,
                       void* workspace, size_t workspace_bytes, uaa_stream_t stream);

/* Attention of the G head groups of one Ulysses step, launched together.
 * "UAA-bwd", What does this PR do: after the seq->head exchange every rank runs
 * the plain attention on its head group with the full key-padding mask; on one
 * device the G groups are G batches of B sequences each, and all of them share
 * the same B mask rows.
 *   q, k, v, out : device, bf16 (G*B, S, H, D) -- batch g*B + b is sequence b of group g
 *   key_mask     : device, uint8 (B, S) or NULL; batch g*B + b uses row b
 *   lse          : device, fp32 (G*B, H, S)
 * Equals G calls of uaa_attn_fwd, one per group, bit for bit.  G >= 1,
 * G*B <= 65535.  Returns UAA_OK or a negative uaa_status. */
int uaa_attn_fwd_groups(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                        void* out, float* lse, int G, int B, int S, int H, int D, float scale,
                        uaa_stream_t stream);

/* Backward of uaa_attn_fwd_groups (same layouts; the mask rows are shared the
 * same way).  workspace: at least uaa_attn_bwd_workspace_bytes(G*B, S, H, D)
 * bytes, 256-byte aligned.  Equals G calls of uaa_attn_bwd bit for bit.
 * Returns UAA_OK or a negative uaa_status. */
int uaa_attn_bwd_groups(const void* q, const void* k, const void* v, const void* out,
                        const void* dout, const float* lse, const uint8_t* key_mask,
                        void* dq, void* dk, void* dv, int G, int B, int S, int H, int D,
                        float scale, void* workspace, size_t workspace_bytes, uaa_stream_t stream);

/* Profiling aid (off by default; the pages have no counterpart): when the
 * three CUDA events (cudaEvent_t, created by the caller) are non-NULL, every
 * later uaa_attn_bwd call of the calling thread records `before_dkdv` just
 * before its dK/dV kernel, `after_dkdv` between the dK/dV and dQ kernels and
 * `after_dq` after the dQ kernel, on the call's stream, so each kernel can be
 * timed on its own.  Pass NULLs to stop.  The events stay owned by the caller. */
void uaa_set_bwd_profile_events(void* before_dkdv, void* after_dkdv, void* after_dq);

/* Allocation-free variant of uaa_attn_bwd.  The source pages have no
 * counterpart; this entry point exists for callers that cannot allocate device
 * memory when they run the backward -- code running inside an allocator
 * callback, plugins that may only enqueue work on a stream they were handed,
 * runtimes whose device allocations are all planned up front, latency-bound
 * loops that must not take the allocator's locks -- and so cannot provide the
 * workspace uaa_attn_bwd asks for.
 *
 * It computes exactly what uaa_attn_bwd computes (same arguments minus the
 * workspace) but uses a scratch array built into the library: a file-scope
 * device array of uaa_attn_bwd_noalloc_max_bytes() bytes (64 MiB), which every
 * GPU that loads the library holds until the process exits.  Requests whose
 * uaa_attn_bwd_workspace_bytes(B, S, H, D) exceeds that size are rejected
 * with UAA_ERR_UNSUPPORTED (use uaa_attn_bwd instead).  The call itself never
 * allocates or frees device memory.
 *  - The first call on each device looks up the array's device address (with
 *    that device current) and caches it; make that first call before any
 *    stream capture begins.  The cached address is not refreshed after the
 *    device is reset (cudaDeviceReset) or its primary context is destroyed and
 *    re-created: do not use this entry point across such a reset.
 *  - All calls share the one array, which keeps the last call's contents.
 *    Calls whose kernels may overlap on the GPU (e.g. on two streams with no
 *    ordering between them) race on it and produce wrong gradients; order
 *    them on one stream or with events.
 *  - Every call re-initialises the parts that must start at zero. */
int uaa_attn_bwd_noalloc(const void* q, const void* k, const void* v, const void* out,
                         const void* dout, const float* lse, const uint8_t* key_mask,
                         void* dq, void* dk, void* dv, int B, int S, int H, int D, float scale,
                         uaa_stream_t stream);

/* Size in bytes of the scratch array used by uaa_attn_bwd_noalloc. */
size_t uaa_attn_bwd_noalloc_max_bytes(void);

/* Ulysses forward exchange on one device: sequence shards -> head groups.
 * "UAA-bwd", What does this PR do (all-to-all with saved partition metadata,
 * uneven shards); "fast-ulysses", Summary (A2A around the attention module).
 *   x : device (P, B, cap, H, D) -- shard p's rows s < shard_lens[p] are valid,
 *       rows s >= shard_lens[p] are transport padding (not read)
 *   y : device (P, B, N, Hg, D), Hg = ceil(H/P), N = sum(shard_lens); group g
 *       holds heads [g*Hg, (g+1)*Hg) of every valid row, shards concatenated in
 *       rank order: y[g, b, off_p + s, h', :] = x[p, b, s, g*Hg + h', :]; heads
 *       g*Hg + h' >= H are zero (padded-head layout when P does not divide H,
 *       "UAA-bwd", What does this PR do)
 *   shard_lens : host, P ints, 0 <= shard_lens[p] <= cap
 *   elem_bytes : bytes per element (2 for bf16, 4 for fp32); D*elem_bytes must
 *       be a multiple of 16
 * x and y must not overlap.  Bit-exact copy. */
int uaa_seq_to_head(const void* x, void* y, int P, const int* shard_lens, int cap,
                    int B, int H, int D, int elem_bytes, uaa_stream_t stream);

/* Ulysses inverse exchange: head groups -> sequence shards (exact inverse of
 * uaa_seq_to_head).  y is (P, B, N, ceil(H/P), D), x is (P, B, cap, H, D) with
 * the true head count H: the padding heads of the groups are dropped.  Padding
 * rows s >= shard_lens[p] of every shard are written as zero.  Used for O in the
 * forward and for dQ (query partition) and dK/dV (key partition) in the backward
 * ("UAA-bwd", What does this PR do). */
int uaa_head_to_seq(const void* y, void* x, int P, const int* shard_lens, int cap,
                    int B, int H, int D, int elem_bytes, uaa_stream_t stream);

/* Ulysses attention with the exchanges fused into the attention kernels.
 * "UAA-bwd", What does this PR do: seq->head all-to-all, attention on the head
 * groups, head->seq all-to-all, with uneven shards; "fast-ulysses", Summary: the
 * all-to-all time around the attention module is what the backend saves.  On
 * one device the head groups together are all H heads, so the result is
 *   out = head_to_seq(attention(seq_to_head(q), seq_to_head(k), seq_to_head(v)))
 * computed without the re-layout round trips: the kernels read their 128-row
 * tiles straight from the shards (one TMA tensor map per shard; a tile never
 * straddles two shards, the last tile of a shard is partial) and write O back
 * into the shards.
 *   q, k, v, out : device, bf16 (P, B, cap, H, D) -- shard p's rows s < shard_lens[p]
 *                  are the sequence positions off_p + s (off_p = sum of the
 *                  earlier shard lengths); rows s >= shard_lens[p] are padding:
 *                  never read, and written as zero in out
 *   key_mask     : device uint8 (B, N) or NULL, N = sum(shard_lens), in sequence
 *                  order (as built by uaa_assemble_key_mask)
 *   lse          : device fp32 (B, H, N), sequence order
 *   shard_lens   : host, P ints, 0 <= shard_lens[p] <= cap; 1 <= P <= 8
 *                  (UAA_ERR_UNSUPPORTED otherwise; use the separate exchanges)
 * The key tiling follows the shards, so the sums run in a different order than
 * in uaa_attn_fwd on the re-laid-out tensors: results agree to rounding, not
 * bit for bit.  Returns UAA_OK or a negative uaa_status. */
int uaa_ulysses_attn_fwd(const void* q, const void* k, const void* v, const uint8_t* key_mask,
                         void* out, float* lse, int P, const int* shard_lens, int cap,
                         int B, int H, int D, float scale, uaa_stream_t stream);

/* Workspace for uaa_ulysses_attn_bwd: Delta and -LSE*log2(e) per query row,
 * each (B, H, T*128) fp32 with T = sum over shards of ceil(shard_lens[p]/128),
 * rounded up to 256 bytes.  Returns 0 for invalid arguments. */
size_t uaa_ulysses_attn_bwd_workspace_bytes(int P, const int* shard_lens, int cap,
                                            int B, int H, int D);

/* Backward of uaa_ulysses_attn_fwd: dq, dk, dv (P, B, cap, H, D) from dout in the
 * same sharded layout, with the exchanges fused the same way ("UAA-bwd", What
 * does this PR do: dQ follows the query partition, dK/dV the key partition).
 * Padding rows of dq, dk, dv are written as zero.  Deterministic (no atomics).
 *   lse : the forward's (B, H, N); key_mask : the forward's mask or NULL
 *   workspace : at least uaa_ulysses_attn_bwd_workspace_bytes() bytes, 256-byte
 *               aligned; contents on entry are ignored
 * Returns UAA_OK or a negative uaa_status. */
int uaa_ulysses_attn_bwd(const void* q, const void* k, const void* v, const void* out,
                         const void* dout, const float* lse, const uint8_t* key_mask,
                         void* dq, void* dk, void* dv, int P, const int* shard_lens, int cap,
                         int B, int H, int D, float scale, void* workspace, size_t workspace_bytes,
                         uaa_stream_t stream);

/* Key-padding mask assembly from gathered per-rank shards, trimming every
 * shard to its true length BEFORE concatenation ("UAA-bwd", What does this PR
 * do: the uneven mask-assembly fix; Validation: the four-rank masked case).
 *   gathered : device uint8 (P, B, cap)
 *   mask     : device uint8 (B, N), N = sum(shard_lens)
 *   mask[b, off_p + s] = gathered[p, b, s] for s < shard_lens[p]. */
int uaa_assemble_key_mask(const uint8_t* gathered, uint8_t* mask, int P, const int* shard_lens,
                          int cap, int B, uaa_stream_t stream);

/* Synchronises `stream`, then reads and clears the library's device status
 * words.  Returns UAA_OK, UAA_ERR_TIMEOUT (a bounded device wait ran out in
 * some kernel since the last check), UAA_ERR_DEBUG_CHECK (debug builds: a
 * device-side range check failed; uaa_last_error() names the first one) or
 * UAA_ERR_CUDA. */
int uaa_check_device_status(uaa_stream_t stream);

/* Diagnostic for the watchdog: launches one block whose thread waits on an
 * mbarrier that nothing arrives on, with a wait bound of `timeout_us`
 * microseconds (1..1000000).  The wait runs out, the kernel records
 * UAA_ERR_TIMEOUT and returns; no copy or tensor-core work is in flight. */
int uaa_watchdog_selftest(unsigned int timeout_us, uaa_stream_t stream);

/* Sets the bound (in milliseconds, default 4000) of every device-side wait in
 * the kernels launched afterwards by the calling process. 0 restores the default. */
void uaa_set_wait_timeout_ms(unsigned int ms);

/* Diagnostic for the abort paths (the pages have no counterpart; off by
 * default): while n >= 0, the producer of every attention kernel launched
 * afterwards skips its n-th ring load (counted from 0 in each CTA: the forward's
 * and the dQ kernel's K/V tile loads, the dK/dV kernel's query-tile loads).
 * Nothing ever fills that buffer, so the waits for it run out after the wait
 * bound, the call's kernels give up through their abort paths and
 * uaa_check_device_status() reports UAA_ERR_TIMEOUT.  No copy is ever issued
 * with a bad address: the load is simply not issued.  n < 0 turns it off. */
void uaa_debug_drop_load(int n);

/* Diagnostic (the pages have no counterpart): evaluates on the device, for
 * tests, the exponential the forward kernel takes on the FMA pipe for one
 * column pair of P in eight: 2^x by rounding x (clamped at -127) to n + f,
 * |f| <= 1/2, a cubic in f fitted in relative error (the coefficients come from
 * ulysses_dit_attention_gb300/exp2_fit.py; relative error below 8e-5) and 2^n
 * written into the exponent field (exactly 0 for x <= -127 and -inf).
 *   x, y : device float32 arrays of n elements, 8-byte aligned; n even
 *   y[i] = that approximation of 2^x[i].
 * Returns UAA_OK, UAA_ERR_INVALID_ARG or UAA_ERR_CUDA. */
int uaa_debug_exp2_fma2(const float* x, float* y, long long n, uaa_stream_t stream);

/* Thread-local, NUL-terminated message for the last non-OK status returned to
 * the calling thread ("" if none).  Owned by the library. */
const char* uaa_last_error(void);

/* Library version string, e.g. "uaa 0.1 sm_103a". */
const char* uaa_version(void);

/* 1 for the debug build of the library (libuaa_debug.so, compiled with
 * -DUAA_DEBUG), 0 otherwise.  The debug build checks, before each access, that
 * every tensor-core operand lies inside the issuing CTA's shared memory and
 * TMEM allocation and that every output store of the attention kernels lies
 * inside its tensor; a failed check skips the access and is reported by
 * uaa_check_device_status() as UAA_ERR_DEBUG_CHECK.  Same entry points and
 * results; slower. */
int uaa_debug_build(void);

#ifdef __cplusplus
}
#endif

#endif /* UAA_H_ */
