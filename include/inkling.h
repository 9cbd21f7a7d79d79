/*
 * inkling.h — C ABI of the Inkling attention-block library (sm_103a / GB300).
 *
 * The block, as the vLLM "Day-0 support for TML Inkling" blog describes it:
 *   - "Model Architecture / Sconv": a short convolution of window 4, per channel, on the
 *     attention keys and on the attention values;
 *   - "vLLM Integration & Optimization / Managing the sconv cache": the conv keeps the
 *     last W-1 = 3 tokens of its input per sequence;
 *   - "Model Architecture / Attention": grouped-query attention, head size 128, full and
 *     sliding-window layers, with a learned relative-position term added to the
 *     pre-softmax logits in place of RoPE;
 *   - "Model Architecture / MTP": up to 9 tokens per decode step (speculative verify);
 *   - "vLLM Integration & Optimization / FA4 with sheared bias": a per-configuration
 *     split factor for the KV dimension ("num_splits");
 *   - the Inkling serving recipe ("Client Usage"): paged KV cache with --block-size 128.
 * The pages do not fix the relative term's form; this library uses a per-query-head
 * table b[h][min(q_pos - k_pos, R - 1)] (fp32, R entries per head).
 *
 * Conventions shared by every entry point
 *   Layouts (row-major, densely packed, element sizes in brackets):
 *     q          [T][Hq][128]                     bf16  (T = all new tokens of the batch)
 *     k_raw,v_raw[T][C]                           bf16  (C = Hkv * 128, c = kv_head*128 + d)
 *     w_k, w_v   [C][4]                           fp32  (w[c][3] multiplies the current
 *                                                        token, w[c][0] the token 3 back)
 *     sconv_state[B][2][3][C]                     bf16  (index 0 = K, 1 = V; raw pre-conv
 *                                                        rows, oldest first)
 *     k_cache, v_cache [num_blocks][Hkv][128][128] bf16 (page, kv head, slot, dim)
 *     block_table[B][max_blocks]                  int32 (logical page -> physical page)
 *     cu_q_lens  [B+1]                            int32 (prefix sums of new tokens)
 *     seq_lens   [B]                              int32 (KV length incl. the new tokens)
 *     slot_mapping[T]                             int64 (page*128 + slot, -1 = skip)
 *     bias       [Hq][R]                          fp32
 *     out        [T][Hq][128]                     bf16 or fp32 (out_dtype)
 *     lse        [T][Hq]                          fp32, natural log (may be NULL)
 *   Positions: query token t of sequence b sits at seq_lens[b] - n_b + t, n_b =
 *   cu_q_lens[b+1] - cu_q_lens[b].  Key j is allowed for a query at p iff 0 <= p - j and
 *   (window == 0 or p - j <= window - 1).  Logit = scale * q.k + bias[h][min(p-j, R-1)].
 *   Query head h reads KV head h / (Hq / Hkv).
 *   Pointers: every array pointer is a DEVICE pointer unless stated otherwise.  The
 *   caller allocates and owns all memory; the library allocates no device memory and
 *   keeps no per-call state.  All work is enqueued on `stream` and never synchronised.
 *   Alignment: q, k_cache, v_cache, k_raw, v_raw and out must be 16-byte aligned.
 *   Errors: argument problems found on the host return a nonzero inkling_status_t and
 *   launch nothing.  Problems found on the device (a physical page id outside
 *   [0, num_blocks), inconsistent lengths, a wait that ran out of time) are written to
 *   `dev_status` (a device int32, first error wins; may be NULL), readable after the
 *   stream is synchronised; the affected rows are left unwritten.  Kernels never trap.
 *   dev_status must hold 0 when a call is enqueued: the attention kernels poll it and
 *   stop waiting once any CTA has reported an error, so that one failure ends the launch
 *   quickly instead of every CTA running into its own time limit.
 *   Ordering: inkling_sconv_kv for a step's new tokens must precede, on the same stream,
 *   the attention call that reads them.  The caller zeroes the sconv state rows of a
 *   sequence that starts from nothing.
 */
#ifndef INKLING_H
#define INKLING_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define INKLING_API __attribute__((visibility("default")))
#else
#define INKLING_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st *inkling_stream_t; /* same object as cudaStream_t; NULL = legacy default stream */

typedef enum {
  INKLING_OK = 0,
  INKLING_ERR_INVALID_ARG = 1, /* host-side argument check failed; nothing launched */
  INKLING_ERR_UNSUPPORTED = 2, /* shape outside what the kernels implement */
  INKLING_ERR_CUDA = 3,        /* a CUDA runtime call or launch failed */
  INKLING_ERR_TIMEOUT = 4,     /* device: a bounded wait ran out (written to dev_status) */
  INKLING_ERR_BAD_BLOCK = 5,   /* device: page id or slot outside the cache */
  INKLING_ERR_BAD_INPUT = 6,   /* device: lengths inconsistent with the host-side limits */
  INKLING_ERR_WORKSPACE = 7    /* workspace missing or too small */
} inkling_status_t;

enum { INKLING_HEAD_DIM = 128, INKLING_BLOCK_SIZE = 128, INKLING_SCONV_WIDTH = 4,
       INKLING_MAX_DECODE_Q = 9 };
enum { INKLING_OUT_BF16 = 0, INKLING_OUT_F32 = 1 };

/* Human-readable name of a status code (static storage, never NULL). */
INKLING_API const char *inkling_status_string(int status);

/* Library version, e.g. 0x000100 = 0.1.0. */
INKLING_API int inkling_version(void);

/*
 * inkling_sconv_kv — the window-4 causal short convolution on K and on V (blog, "Model
 * Architecture / Sconv") for the new tokens of every sequence, written straight into the
 * paged KV cache, then the sconv cache moved forward ("Managing the sconv cache").
 *
 *   x~ = [sconv_state[b][kv] rows 0..2 ; new raw rows of b]
 *   y[t][c] = sum_{j=0..3} w[c][j] * x~[t + j][c]        (fp32 arithmetic)
 *   cache[slot_mapping[t]] = bf16_rne(y[t])   (skipped when slot_mapping[t] == -1)
 *   sconv_state[b][kv] = the last 3 rows of x~ (raw, pre-conv)
 *
 * B sequences, T = cu_q_lens[B] new tokens in total, max_q_len >= every n_b (host-side
 * bound used to size the launch).  num_blocks = pages in each cache.  The raw rows never
 * round-trip through HBM: they are read once and the conv output lands in the cache.
 * Device errors: slot >= num_blocks*128 -> INKLING_ERR_BAD_BLOCK; n_b > max_q_len or
 * cu_q_lens not monotone -> INKLING_ERR_BAD_INPUT.
 */
INKLING_API int inkling_sconv_kv(const void *k_raw, const void *v_raw, const float *w_k, const float *w_v,
                     void *sconv_state, const int32_t *cu_q_lens, const int64_t *slot_mapping,
                     void *k_cache, void *v_cache, int32_t B, int32_t T, int32_t Hkv,
                     int64_t num_blocks, int32_t max_q_len, int32_t *dev_status,
                     inkling_stream_t stream);

/*
 * inkling_sconv_kv_fp8 — inkling_sconv_kv writing an FP8 KV cache (blog, "Roadmap": FP8
 * for the global-attention layers).  The caches hold one OCP E4M3
 * byte per element in the same page layout, [num_blocks][Hkv][128 slots][128 dims] uint8:
 *
 *   cache[slot_mapping[t]] = e4m3(y[t] / scale)   (round to nearest even, saturating at
 *                                                  +-448; k_scale for K, v_scale for V)
 *
 * with y computed as in inkling_sconv_kv (fp32); the sconv state update is unchanged.
 * k_scale, v_scale: finite and > 0 (else INKLING_ERR_INVALID_ARG).  Other arguments and
 * errors as inkling_sconv_kv.
 */
INKLING_API int inkling_sconv_kv_fp8(const void *k_raw, const void *v_raw, const float *w_k,
                         const float *w_v, void *sconv_state, const int32_t *cu_q_lens,
                         const int64_t *slot_mapping, void *k_cache, void *v_cache,
                         float k_scale, float v_scale, int32_t B, int32_t T, int32_t Hkv,
                         int64_t num_blocks, int32_t max_q_len, int32_t *dev_status,
                         inkling_stream_t stream);

/*
 * inkling_sconv — the same window-4 causal short convolution on one dense stream with
 * its own 3-row cache (blog, "Model Architecture / Sconv": the conv also follows the
 * attention output projection, "all-reduce (after o_proj) -> sconv -> residual").
 *
 *   x[T][C] bf16 raw rows, w[C][4] fp32 taps, sconv_state[B][3][C] bf16 (in/out, raw rows,
 *   oldest first), y[T][C] bf16 out.
 *   x~ = [sconv_state[b] ; new rows of b];  y[t][c] = bf16_rne(sum_j w[c][j] * x~[t + j][c]);
 *   sconv_state[b] = the last 3 rows of x~.
 *
 * C % 8 == 0; y must not be x.  T = cu_q_lens[B]; max_q_len >= every n_b.  Device
 * errors: n_b > max_q_len, or cu_q_lens not monotone or past T -> INKLING_ERR_BAD_INPUT.
 */
INKLING_API int inkling_sconv(const void *x, const float *w, void *sconv_state, const int32_t *cu_q_lens,
                  void *y, int32_t B, int32_t T, int32_t C, int32_t max_q_len,
                  int32_t *dev_status, inkling_stream_t stream);

/*
 * inkling_sconv_state_rollback — the sconv cache after a speculative (MTP verify) step
 * of which only the first accepted[b] of its n_b new tokens are kept (blog, "Model
 * Architecture / MTP" and "Re-computing MTP KV cache": drafts past the first rejection
 * are dropped).  The conv is causal, so the cache rows written for the kept tokens are
 * already right; only the 3-row state must be recomputed:
 *
 *   state_after[b][s] = the last 3 rows of [state_before[b][s] ; raw rows
 *                       cu_q_lens[b] .. cu_q_lens[b] + accepted[b] - 1 of stream s]
 *
 * streams = 2: the K/V pair, x0 = k_raw, x1 = v_raw, state [B][2][3][C] (the layout of
 * inkling_sconv_kv); streams = 1: one dense stream, x1 unused, state [B][3][C].
 * state_before is the state as it was before the step's conv call (the caller keeps that
 * copy: 3*C*streams*2 bytes per sequence); state_after may be the same buffer.  accepted
 * is a device array [B] (0 <= accepted[b] <= n_b, else INKLING_ERR_BAD_INPUT and the
 * sequence's state is left unwritten); accepted[b] = n_b reproduces the conv call's own
 * state update.  T = cu_q_lens[B].  The pages state the requirement, not an API: the
 * entry point itself is this library's.
 */
INKLING_API int inkling_sconv_state_rollback(const void *state_before, const void *x0, const void *x1,
                                 const int32_t *cu_q_lens, const int32_t *accepted,
                                 void *state_after, int32_t B, int32_t T, int32_t C,
                                 int32_t streams, int32_t *dev_status, inkling_stream_t stream);

/*
 * inkling_rel_attn_prefill — relative-bias GQA attention (blog, "Model Architecture /
 * Attention") for every new token of every sequence, reading keys and values from the
 * paged cache (so a cached prefix is attended to as well: chunked prefill).
 *
 *   out[t][h] = sum_j softmax_j(scale * q[t][h].K[j] + bias[h][min(p - j, R-1)]) V[j]
 *
 * Hq % Hkv == 0, head size 128, R >= 1, window >= 0 (0 = full causal), out_dtype
 * INKLING_OUT_BF16 or INKLING_OUT_F32.  max_q_len >= every n_b (sizes the grid).
 * lse (nullable) receives log(sum_j exp(logit_j)).
 */
INKLING_API int inkling_rel_attn_prefill(const void *q, const void *k_cache, const void *v_cache,
                             const int32_t *block_table, int32_t max_blocks,
                             const int32_t *cu_q_lens, const int32_t *seq_lens,
                             const float *bias, int32_t R, float scale, int32_t window,
                             void *out, int32_t out_dtype, float *lse, int32_t B, int32_t T,
                             int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len,
                             int32_t *dev_status, inkling_stream_t stream);

/*
 * inkling_rel_attn_prefill_fp8 — inkling_rel_attn_prefill over the FP8 (E4M3) caches that
 * inkling_sconv_kv_fp8 writes (blog, "Roadmap": FP8 for the global-attention layers):
 * K = code * k_scale, V = code * v_scale, same page layout as the decode's FP8 caches.
 * The call first widens every page that a step's query can see (window-aware) into a
 * bf16 page pool in the caller's workspace, exactly (E4M3 values are bf16 values), then
 * runs the bf16 prefill on that pool with scale * k_scale as the logit scale and v_scale
 * applied to the output.  max_seq_len >= every seq_lens[b] (host bound that sizes the
 * pool).  workspace: 16-byte aligned device memory of at least
 * inkling_rel_attn_prefill_fp8_workspace_size(B, Hkv, max_blocks, max_q_len, max_seq_len,
 * window) bytes, owned by the caller, reused by the next call on the stream; too small ->
 * INKLING_ERR_WORKSPACE, nothing launched.  Device errors as for the prefill (a sequence
 * whose pages exceed the max_seq_len bound -> INKLING_ERR_BAD_INPUT).
 */
INKLING_API size_t inkling_rel_attn_prefill_fp8_workspace_size(int32_t B, int32_t Hkv,
                                                               int32_t max_blocks,
                                                               int32_t max_q_len,
                                                               int32_t max_seq_len,
                                                               int32_t window);
INKLING_API int inkling_rel_attn_prefill_fp8(
    const void *q, const void *k_cache, const void *v_cache, float k_scale, float v_scale,
    const int32_t *block_table, int32_t max_blocks, const int32_t *cu_q_lens,
    const int32_t *seq_lens, const float *bias, int32_t R, float scale, int32_t window,
    void *out, int32_t out_dtype, float *lse, int32_t B, int32_t T, int32_t Hq, int32_t Hkv,
    int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len, void *workspace,
    size_t workspace_bytes, int32_t *dev_status, inkling_stream_t stream);

/*
 * inkling_rel_attn_decode_workspace_size — bytes of device workspace that
 * inkling_rel_attn_decode needs for these limits (0 when no split is needed).
 * num_splits: 0 = the library's choice for this device (same rule as the decode call).
 */
INKLING_API size_t inkling_rel_attn_decode_workspace_size(int32_t B, int32_t Hq, int32_t Hkv,
                                              int32_t max_q_len, int32_t max_seq_len,
                                              int32_t window, int32_t num_splits);

/*
 * inkling_rel_attn_decode_plan — how inkling_rel_attn_decode and
 * inkling_rel_attn_decode_fp8 split the keys for these limits on the current device (the
 * rule of the decode calls and of the workspace query).  plan: caller's array of 4 int32:
 *   [0] splits per (sequence, KV head): the page ranges processed by separate CTAs;
 *   [1] CTAs of the decode launch (splits x Hkv x B, saturating at INT32_MAX);
 *   [2] pages per split;
 *   [3] 1 when a merge kernel follows the decode kernel (more than one split), else 0.
 * Returns INKLING_ERR_INVALID_ARG for bad limits (or a NULL plan), INKLING_ERR_CUDA when
 * num_splits = 0 and no device is current.
 */
INKLING_API int inkling_rel_attn_decode_plan(int32_t B, int32_t Hq, int32_t Hkv, int32_t max_q_len,
                                 int32_t max_seq_len, int32_t window, int32_t num_splits,
                                 int32_t *plan);

/*
 * inkling_rel_attn_decode — the same attention for decode steps of up to
 * INKLING_MAX_DECODE_Q (9) new tokens per sequence (MTP verify, blog "Model Architecture /
 * MTP"), with the keys of each sequence split into `num_splits` page ranges processed in
 * parallel and merged exactly (the blog's FA4 "num_splits", "FA4 with sheared bias").
 * The G = Hq/Hkv query heads and n_b tokens that share a KV head are packed into one
 * tile, so every K/V page is read once per KV head.
 *
 * max_q_len <= 9; max_seq_len >= every seq_lens[b] (host bound used to size the split).
 * num_splits: 0 = automatic.  workspace: device memory of at least
 * inkling_rel_attn_decode_workspace_size(...) bytes with the same arguments (may be NULL
 * when that size is 0); owned by the caller, contents need no initialisation and are
 * scratch after the call.  Concurrent calls must not share a workspace.
 */
INKLING_API int inkling_rel_attn_decode(const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_table, int32_t max_blocks,
                            const int32_t *cu_q_lens, const int32_t *seq_lens,
                            const float *bias, int32_t R, float scale, int32_t window,
                            void *out, int32_t out_dtype, float *lse, int32_t B, int32_t T,
                            int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len,
                            int32_t max_seq_len, int32_t num_splits, void *workspace,
                            size_t workspace_bytes, int32_t *dev_status,
                            inkling_stream_t stream);

/*
 * inkling_rel_attn_decode_sconv — one decode step with the sconv of its new tokens fused
 * into the decode kernel's prologue (blog "vLLM Integration & Optimization", closing
 * paragraph: kernel fusion and PDL; "Managing the sconv cache": the last W-1 = 3 raw rows
 * per sequence).  The same results as inkling_sconv_kv followed by inkling_rel_attn_decode
 * on the same stream, with one launch (two when the keys are split) instead of two (three):
 * the cache rows and the state are bit-identical to the separate conv's, and the
 * attention output to the separate decode's.
 *
 * k_raw, v_raw [T][Hkv*128] bf16: the new tokens' raw (pre-conv) K and V rows, packed as
 *   q (sequence b's rows at cu_q_lens[b] ..);
 * w_k, w_v [Hkv*128][4] fp32 taps (w[c][3] multiplies the current token);
 * sconv_state [B][2][3][Hkv*128] bf16, in/out, as for inkling_sconv_kv;
 * k_cache, v_cache: the bf16 paged caches, written at the new rows' slots and read by the
 *   attention.  Sequence b's new row t (position L_b - n_b + t) goes to page
 *   block_table[b][pos / 128], slot pos % 128: the slots a decode step's slot mapping
 *   names (no slot_mapping argument; the block table alone decides where a row lives).
 * Every other argument, the workspace, num_splits and the errors are those of
 * inkling_rel_attn_decode; k_raw, v_raw, w_k, w_v and sconv_state must be non-NULL and
 * 16-byte aligned (INKLING_ERR_INVALID_ARG).  Each (split, KV head, sequence) CTA
 * convolves the new rows that fall in its own pages before it loads them; the state of a
 * sequence whose keys are split is written by the merge kernel, after every CTA that
 * reads the old state has finished.  bf16 caches only.
 */
INKLING_API int inkling_rel_attn_decode_sconv(
    const void *q, const void *k_raw, const void *v_raw, const float *w_k, const float *w_v,
    void *sconv_state, void *k_cache, void *v_cache, const int32_t *block_table,
    int32_t max_blocks, const int32_t *cu_q_lens, const int32_t *seq_lens, const float *bias,
    int32_t R, float scale, int32_t window, void *out, int32_t out_dtype, float *lse,
    int32_t B, int32_t T, int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len,
    int32_t max_seq_len, int32_t num_splits, void *workspace, size_t workspace_bytes,
    int32_t *dev_status, inkling_stream_t stream);

/*
 * inkling_rel_attn_decode_fp8 — inkling_rel_attn_decode over an FP8 KV cache written by
 * inkling_sconv_kv_fp8: K = e4m3(code) * k_scale, V = e4m3(code) * v_scale.  The pages
 * are read as bytes (half the HBM traffic of the bf16 cache) and widened to f16 in shared
 * memory, which is exact; Q, P and the products then run on the f16 tensor core with
 * fp32 accumulation, so Q must lie in the f16 range (|q| < 65504).  Arguments, workspace
 * and errors as inkling_rel_attn_decode (the workspace size query is the same call).
 */
INKLING_API int inkling_rel_attn_decode_fp8(const void *q, const void *k_cache, const void *v_cache,
                                float k_scale, float v_scale, const int32_t *block_table,
                                int32_t max_blocks, const int32_t *cu_q_lens,
                                const int32_t *seq_lens, const float *bias, int32_t R,
                                float scale, int32_t window, void *out, int32_t out_dtype,
                                float *lse, int32_t B, int32_t T, int32_t Hq, int32_t Hkv,
                                int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
                                int32_t num_splits, void *workspace, size_t workspace_bytes,
                                int32_t *dev_status, inkling_stream_t stream);

/*
 * inkling_rel_attn_decode_noalloc — inkling_rel_attn_decode for callers that cannot give
 * the library a device buffer: a runtime that reserves all device memory at start-up and
 * forbids cudaMalloc while serving (it can synchronise the device, and it is not allowed
 * inside a stream that is being captured), or code that runs inside another framework's
 * allocator and must not re-enter it.  The pages have no counterpart to this call.
 *
 * Arguments and results are those of inkling_rel_attn_decode without the workspace.
 * The split partials go to a static device array of
 * inkling_rel_attn_decode_noalloc_capacity() bytes (32 MiB) that is part of the library:
 * every GPU that loads the library holds it until the process exits.  A request whose
 * partials would not fit (inkling_rel_attn_decode_workspace_size(...) with the same
 * arguments above the capacity) returns INKLING_ERR_WORKSPACE and launches nothing.
 * Argument checks and their order are those of inkling_rel_attn_decode: the capacity
 * is compared last, so a call with a bad argument reports that argument's error.
 * The first call on a device looks up the array's device address (cudaGetSymbolAddress,
 * with that device current); make that first call before any stream capture.  The address
 * is kept per device and CUDA context (by the context's process-unique id), so the first
 * call after the device's context has been replaced (cudaDeviceReset, or the primary
 * context released and made again) looks it up again and is again a first call.  No
 * device memory is allocated or freed.  All calls share the one array and it keeps the
 * last call's contents (the kernels need none of it zeroed): calls whose work can overlap
 * on the GPU (other streams, other threads) race on it and must be serialised by the
 * caller.
 */
INKLING_API size_t inkling_rel_attn_decode_noalloc_capacity(void);
INKLING_API int inkling_rel_attn_decode_noalloc(
    const void *q, const void *k_cache, const void *v_cache, const int32_t *block_table,
    int32_t max_blocks, const int32_t *cu_q_lens, const int32_t *seq_lens, const float *bias,
    int32_t R, float scale, int32_t window, void *out, int32_t out_dtype, float *lse, int32_t B,
    int32_t T, int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len,
    int32_t max_seq_len, int32_t num_splits, int32_t *dev_status, inkling_stream_t stream);

/*
 * inkling_prefill_step_host / inkling_decode_step_host — one whole step, the sconv of the
 * new tokens (inkling_sconv_kv) then the attention (inkling_rel_attn_prefill, or
 * inkling_rel_attn_decode with its workspace and split arguments), for a caller whose
 * per-step tensors live in page-locked host memory:
 *   q_host [T][Hq][128] bf16, k_raw_host / v_raw_host [T][Hkv*128] bf16   (read)
 *   out_host [T][Hq][128], bf16 or f32 by out_dtype                       (written)
 * q_dev, k_raw_dev, v_raw_dev, out_dev are device staging buffers of the same shapes,
 * owned by the caller; every other pointer is the device pointer the separate calls take
 * (cu_q_lens on the device, and cu_q_lens_host, its host copy, which gives the sequence
 * boundaries).  The step is cut into `chunks` groups of whole sequences with about T /
 * chunks tokens each.  Group g's rows go up on h2d_stream, group g is computed on
 * `stream` once they have landed, and its output rows come down on d2h_stream, so the
 * host link carries one group while the GPU computes another (groups are independent:
 * a sequence's attention reads only its own pages).  h2d_stream first waits for the work
 * already on `stream` (the staging buffers may still be in use), and `stream` ends
 * waiting for the last copy down, so an event recorded on `stream` after the call marks
 * the end of the whole step.  The three streams must be distinct; chunks >= 1 (more
 * chunks than sequences are capped at B).  Nothing is synchronised: the call returns
 * once everything is enqueued, and out_host is complete when `stream` reaches that point.
 * Host-side argument errors are returned before anything is enqueued; an error from one
 * group's launch stops the enqueueing and is returned (earlier groups stay enqueued).
 * Device-side errors land in dev_status as for the separate calls.  The prefill form may
 * also cut a sequence with more than its group's share of tokens into pieces of whole
 * 128-token query tiles, each computed as a chunked prefill of that sequence (outputs
 * bit-identical to the uncut call); it does so only when given dev_scratch, device
 * memory for 4 * chunks int32 lengths (NULL: groups of whole sequences only).  The decode
 * form takes
 * a workspace sized for all B sequences (inkling_rel_attn_decode_workspace_size); the
 * groups reuse it one after another on `stream`, all with the split count the whole batch
 * would get (num_splits = 0) or the one given.
 */
INKLING_API int inkling_prefill_step_host(
    const void *q_host, const void *k_raw_host, const void *v_raw_host, void *out_host,
    void *q_dev, void *k_raw_dev, void *v_raw_dev, void *out_dev, const int32_t *cu_q_lens_host,
    const float *w_k, const float *w_v, void *sconv_state, const int32_t *cu_q_lens,
    const int64_t *slot_mapping, void *k_cache, void *v_cache, const int32_t *block_table,
    int32_t max_blocks, const int32_t *seq_lens, const float *bias, int32_t R, float scale,
    int32_t window, int32_t out_dtype, float *lse, int32_t B, int32_t T, int32_t Hq,
    int32_t Hkv, int64_t num_blocks, int32_t max_q_len, int32_t chunks, int32_t *dev_scratch,
    int32_t *dev_status, inkling_stream_t stream, inkling_stream_t h2d_stream,
    inkling_stream_t d2h_stream);
INKLING_API int inkling_decode_step_host(
    const void *q_host, const void *k_raw_host, const void *v_raw_host, void *out_host,
    void *q_dev, void *k_raw_dev, void *v_raw_dev, void *out_dev, const int32_t *cu_q_lens_host,
    const float *w_k, const float *w_v, void *sconv_state, const int32_t *cu_q_lens,
    const int64_t *slot_mapping, void *k_cache, void *v_cache, const int32_t *block_table,
    int32_t max_blocks, const int32_t *seq_lens, const float *bias, int32_t R, float scale,
    int32_t window, int32_t out_dtype, float *lse, int32_t B, int32_t T, int32_t Hq,
    int32_t Hkv, int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
    int32_t num_splits, void *workspace, size_t workspace_bytes, int32_t chunks,
    int32_t *dev_status, inkling_stream_t stream, inkling_stream_t h2d_stream,
    inkling_stream_t d2h_stream);

/*
 * inkling_prefill_step_host_fp8 / inkling_decode_step_host_fp8 — the same whole steps over
 * an E4M3 cache (vLLM Day-0 Inkling blog, "Roadmap": FP8 for the global-attention
 * layers): each group runs inkling_sconv_kv_fp8 (codes written with k_scale / v_scale),
 * then inkling_rel_attn_prefill_fp8 or inkling_rel_attn_decode_fp8.  Arguments as for the
 * bf16 forms, plus the scales (positive and finite), max_seq_len, and the workspace of the
 * FP8 call: for the prefill, inkling_rel_attn_prefill_fp8_workspace_size(B, Hkv,
 * max_blocks, max_q_len, max_seq_len, window) bytes, into which each group widens the
 * pages it reads (the groups reuse it one after another on `stream`); for the decode, as
 * inkling_decode_step_host.  Outputs are bit-identical to the separate FP8 calls.
 */
INKLING_API int inkling_prefill_step_host_fp8(
    const void *q_host, const void *k_raw_host, const void *v_raw_host, void *out_host,
    void *q_dev, void *k_raw_dev, void *v_raw_dev, void *out_dev, const int32_t *cu_q_lens_host,
    const float *w_k, const float *w_v, void *sconv_state, const int32_t *cu_q_lens,
    const int64_t *slot_mapping, void *k_cache, void *v_cache, float k_scale, float v_scale,
    const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens, const float *bias,
    int32_t R, float scale, int32_t window, int32_t out_dtype, float *lse, int32_t B, int32_t T,
    int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
    void *workspace, size_t workspace_bytes, int32_t chunks, int32_t *dev_scratch,
    int32_t *dev_status, inkling_stream_t stream, inkling_stream_t h2d_stream,
    inkling_stream_t d2h_stream);
INKLING_API int inkling_decode_step_host_fp8(
    const void *q_host, const void *k_raw_host, const void *v_raw_host, void *out_host,
    void *q_dev, void *k_raw_dev, void *v_raw_dev, void *out_dev, const int32_t *cu_q_lens_host,
    const float *w_k, const float *w_v, void *sconv_state, const int32_t *cu_q_lens,
    const int64_t *slot_mapping, void *k_cache, void *v_cache, float k_scale, float v_scale,
    const int32_t *block_table, int32_t max_blocks, const int32_t *seq_lens, const float *bias,
    int32_t R, float scale, int32_t window, int32_t out_dtype, float *lse, int32_t B, int32_t T,
    int32_t Hq, int32_t Hkv, int64_t num_blocks, int32_t max_q_len, int32_t max_seq_len,
    int32_t num_splits, void *workspace, size_t workspace_bytes, int32_t chunks,
    int32_t *dev_status, inkling_stream_t stream, inkling_stream_t h2d_stream,
    inkling_stream_t d2h_stream);

/*
 * inkling_selftest_bounded_wait — checks, on the device, the bounded waits that every
 * pipeline kernel uses (their failure detection).  `ctas` CTAs each wait, with the
 * kernels' own wait, on a barrier that nothing arrives on.  mode 0: every wait must give
 * up after its cycle budget (about 2 s); dev_status becomes INKLING_ERR_TIMEOUT and
 * *dev_gave_up counts the waits that gave up.  mode 1: CTA 0 first writes
 * INKLING_ERR_BAD_INPUT to dev_status, and the other waits must see it and give up within
 * about a millisecond.  dev_status and dev_gave_up are device int32s the caller zeroes.
 * Nothing faults or hangs; the context stays usable afterwards.
 */
INKLING_API int inkling_selftest_bounded_wait(int32_t mode, int32_t ctas, int32_t *dev_status,
                                              int32_t *dev_gave_up, inkling_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* INKLING_H */
