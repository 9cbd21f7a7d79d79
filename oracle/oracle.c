/*
 * fp64 CPU oracle for the Inkling attention block.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg may load this library.  It shares no code, header, table or helper
 * with the CUDA library: it is the plain definition of what the block computes, written
 * out with no blocking, fusion or reordering, so that a reader can check it by eye.
 *
 * Sources (the vLLM "Day-0 support for TML Inkling" blog and the Inkling serving
 * recipes):
 *  - Sconv: "Model Architecture / Sconv" (a window-4 short convolution applied to the
 *    attention keys and values, per channel) and "vLLM Integration & Optimization /
 *    Managing the sconv cache" (the cache keeps the last W-1 = 3 tokens).
 *  - Relative attention: "Model Architecture / Attention" (GQA, head size 128, full and
 *    sliding-window layers; a learned relative-position term added to the pre-softmax
 *    logits instead of RoPE).  The pages do not fix the term's parameterisation; this
 *    oracle uses a per-query-head table b[h, min(q-k, R-1)].
 *  - MTP verify: "Model Architecture / MTP" (up to 9 query tokens per decode step);
 *    decode and prefill share one definition and differ only in the number of new
 *    tokens per sequence.
 *
 * Readings taken where the pages are silent (each listed in the design notes):
 *  tap order w[c,3] * current token + ... + w[c,0] * token three back; no bias, no
 *  activation, no residual in the sconv; zero history at sequence start; the cache
 *  holds raw (pre-conv) rows; conv output rounded to bf16 (round to nearest even) before
 *  it enters the bf16 KV cache; logit = scale * q.k + b[h, min(p_q - p_k, R-1)]; key
 *  allowed iff 0 <= p_q - p_k and (window == 0 or p_q - p_k <= window - 1); query head h
 *  reads KV head h / (Hq/Hkv); query token t of sequence b sits at position
 *  seq_len[b] - n_b + t.
 *
 * Storage: the KV cache is paged, [num_blocks][Hkv][128 slots][128 dims] bf16; logical
 * key j of sequence b lives in page block_table[b][j / 128], slot j % 128.  bf16 values
 * are passed as their 16-bit patterns.
 *
 * FP8 KV cache (the blog's "Roadmap" plans FP8 for the global-attention layers, whose
 * BF16 compute and KV cache it names as a bottleneck; nothing more is specified): the same pages hold one byte per element in the OCP
 * E4M3 format, code = e4m3(y / scale) rounded to nearest even and saturated at +-448,
 * with one fp32 scale for K and one for V; attention reads K = e4m3(code) * k_scale and
 * V = e4m3(code) * v_scale.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define OR_D 128
#define OR_PAGE 128
#define OR_TAPS 4

enum { OR_OK = 0, OR_ERR_ARG = 1, OR_ERR_BLOCK = 2, OR_ERR_NOMEM = 3 };

/* bf16 -> double: the 16 bits are the top half of an IEEE binary32; exact. */
double oracle_bf16_to_double(uint16_t b)
{
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* double -> bf16, round to nearest, ties to even, in one step (no detour through
 * binary32, which would round twice).  bf16 keeps 8 significant bits and the binary32
 * exponent range, so the spacing of bf16 values around y is 2^(e-7) with
 * e = max(floor(log2|y|), -126); subnormals share the spacing 2^-133. */
uint16_t oracle_bf16_round(double y)
{
    uint32_t u;
    float f;
    if (isnan(y)) return 0x7fc0;
    if (y == 0.0) {
        f = (float)y; /* keeps the sign of zero */
        memcpy(&u, &f, sizeof u);
        return (uint16_t)(u >> 16);
    }
    int e;
    frexp(y, &e); /* |y| = m * 2^e, m in [0.5, 1): floor(log2|y|) = e - 1 */
    int ex = e - 1;
    if (ex < -126) ex = -126;
    double ulp = ldexp(1.0, ex - 7);
    double r = nearbyint(y / ulp) * ulp; /* default rounding mode: nearest-even */
    /* largest finite bf16 is (2 - 2^-7) * 2^127; anything rounding past it is inf */
    if (fabs(r) >= ldexp(1.0, 128)) r = y > 0 ? INFINITY : -INFINITY;
    f = (float)r; /* exact: r has at most 8 significant bits */
    memcpy(&u, &f, sizeof u);
    return (uint16_t)(u >> 16);
}

/*
 * Sconv on K and on V for the new tokens of every sequence, written into the paged
 * cache, then the sconv state moved forward.
 *
 *   x~ = [state rows 0..2 (oldest first) ; the n_b new raw rows]
 *   y[t, c] = sum_{j=0..3} w[c, j] * x~[t + j, c]          (x~[t + 3] = new row t)
 *   cache[slot_mapping[t]] <- bf16(y[t])   (slot -1: not stored)
 *   state <- x~[n_b], x~[n_b + 1], x~[n_b + 2]
 *
 * k_raw, v_raw [T][C]; w_k, w_v [C][4]; state [B][2][3][C] (index 0 = K, 1 = V);
 * caches [num_blocks][Hkv][128][128]; C = Hkv * 128.
 */
int oracle_sconv_kv(const uint16_t *k_raw, const uint16_t *v_raw, const float *w_k,
                    const float *w_v, uint16_t *state, const int32_t *cu_q_lens,
                    const int64_t *slot_mapping, uint16_t *k_cache, uint16_t *v_cache,
                    int B, int T, int Hkv, int64_t num_blocks)
{
    if (B < 0 || T < 0 || Hkv <= 0 || num_blocks < 0) return OR_ERR_ARG;
    if (cu_q_lens[0] != 0 || cu_q_lens[B] != T) return OR_ERR_ARG;
    const int C = Hkv * OR_D;
    for (int b = 0; b < B; ++b) {
        const int t0 = cu_q_lens[b];
        const int n = cu_q_lens[b + 1] - t0;
        if (n < 0) return OR_ERR_ARG;
        for (int which = 0; which < 2; ++which) {
            const uint16_t *x = which == 0 ? k_raw : v_raw;
            const float *w = which == 0 ? w_k : w_v;
            uint16_t *cache = which == 0 ? k_cache : v_cache;
            uint16_t *st = state + ((size_t)b * 2 + which) * 3 * C;
            /* x~ rows as bit patterns: rows 0..2 from the state, rows 3.. from x */
            uint16_t *ext = malloc(sizeof(uint16_t) * (size_t)(n + 3) * C);
            if (!ext) return OR_ERR_NOMEM;
            memcpy(ext, st, sizeof(uint16_t) * 3 * (size_t)C);
            memcpy(ext + 3 * (size_t)C, x + (size_t)t0 * C, sizeof(uint16_t) * (size_t)n * C);
            for (int t = 0; t < n; ++t) {
                const int64_t slot = slot_mapping[t0 + t];
                if (slot < 0) continue;
                if (slot >= num_blocks * OR_PAGE) { free(ext); return OR_ERR_BLOCK; }
                const int64_t blk = slot / OR_PAGE, off = slot % OR_PAGE;
                for (int c = 0; c < C; ++c) {
                    double y = 0.0;
                    for (int j = 0; j < OR_TAPS; ++j)
                        y += (double)w[(size_t)c * OR_TAPS + j] *
                             oracle_bf16_to_double(ext[(size_t)(t + j) * C + c]);
                    const int h = c / OR_D, d = c % OR_D;
                    cache[(((size_t)blk * Hkv + h) * OR_PAGE + off) * OR_D + d] =
                        oracle_bf16_round(y);
                }
            }
            memcpy(st, ext + (size_t)n * C, sizeof(uint16_t) * 3 * (size_t)C);
            free(ext);
        }
    }
    return OR_OK;
}

/* ---------------------------------------------------------------- attention ---- */

typedef struct {
    const uint16_t *q;
    const void *k_cache, *v_cache;  /* bf16 patterns, or e4m3 codes when kv_fp8 */
    const int32_t *block_table, *cu_q_lens, *seq_lens, *rows;
    const float *bias;
    int max_blocks, R, window, B, T, Hq, Hkv, n_rows;
    int64_t num_blocks;
    double scale;
    double *out, *lse;
    long next;  /* shared work counter over (row, head) items */
    int status;
    int kv_fp8;
    double k_scale, v_scale;
} attn_job;

double oracle_e4m3_to_double(uint8_t c);

/* Element d of cache row `row` (an element index) as a double: a bf16 pattern, or an
 * e4m3 code times the cache's scale. */
static double kv_elem(const attn_job *jb, const void *cache, size_t idx, double scale)
{
    if (jb->kv_fp8) return oracle_e4m3_to_double(((const uint8_t *)cache)[idx]) * scale;
    return oracle_bf16_to_double(((const uint16_t *)cache)[idx]);
}

static int seq_of_token(const int32_t *cu, int B, int t)
{
    for (int b = 0; b < B; ++b)
        if (t >= cu[b] && t < cu[b + 1]) return b;
    return -1;
}

/* One query row (token t, head h):
 *   s_j = scale * sum_d q[t,h,d] K[j,kv,d] + b[h, min(p - j, R - 1)]  for allowed j
 *   o   = sum_j softmax(s)_j V[j,kv,:],   lse = log sum_j exp(s_j)
 * softmax is evaluated as exp(s_j - max s) / sum exp(s_k - max s), the same quantity. */
static int attend_one(attn_job *jb, int item, double *s)
{
    const int ri = item / jb->Hq, h = item % jb->Hq;
    const int t = jb->rows[ri];
    const int b = seq_of_token(jb->cu_q_lens, jb->B, t);
    if (b < 0) return OR_ERR_ARG;
    const int n = jb->cu_q_lens[b + 1] - jb->cu_q_lens[b];
    const int L = jb->seq_lens[b];
    const int p = L - n + (t - jb->cu_q_lens[b]);
    const int G = jb->Hq / jb->Hkv, kv = h / G;
    const uint16_t *qrow = jb->q + ((size_t)t * jb->Hq + h) * OR_D;
    double qd[OR_D];
    for (int d = 0; d < OR_D; ++d) qd[d] = oracle_bf16_to_double(qrow[d]);

    /* allowed keys: 0 <= p - j, and p - j <= window - 1 when a window is set */
    const int j_lo = (jb->window > 0 && p - jb->window + 1 > 0) ? p - jb->window + 1 : 0;
    const int j_hi = p; /* p <= L - 1 */
    double smax = -INFINITY;
    for (int j = j_lo; j <= j_hi; ++j) {
        const int32_t blk = jb->block_table[(size_t)b * jb->max_blocks + j / OR_PAGE];
        if (blk < 0 || blk >= jb->num_blocks) return OR_ERR_BLOCK;
        const size_t krow = (((size_t)blk * jb->Hkv + kv) * OR_PAGE + j % OR_PAGE) * OR_D;
        double dot = 0.0;
        for (int d = 0; d < OR_D; ++d) dot += qd[d] * kv_elem(jb, jb->k_cache, krow + d, jb->k_scale);
        const int dist = p - j;
        const int bi = dist < jb->R - 1 ? dist : jb->R - 1;
        s[j - j_lo] = jb->scale * dot + (double)jb->bias[(size_t)h * jb->R + bi];
        if (s[j - j_lo] > smax) smax = s[j - j_lo];
    }
    double denom = 0.0, acc[OR_D];
    for (int d = 0; d < OR_D; ++d) acc[d] = 0.0;
    for (int j = j_lo; j <= j_hi; ++j) {
        const double e = exp(s[j - j_lo] - smax);
        denom += e;
        const int32_t blk = jb->block_table[(size_t)b * jb->max_blocks + j / OR_PAGE];
        const size_t vrow = (((size_t)blk * jb->Hkv + kv) * OR_PAGE + j % OR_PAGE) * OR_D;
        for (int d = 0; d < OR_D; ++d) acc[d] += e * kv_elem(jb, jb->v_cache, vrow + d, jb->v_scale);
    }
    double *o = jb->out + ((size_t)ri * jb->Hq + h) * OR_D;
    for (int d = 0; d < OR_D; ++d) o[d] = acc[d] / denom;
    if (jb->lse) jb->lse[(size_t)ri * jb->Hq + h] = smax + log(denom);
    return OR_OK;
}

static void *attn_worker(void *arg)
{
    attn_job *jb = (attn_job *)arg;
    int maxL = 1;
    for (int b = 0; b < jb->B; ++b)
        if (jb->seq_lens[b] > maxL) maxL = jb->seq_lens[b];
    double *s = malloc(sizeof(double) * (size_t)maxL);
    if (!s) { __atomic_store_n(&jb->status, OR_ERR_NOMEM, __ATOMIC_RELAXED); return NULL; }
    const long total = (long)jb->n_rows * jb->Hq;
    for (;;) {
        const long item = __atomic_fetch_add(&jb->next, 1, __ATOMIC_RELAXED);
        if (item >= total) break;
        const int rc = attend_one(jb, (int)item, s);
        if (rc != OR_OK) { __atomic_store_n(&jb->status, rc, __ATOMIC_RELAXED); break; }
    }
    free(s);
    return NULL;
}

/*
 * Attention rows for the listed query tokens (global token indices into q), all heads.
 * q [T][Hq][128]; block_table [B][max_blocks]; bias [Hq][R] fp32;
 * out [n_rows][Hq][128] fp64; lse [n_rows][Hq] fp64 (natural log; may be NULL).
 */
static int run_attn(const uint16_t *q, const void *k_cache, const void *v_cache, int kv_fp8,
                    double k_scale, double v_scale, const int32_t *block_table, int max_blocks,
                    const int32_t *cu_q_lens, const int32_t *seq_lens, const float *bias,
                    int R, double scale, int window, int B, int T, int Hq, int Hkv,
                    int64_t num_blocks, const int32_t *rows, int n_rows, double *out,
                    double *lse, int n_threads)
{
    if (B <= 0 || T < 0 || Hq <= 0 || Hkv <= 0 || Hq % Hkv != 0 || R < 1 || window < 0 ||
        n_rows < 0 || max_blocks <= 0)
        return OR_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        const int n = cu_q_lens[b + 1] - cu_q_lens[b];
        if (n < 0 || seq_lens[b] < n || seq_lens[b] > max_blocks * OR_PAGE) return OR_ERR_ARG;
    }
    for (int i = 0; i < n_rows; ++i)
        if (rows[i] < 0 || rows[i] >= T) return OR_ERR_ARG;
    attn_job jb = {q, k_cache, v_cache, block_table, cu_q_lens, seq_lens, rows, bias,
                   max_blocks, R, window, B, T, Hq, Hkv, n_rows, num_blocks, scale,
                   out, lse, 0, OR_OK, kv_fp8, k_scale, v_scale};
    if (n_threads < 1) n_threads = 1;
    if (n_threads > 512) n_threads = 512;
    pthread_t th[512];
    int started = 0;
    for (int i = 0; i < n_threads; ++i) {
        if (pthread_create(&th[i], NULL, attn_worker, &jb) != 0) break;
        ++started;
    }
    if (started == 0) attn_worker(&jb);
    for (int i = 0; i < started; ++i) pthread_join(th[i], NULL);
    return jb.status;
}

int oracle_rel_attn(const uint16_t *q, const uint16_t *k_cache, const uint16_t *v_cache,
                    const int32_t *block_table, int max_blocks, const int32_t *cu_q_lens,
                    const int32_t *seq_lens, const float *bias, int R, double scale,
                    int window, int B, int T, int Hq, int Hkv, int64_t num_blocks,
                    const int32_t *rows, int n_rows, double *out, double *lse, int n_threads)
{
    return run_attn(q, k_cache, v_cache, 0, 1.0, 1.0, block_table, max_blocks, cu_q_lens,
                    seq_lens, bias, R, scale, window, B, T, Hq, Hkv, num_blocks, rows, n_rows,
                    out, lse, n_threads);
}

/* The same attention over an FP8 cache: K = e4m3(code) * k_scale, V = e4m3(code) * v_scale. */
int oracle_rel_attn_fp8(const uint16_t *q, const uint8_t *k_cache, const uint8_t *v_cache,
                        double k_scale, double v_scale, const int32_t *block_table,
                        int max_blocks, const int32_t *cu_q_lens, const int32_t *seq_lens,
                        const float *bias, int R, double scale, int window, int B, int T,
                        int Hq, int Hkv, int64_t num_blocks, const int32_t *rows, int n_rows,
                        double *out, double *lse, int n_threads)
{
    return run_attn(q, k_cache, v_cache, 1, k_scale, v_scale, block_table, max_blocks,
                    cu_q_lens, seq_lens, bias, R, scale, window, B, T, Hq, Hkv, num_blocks,
                    rows, n_rows, out, lse, n_threads);
}

/* ------------------------------------------------- sconv on a dense stream ---- */

/*
 * The same window-4 causal conv on one dense stream (the blog's "Model Architecture /
 * Sconv" also applies sconv to the attention output and the MoE output), with its own
 * 3-row cache and a dense output:
 *   x~ = [state[b] rows 0..2 ; new rows of b],  y[t] = bf16(sum_j w[c][j] x~[t + j])
 *   state[b] <- last 3 rows of x~
 * x, y [T][C] bf16; w [C][4]; state [B][3][C] bf16 (in/out).
 */
int oracle_sconv_dense(const uint16_t *x, const float *w, uint16_t *state,
                       const int32_t *cu_q_lens, uint16_t *y, int B, int T, int C)
{
    if (B < 0 || T < 0 || C <= 0) return OR_ERR_ARG;
    if (cu_q_lens[0] != 0 || cu_q_lens[B] != T) return OR_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        const int t0 = cu_q_lens[b];
        const int n = cu_q_lens[b + 1] - t0;
        if (n < 0) return OR_ERR_ARG;
        uint16_t *st = state + (size_t)b * 3 * C;
        uint16_t *ext = malloc(sizeof(uint16_t) * (size_t)(n + 3) * C);
        if (!ext) return OR_ERR_NOMEM;
        memcpy(ext, st, sizeof(uint16_t) * 3 * (size_t)C);
        memcpy(ext + 3 * (size_t)C, x + (size_t)t0 * C, sizeof(uint16_t) * (size_t)n * C);
        for (int t = 0; t < n; ++t)
            for (int c = 0; c < C; ++c) {
                double acc = 0.0;
                for (int j = 0; j < OR_TAPS; ++j)
                    acc += (double)w[(size_t)c * OR_TAPS + j] *
                           oracle_bf16_to_double(ext[(size_t)(t + j) * C + c]);
                y[(size_t)(t0 + t) * C + c] = oracle_bf16_round(acc);
            }
        memcpy(st, ext + (size_t)n * C, sizeof(uint16_t) * 3 * (size_t)C);
        free(ext);
    }
    return OR_OK;
}

/*
 * Sconv-cache rollback after a speculative (MTP) verify step (blog, "Model Architecture /
 * MTP" and "Re-computing MTP KV cache": drafts can be rejected): only the first
 * accepted[b] of the step's n_b new tokens are kept, so the cache must hold the last 3 raw
 * rows of [state before the step ; the first accepted[b] new rows].  streams = 2 for the
 * K/V pair layout of oracle_sconv_kv ([B][2][3][C] state, k and v rows), 1 for a dense
 * stream ([B][3][C], rows in x0).  The conv outputs of the kept tokens need no change:
 * the conv is causal.
 */
int oracle_sconv_rollback(const uint16_t *state_before, const uint16_t *x0,
                          const uint16_t *x1, const int32_t *cu_q_lens,
                          const int32_t *accepted, uint16_t *state_after, int B, int C,
                          int streams)
{
    if (B < 0 || C <= 0 || (streams != 1 && streams != 2)) return OR_ERR_ARG;
    for (int b = 0; b < B; ++b) {
        const int t0 = cu_q_lens[b];
        const int n = cu_q_lens[b + 1] - t0;
        const int a = accepted[b];
        if (n < 0 || a < 0 || a > n) return OR_ERR_ARG;
        for (int s = 0; s < streams; ++s) {
            const uint16_t *x = s == 0 ? x0 : x1;
            const uint16_t *sb = state_before + ((size_t)b * streams + s) * 3 * C;
            uint16_t *sa = state_after + ((size_t)b * streams + s) * 3 * C;
            for (int r = 0; r < 3; ++r) {
                /* row r of the new state is row (a + r) of [state_before ; kept rows] */
                const int e = a + r;
                const uint16_t *src = e < 3 ? sb + (size_t)e * C : x + (size_t)(t0 + e - 3) * C;
                memcpy(sa + (size_t)r * C, src, sizeof(uint16_t) * (size_t)C);
            }
        }
    }
    return OR_OK;
}

/* ------------------------------------------------------------ FP8 (E4M3) ---- */

/* e4m3 code -> double, exact.  Bit 7 sign, bits 6..3 exponent (bias 7), bits 2..0
 * mantissa; exponent 0 holds subnormals m * 2^-9; S.1111.111 is NaN (no infinities), so
 * the largest finite value is 1.75 * 2^8 = 448. */
double oracle_e4m3_to_double(uint8_t c)
{
    const int e = (c >> 3) & 15, m = c & 7;
    if (e == 15 && m == 7) return NAN;
    const double v = e == 0 ? ldexp((double)m, -9) : ldexp((double)(8 + m), e - 10);
    return (c & 0x80) ? -v : v;
}

/* double -> e4m3 code, round to nearest with ties to even, saturating: |y| >= 448 gives
 * +-448, NaN gives 0x7f.  The non-negative finite codes 0..126 increase with their value,
 * so the two neighbours of |y| are found by walking the codes; on a tie the even code
 * (mantissa LSB 0) wins. */
uint8_t oracle_e4m3_round(double y)
{
    if (isnan(y)) return 0x7f;
    const uint8_t sign = signbit(y) ? 0x80 : 0;
    const double a = fabs(y);
    if (a >= 448.0) return sign | 0x7e;
    int lo = 0;
    while (lo < 126 && oracle_e4m3_to_double((uint8_t)(lo + 1)) <= a) ++lo;
    const double vlo = oracle_e4m3_to_double((uint8_t)lo);
    if (vlo == a) return sign | (uint8_t)lo;
    const double vhi = oracle_e4m3_to_double((uint8_t)(lo + 1));
    const double dlo = a - vlo, dhi = vhi - a;
    const int c = dlo < dhi ? lo : (dhi < dlo ? lo + 1 : ((lo & 1) ? lo + 1 : lo));
    return sign | (uint8_t)c;
}

/*
 * oracle_sconv_kv with an FP8 cache: the same conv sum y in fp64, stored as
 * e4m3(y / k_scale) in the K cache and e4m3(y / v_scale) in the V cache; the state update
 * is unchanged.  Caches [num_blocks][Hkv][128][128] bytes.
 */
int oracle_sconv_kv_fp8(const uint16_t *k_raw, const uint16_t *v_raw, const float *w_k,
                        const float *w_v, uint16_t *state, const int32_t *cu_q_lens,
                        const int64_t *slot_mapping, uint8_t *k_cache, uint8_t *v_cache,
                        double k_scale, double v_scale, int B, int T, int Hkv,
                        int64_t num_blocks)
{
    if (B < 0 || T < 0 || Hkv <= 0 || num_blocks < 0 || !(k_scale > 0) || !(v_scale > 0))
        return OR_ERR_ARG;
    if (cu_q_lens[0] != 0 || cu_q_lens[B] != T) return OR_ERR_ARG;
    const int C = Hkv * OR_D;
    for (int b = 0; b < B; ++b) {
        const int t0 = cu_q_lens[b];
        const int n = cu_q_lens[b + 1] - t0;
        if (n < 0) return OR_ERR_ARG;
        for (int which = 0; which < 2; ++which) {
            const uint16_t *x = which == 0 ? k_raw : v_raw;
            const float *w = which == 0 ? w_k : w_v;
            uint8_t *cache = which == 0 ? k_cache : v_cache;
            const double scale = which == 0 ? k_scale : v_scale;
            uint16_t *st = state + ((size_t)b * 2 + which) * 3 * C;
            uint16_t *ext = malloc(sizeof(uint16_t) * (size_t)(n + 3) * C);
            if (!ext) return OR_ERR_NOMEM;
            memcpy(ext, st, sizeof(uint16_t) * 3 * (size_t)C);
            memcpy(ext + 3 * (size_t)C, x + (size_t)t0 * C, sizeof(uint16_t) * (size_t)n * C);
            for (int t = 0; t < n; ++t) {
                const int64_t slot = slot_mapping[t0 + t];
                if (slot < 0) continue;
                if (slot >= num_blocks * OR_PAGE) { free(ext); return OR_ERR_BLOCK; }
                const int64_t blk = slot / OR_PAGE, off = slot % OR_PAGE;
                for (int c = 0; c < C; ++c) {
                    double y = 0.0;
                    for (int j = 0; j < OR_TAPS; ++j)
                        y += (double)w[(size_t)c * OR_TAPS + j] *
                             oracle_bf16_to_double(ext[(size_t)(t + j) * C + c]);
                    const int h = c / OR_D, d = c % OR_D;
                    cache[(((size_t)blk * Hkv + h) * OR_PAGE + off) * OR_D + d] =
                        oracle_e4m3_round(y / scale);
                }
            }
            memcpy(st, ext + (size_t)n * C, sizeof(uint16_t) * 3 * (size_t)C);
            free(ext);
        }
    }
    return OR_OK;
}
