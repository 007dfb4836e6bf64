/*
 * Relay decode attention -- CPU ORACLE.  TEST INFRASTRUCTURE ONLY.
 *
 * This file is the slow, obviously correct definition that the CUDA library
 * is checked against.  Only the tests, the smoke check and the benchmark's
 * CPU-baseline leg may load it; the library itself never does.  It shares no
 * code, header, table or helper with the CUDA path.
 *
 * What it computes (RelayAttention for Efficient Large Language Model Serving
 * with Long System Prompts, arXiv 2402.14808, Abstract: the method is "a
 * mathematical reformulation of causal attention", so it must give exactly
 * causal attention):
 *
 *   for every request b, query row i < q_lens[b], head h:
 *     keys   = [ system keys 0..Ls-1 ;  context keys t = 0..v-1 ]  of KV head
 *              h / (H / Hkv)   (grouped-query attention: H / Hkv consecutive
 *              query heads share one KV head; Hkv = H is multi-head)
 *     v      = max(0, ctx_lens[b] - q_lens[b] + 1 + i)      (causal visibility:
 *              the query rows are the last q_lens[b] positions of the context)
 *     s_j    = scale * <q[b,i,h], k_j>
 *     out    = sum_j softmax(s)_j v_j,   lse = log sum_j exp(s_j)
 *
 * Context key t of request b lives in the paged pool at block
 * block_tables[b][t / bs], row t % bs (PagedAttention block tables; the pool
 * layout is [num_blocks, Hkv, bs, D]).  System keys live in a separate cache
 * [Ls, Hkv, D] (atyun.com RelayAttention article, section "RelayAttention": a
 * separate cache for the system KVs, filled offline).
 *
 * A second set of entry points computes the method's three steps separately
 * (same article, section "RelayAttention": system attention, context
 * attention, and relay fusion as a convex combination of the two), so tests
 * can check that the steps reproduce the direct definition.
 *
 * Precision: every input is fp16 (decoded exactly below); all arithmetic is
 * IEEE double in the order written.  No blocking, no fusion, no reordering.
 *
 * Parity pins (tests, CPU only): a hand-worked example, closed forms (single
 * key, all-equal scores), brute force with numpy matrices, fp64 scaled dot
 * product attention from torch over the explicit concatenation, the relay
 * identity, the empty-segment special cases, pool relabelling invariance.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

typedef struct {
    int32_t B, Lq, H, D, Ls, block_size, num_blocks, max_blocks;
    int32_t Hkv;      /* KV heads of the caches; H is a multiple of Hkv */
    double scale;
} oracle_dims_t;

enum { ORACLE_OK = 0, ORACLE_BAD_ARG = 1, ORACLE_BAD_BLOCK = 2 };
enum { PART_FULL = 0, PART_SYS = 1, PART_CTX = 2 };

/* IEEE 754 binary16 -> double, straight from the format's definition:
 * sign, 5-bit exponent (bias 15), 10-bit fraction; exponent 0 is subnormal. */
static double half_to_double(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);
    else if (e == 31)
        v = m ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + m), e - 25);
    return sign ? -v : v;
}

/* Plain softmax attention of one query over an explicit list of n keys.
 * n == 0: no keys at all -> out = 0, lse = -inf (convention for an empty
 * segment; the pages are silent on it). */
static void attend(const uint16_t *qrow, int D, double scale, int n,
                   const uint16_t *const *krows, const uint16_t *const *vrows,
                   double *scores, double *out, double *lse)
{
    for (int d = 0; d < D; d++) out[d] = 0.0;
    if (n == 0) {
        *lse = -INFINITY;
        return;
    }
    double smax = -INFINITY;
    for (int j = 0; j < n; j++) {
        double dot = 0.0;
        for (int d = 0; d < D; d++)
            dot += half_to_double(qrow[d]) * half_to_double(krows[j][d]);
        scores[j] = scale * dot;
        if (scores[j] > smax) smax = scores[j];
    }
    double denom = 0.0;
    for (int j = 0; j < n; j++) {
        scores[j] = exp(scores[j] - smax);
        denom += scores[j];
    }
    for (int j = 0; j < n; j++) {
        double p = scores[j] / denom;
        for (int d = 0; d < D; d++) out[d] += p * half_to_double(vrows[j][d]);
    }
    *lse = smax + log(denom);
}

/* Number of context positions query row i of request b may see. */
static int visible_ctx(int n_ctx, int q_len, int i)
{
    int v = n_ctx - q_len + 1 + i;
    if (v < 0) v = 0;
    if (v > n_ctx) v = n_ctx;
    return v;
}

/* Attention for a list of output rows (b, i, h) over the keys selected by
 * `part`: the concatenation (PART_FULL), the system prompt only (PART_SYS),
 * or the request's visible context only (PART_CTX).
 * out: [n_rows, D], lse: [n_rows] (natural log). */
int oracle_attention_rows(const oracle_dims_t *dm, int part,
                          const uint16_t *q, const uint16_t *sys_k, const uint16_t *sys_v,
                          const uint16_t *k_cache, const uint16_t *v_cache,
                          const int32_t *block_tables, const int32_t *ctx_lens,
                          const int32_t *q_lens, int64_t n_rows,
                          const int32_t *row_b, const int32_t *row_i, const int32_t *row_h,
                          double *out, double *lse, int n_threads)
{
    if (!dm || !out || !lse || n_rows < 0) return ORACLE_BAD_ARG;
    const int B = dm->B, Lq = dm->Lq, H = dm->H, D = dm->D, Ls = dm->Ls, Hkv = dm->Hkv;
    const int bs = dm->block_size, MB = dm->max_blocks;
    if (D <= 0 || H <= 0 || bs <= 0 || Ls < 0 || Hkv <= 0 || H % Hkv != 0) return ORACLE_BAD_ARG;
    const int group = H / Hkv;   /* query heads per KV head */

    /* Validate every row and every block id before computing anything. */
    for (int64_t r = 0; r < n_rows; r++) {
        int b = row_b[r], i = row_i[r], h = row_h[r];
        if (b < 0 || b >= B || h < 0 || h >= H || i < 0 || i >= Lq) return ORACLE_BAD_ARG;
        int ql = q_lens ? q_lens[b] : Lq;
        if (i >= ql) return ORACLE_BAD_ARG;
        int n = ctx_lens[b];
        if (n < 0 || n > MB * bs) return ORACLE_BAD_ARG;
        for (int t = 0; t < n; t += bs) {
            int blk = block_tables[(int64_t)b * MB + t / bs];
            if (blk < 0 || blk >= dm->num_blocks) return ORACLE_BAD_BLOCK;
        }
    }

    int max_keys = Ls;
    for (int b = 0; b < B; b++) max_keys = (ctx_lens[b] + Ls > max_keys) ? ctx_lens[b] + Ls : max_keys;
    if (max_keys < 1) max_keys = 1;

#ifdef _OPENMP
    /* n_threads > 0 applies to this call only */
    const int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
#else
    (void)n_threads;
#endif

#pragma omp parallel num_threads(nt)
    {
        const uint16_t **krows = (const uint16_t **)malloc(sizeof(void *) * (size_t)max_keys);
        const uint16_t **vrows = (const uint16_t **)malloc(sizeof(void *) * (size_t)max_keys);
        double *scores = (double *)malloc(sizeof(double) * (size_t)max_keys);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; r++) {
            int b = row_b[r], i = row_i[r], h = row_h[r];
            int hk = h / group;   /* the KV head this query head reads */
            int ql = q_lens ? q_lens[b] : Lq;
            int n = 0;
            if (part != PART_CTX) {
                for (int t = 0; t < Ls; t++) {
                    krows[n] = sys_k + ((int64_t)t * Hkv + hk) * D;
                    vrows[n] = sys_v + ((int64_t)t * Hkv + hk) * D;
                    n++;
                }
            }
            if (part != PART_SYS) {
                int v = visible_ctx(ctx_lens[b], ql, i);
                for (int t = 0; t < v; t++) {
                    int64_t blk = block_tables[(int64_t)b * MB + t / bs];
                    int64_t row = (blk * Hkv + hk) * bs + t % bs;
                    krows[n] = k_cache + row * D;
                    vrows[n] = v_cache + row * D;
                    n++;
                }
            }
            const uint16_t *qrow = q + (((int64_t)b * Lq + i) * H + h) * D;
            attend(qrow, D, dm->scale, n, krows, vrows, scores, out + r * D, lse + r);
        }
        free(krows);
        free(vrows);
        free(scores);
    }
    return ORACLE_OK;
}

/* Prefill attention of the system prompt (atyun.com RelayAttention article,
 * section "RelayAttention": the system KVs are computed offline into their
 * own cache): causal self-attention of its Ls tokens.  Row (t, h) attends to
 * system keys 0..t of KV head h / (H / Hkv):
 *     out = sum_{j<=t} softmax(scale * <q_sys[t,h], k_j>) v_j,  lse = log sum exp.
 * q_sys [Ls, H, D], sys_k / sys_v [Ls, Hkv, D] (fp16 bit patterns); only the
 * (t, h) rows listed are computed. */
int oracle_sys_prefill(const oracle_dims_t *dm, const uint16_t *q_sys, const uint16_t *sys_k,
                       const uint16_t *sys_v, int64_t n_rows, const int32_t *row_t, const int32_t *row_h,
                       double *out, double *lse, int n_threads)
{
    if (!dm || !q_sys || !sys_k || !sys_v || !out || !lse || n_rows < 0) return ORACLE_BAD_ARG;
    const int H = dm->H, D = dm->D, Ls = dm->Ls, Hkv = dm->Hkv;
    if (D <= 0 || H <= 0 || Ls <= 0 || Hkv <= 0 || H % Hkv != 0) return ORACLE_BAD_ARG;
    for (int64_t r = 0; r < n_rows; r++)
        if (row_t[r] < 0 || row_t[r] >= Ls || row_h[r] < 0 || row_h[r] >= H) return ORACLE_BAD_ARG;
    const int group = H / Hkv;
#ifdef _OPENMP
    /* n_threads > 0 applies to this call only */
    const int nt = n_threads > 0 ? n_threads : omp_get_max_threads();
#else
    (void)n_threads;
#endif
#pragma omp parallel num_threads(nt)
    {
        const uint16_t **krows = (const uint16_t **)malloc(sizeof(void *) * (size_t)Ls);
        const uint16_t **vrows = (const uint16_t **)malloc(sizeof(void *) * (size_t)Ls);
        double *scores = (double *)malloc(sizeof(double) * (size_t)Ls);
#pragma omp for schedule(dynamic, 1)
        for (int64_t r = 0; r < n_rows; r++) {
            int t = row_t[r], h = row_h[r], hk = h / group;
            for (int j = 0; j <= t; j++) {
                krows[j] = sys_k + ((int64_t)j * Hkv + hk) * D;
                vrows[j] = sys_v + ((int64_t)j * Hkv + hk) * D;
            }
            attend(q_sys + ((int64_t)t * H + h) * D, D, dm->scale, t + 1, krows, vrows, scores, out + r * D, lse + r);
        }
        free(krows);
        free(vrows);
        free(scores);
    }
    return ORACLE_OK;
}

/* Rotary position embedding with the system-prompt offset (atyun.com
 * RelayAttention article, section "RelayAttention": the request tokens'
 * positions are shifted by the system prompt's length).  Row i < q_lens[b]
 * of request b is at position p = Ls + ctx_lens[b] - q_lens[b] + i; for
 * j < D/2 the pair (x[j], x[j + D/2]) is rotated by the angle
 * p * base^(-2j/D).  x: [B, Lq, heads, D] fp16 bit patterns; out (fp64, same
 * shape) receives the rotated rows; rows i >= q_lens[b] are NaN. */
int oracle_rope(const oracle_dims_t *dm, double base, int heads, const int32_t *ctx_lens,
                const int32_t *q_lens, const uint16_t *x, double *out)
{
    if (!dm || !x || !out || !ctx_lens || heads < 1 || dm->D < 2 || dm->D % 2 || !(base > 1.0)) return ORACLE_BAD_ARG;
    const int B = dm->B, Lq = dm->Lq, D = dm->D, half = dm->D / 2;
    for (int b = 0; b < B; b++) {
        int ql = q_lens ? q_lens[b] : Lq;
        if (ql < 0 || ql > Lq || ctx_lens[b] < ql) return ORACLE_BAD_ARG;
    }
    for (int b = 0; b < B; b++) {
        int ql = q_lens ? q_lens[b] : Lq;
        for (int i = 0; i < Lq; i++) {
            double p = (double)dm->Ls + (double)(ctx_lens[b] - ql + i);
            for (int h = 0; h < heads; h++) {
                const uint16_t *xr = x + (((int64_t)b * Lq + i) * heads + h) * D;
                double *o = out + (((int64_t)b * Lq + i) * heads + h) * D;
                for (int j = 0; j < half; j++) {
                    if (i >= ql) {
                        o[j] = o[j + half] = NAN;
                        continue;
                    }
                    double ang = p * pow(base, -2.0 * j / D);
                    double c = cos(ang), s = sin(ang);
                    double x0 = half_to_double(xr[j]), x1 = half_to_double(xr[j + half]);
                    o[j] = x0 * c - x1 * s;
                    o[j + half] = x1 * c + x0 * s;
                }
            }
        }
    }
    return ORACLE_OK;
}

/* KV append, the cache write that precedes attention in a decode step: row
 * i < q_lens[b] of request b is context position pos = ctx_lens[b] -
 * q_lens[b] + i (its new token is the last of the context), and its K and V
 * rows of every KV head hk are copied into the pool at block
 * block_tables[b][pos / bs], row pos % bs.  k_new, v_new are [B, Lq, Hkv, D]
 * fp16 bit patterns; the pools are updated in place.  Everything is checked
 * before anything is written. */
int oracle_kv_append(const oracle_dims_t *dm, const uint16_t *k_new, const uint16_t *v_new,
                     const int32_t *block_tables, const int32_t *ctx_lens, const int32_t *q_lens,
                     uint16_t *k_cache, uint16_t *v_cache)
{
    if (!dm || !k_new || !v_new || !block_tables || !ctx_lens || !k_cache || !v_cache) return ORACLE_BAD_ARG;
    const int B = dm->B, Lq = dm->Lq, D = dm->D, Hkv = dm->Hkv, bs = dm->block_size, MB = dm->max_blocks;
    if (B < 0 || Lq < 1 || D < 1 || Hkv < 1 || bs < 1 || MB < 1) return ORACLE_BAD_ARG;
    for (int b = 0; b < B; b++) {
        int ql = q_lens ? q_lens[b] : Lq, n = ctx_lens[b];
        if (ql < 0 || ql > Lq || n < ql || n > MB * bs) return ORACLE_BAD_ARG;
        for (int i = 0; i < ql; i++) {
            int pos = n - ql + i;
            int blk = block_tables[(int64_t)b * MB + pos / bs];
            if (blk < 0 || blk >= dm->num_blocks) return ORACLE_BAD_BLOCK;
        }
    }
    for (int b = 0; b < B; b++) {
        int ql = q_lens ? q_lens[b] : Lq, n = ctx_lens[b];
        for (int i = 0; i < ql; i++) {
            int pos = n - ql + i;
            int64_t blk = block_tables[(int64_t)b * MB + pos / bs];
            for (int hk = 0; hk < Hkv; hk++) {
                int64_t src = (((int64_t)b * Lq + i) * Hkv + hk) * D;
                int64_t dst = ((blk * Hkv + hk) * bs + pos % bs) * D;
                for (int d = 0; d < D; d++) {
                    k_cache[dst + d] = k_new[src + d];
                    v_cache[dst + d] = v_new[src + d];
                }
            }
        }
    }
    return ORACLE_OK;
}

/* Relay fusion of two partial results (atyun.com RelayAttention article,
 * section "RelayAttention": the final output is a convex combination of the
 * system-only and context-only outputs).  The weights that make the
 * combination equal attention over the concatenation are each part's share
 * of the total softmax mass, exp(lse_part) / (exp(lse_sys) + exp(lse_ctx)).
 * alpha_sys receives the system weight; the context weight is 1 - alpha_sys.
 * Both parts empty (both lse = -inf): out = 0, lse = -inf, alpha_sys = NaN. */
void oracle_relay_fuse(int64_t n_rows, int D,
                       const double *o_sys, const double *lse_sys,
                       const double *o_ctx, const double *lse_ctx,
                       double *out, double *lse_out, double *alpha_sys)
{
    for (int64_t r = 0; r < n_rows; r++) {
        double ls = lse_sys[r], lc = lse_ctx[r];
        if (ls == -INFINITY && lc == -INFINITY) {
            for (int d = 0; d < D; d++) out[r * D + d] = 0.0;
            lse_out[r] = -INFINITY;
            alpha_sys[r] = NAN;
            continue;
        }
        double m = ls > lc ? ls : lc;
        double ws = exp(ls - m);
        double wc = exp(lc - m);
        double a = ws / (ws + wc);
        double c = wc / (ws + wc);
        for (int d = 0; d < D; d++)
            out[r * D + d] = a * o_sys[r * D + d] + c * o_ctx[r * D + d];
        lse_out[r] = m + log(ws + wc);
        alpha_sys[r] = a;
    }
}

/* Threads the OpenMP runtime would use for the next parallel region. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Exposed for the decoder pin: decode n fp16 bit patterns. */
void oracle_half_to_double(int64_t n, const uint16_t *h, double *out)
{
    for (int64_t k = 0; k < n; k++) out[k] = half_to_double(h[k]);
}
