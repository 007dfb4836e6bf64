/*
 * relay.h -- C ABI of librelay.so: RelayAttention decode attention on GB300.
 *
 * The operation (RelayAttention for Efficient Large Language Model Serving
 * with Long System Prompts, arXiv 2402.14808, Abstract; atyun.com article on
 * RelayAttention, section "RelayAttention"): causal attention for a batch of
 * requests that all share one system prompt, computed in three steps --
 *   1. system attention: every query row of the batch against the shared
 *      system-prompt KV cache, which is read from memory once per batch
 *      (the per-request matrix-vector products become one matrix-matrix
 *      product per head);
 *   2. context attention: every query row against its own request's paged
 *      context KV cache;
 *   3. relay fusion: the two partial outputs combined as a convex
 *      combination weighted by each part's softmax mass (its log-sum-exp).
 * The result equals causal attention over the concatenation
 * [system prompt; request context] exactly, up to rounding.
 *
 * Entry points: relay_attention_decode (all three steps; also an
 * allocation-free variant), relay_sys_attn / relay_ctx_attn / relay_fuse
 * (the steps one at a time), relay_attention_decode_prefixes (a tree of
 * shared prefixes in one unit) and relay_fuse_n (fusion of K parts, for
 * composing such a tree from the separate steps), relay_baseline_decode (the
 * non-relay formulation), and
 * the steps on either side of the path: relay_kv_append (cache write),
 * relay_rope (rotary positions offset by the system prompt) and
 * relay_sys_prefill (causal attention of the system prompt itself).
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - fp16 arrays are IEEE binary16 (`const void*` here); accumulation is fp32.
 *  - Every pointer is a DEVICE pointer unless stated otherwise; the caller
 *    owns every buffer, including the workspace.  The library never
 *    allocates, frees or synchronises (except relay_device_status, which
 *    says so).  All work is queued on `stream`; the calls return at once.
 *  - Layouts are contiguous, row-major:
 *      q, out             [B, Lq, H, D]            fp16
 *      sys_k, sys_v       [Ls, Hkv, D]             fp16
 *      k_cache, v_cache   [num_blocks, Hkv, 16, D] fp16 (paged pool; one
 *                                                  head of one block is 16
 *                                                  contiguous rows of D)
 *      block_tables       [B, max_blocks_per_seq]  int32 (physical block of
 *                                                  context token t of request
 *                                                  b is block_tables[b][t/16],
 *                                                  row t%16)
 *      ctx_lens           [B]                      int32 context tokens
 *      q_lens             [B]                      int32 query rows (nullable:
 *                                                  every request has Lq)
 *      lse arrays         [B, Lq, H]               fp32, natural log
 *      o_sys, o_ctx       [B, Lq, H, D]            fp32
 *    q, out, sys_k, sys_v, k_cache, v_cache must be 16-byte aligned.
 *  - Hkv KV heads serve H query heads (grouped-query attention; Hkv = H is
 *    multi-head, Hkv = 1 multi-query): query head h reads KV head
 *    h / (H / Hkv), i.e. each run of H / Hkv consecutive query heads shares
 *    one KV head.
 *  - Query row i of request b is context position ctx_lens[b]-q_lens[b]+i;
 *    it sees the whole system prompt and context tokens
 *    t < max(0, ctx_lens[b] - q_lens[b] + 1 + i).  Rows i >= q_lens[b] of
 *    the outputs are left untouched.
 *  - A row with no visible key at all gets out = 0 and lse = -inf.
 *  - Supported: D in {64, 128}; block size 16; B <= 512; any Hkv that
 *    divides H (Hkv = 0 means Hkv = H); B*Lq, B*H, B*Lq*H and
 *    16*max_blocks_per_seq + Ls each below 2^30 (32-bit counters on the
 *    device).  Other shapes return RELAY_ERR_UNSUPPORTED; an Hkv that does
 *    not divide H returns RELAY_ERR_INVALID_ARG.
 *  - Errors: argument problems are found on the host before anything is
 *    queued and returned synchronously.  Launch failures return
 *    RELAY_ERR_CUDA.  Values that can only be checked on the device (a
 *    q_lens or ctx_lens entry out of range, a block id outside the pool, a
 *    sum of q_lens above the bound) set a flag word in the workspace; the
 *    kernel then skips the bad access (or the whole batch), and
 *    relay_device_status reports it.  Nothing traps.
 */
#ifndef RELAY_H
#define RELAY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    RELAY_OK = 0,
    RELAY_ERR_INVALID_ARG = 1,   /* null/misaligned pointer, negative size, ... */
    RELAY_ERR_UNSUPPORTED = 2,   /* valid but outside the supported shapes */
    RELAY_ERR_WORKSPACE = 3,     /* workspace missing or smaller than required */
    RELAY_ERR_CUDA = 4,          /* a CUDA runtime call or launch failed */
    RELAY_ERR_DEVICE_CHECK = 5,  /* relay_device_status: a device-side check failed */
    RELAY_ERR_TIMEOUT = 6        /* reserved: a bounded device wait gave up */
} relay_status_t;

/* Device-side check flags (bit mask reported by relay_device_status). */
#define RELAY_FLAG_BAD_Q_LEN    1u  /* q_lens[b] outside [0, Lq] */
#define RELAY_FLAG_BAD_CTX_LEN  2u  /* ctx_lens[b] outside [0, 16*max_blocks_per_seq] */
#define RELAY_FLAG_BAD_BLOCK    4u  /* a block id outside [0, num_blocks) */
#define RELAY_FLAG_Q_TOTAL      8u  /* sum of q_lens above max_q_total */
#define RELAY_FLAG_WAIT_TIMEOUT 16u  /* a bounded wait inside the tensor-core kernel gave up;
                                       that call's outputs are not valid */

/* Opaque CUDA stream (binary-compatible with cudaStream_t); NULL = legacy stream. */
typedef struct CUstream_st *relay_stream_t;

/* Problem shape.  Value semantics; the library keeps no pointer to it. */
typedef struct {
    int32_t B;                  /* requests in the batch (0: nothing to do) */
    int32_t Lq;                 /* query-row stride of q/out (max q_lens) */
    int32_t H;                  /* heads */
    int32_t D;                  /* head dimension: 64 or 128 */
    int32_t Ls;                 /* system-prompt tokens (0 allowed) */
    int32_t block_size;         /* paged block size: must be 16 */
    int32_t num_blocks;         /* blocks in the paged pool */
    int32_t max_blocks_per_seq; /* row stride of block_tables */
    int32_t max_q_total;        /* bound on sum(q_lens); 0 means B*Lq.  A call
                                   without q_lens needs 0 or >= B*Lq, else it
                                   returns RELAY_ERR_INVALID_ARG */
    int32_t ctx_split;          /* context keys per work item for 1-row requests;
                                   0 = automatic; else a multiple of 64 */
    int32_t sys_range;          /* system keys per work item; 0 = automatic;
                                   else a multiple of 64 */
    float scale;                /* softmax scale; <= 0 means 1/sqrt(D) */
    int32_t Hkv;                /* KV heads of sys_k/sys_v and the pool; 0 means H
                                   (multi-head); else H must be a multiple of it */
} relay_dims_t;

/* Bytes of workspace any entry point below needs for `dims` (0 if `dims` is
 * invalid).  The workspace holds fp32 partial results of the work items, the
 * schedule handed from the first kernel to the merge kernel, and the work
 * queue counters.  It must be zero-filled once when first allocated (or by
 * relay_workspace_init); every call leaves its counters at zero again.
 * Calls that share one workspace must be ordered (same stream, or events). */
size_t relay_workspace_size(const relay_dims_t *dims);

/* Queue a zero-fill of the workspace's counter header on `stream`. */
relay_status_t relay_workspace_init(void *ws, size_t ws_bytes, relay_stream_t stream);

/* Step 1, system attention (atyun.com RelayAttention article, section
 * "RelayAttention": the intermediate output as if only the shared system
 * prompt were present).  For every valid row: o_sys = softmax(scale q K_sys^T)
 * V_sys over all Ls system tokens, lse_sys its natural-log normaliser.
 * Ls == 0 gives o_sys = 0, lse_sys = -inf. */
relay_status_t relay_sys_attn(const relay_dims_t *dims, const void *q,
                              const void *sys_k, const void *sys_v, const int32_t *q_lens,
                              float *o_sys, float *lse_sys,
                              void *ws, size_t ws_bytes, relay_stream_t stream);

/* Step 2, context attention (same section: the intermediate output as if only
 * the request-specific context were present), over the causally visible
 * context tokens read through the block tables (PagedAttention layout). */
relay_status_t relay_ctx_attn(const relay_dims_t *dims, const void *q,
                              const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, const int32_t *ctx_lens,
                              const int32_t *q_lens, float *o_ctx, float *lse_ctx,
                              void *ws, size_t ws_bytes, relay_stream_t stream);

/* Step 3, relay fusion (same section: the final output is a convex
 * combination of the two intermediate outputs).  With
 * a = exp(lse_sys) / (exp(lse_sys) + exp(lse_ctx)):
 *   out = a * o_sys + (1 - a) * o_ctx   (stored fp16),
 *   lse_out = log(exp(lse_sys) + exp(lse_ctx))   (lse_out nullable).
 * Both lse = -inf gives out = 0, lse_out = -inf.  Needs no workspace. */
relay_status_t relay_fuse(const relay_dims_t *dims, const float *o_sys, const float *lse_sys,
                          const float *o_ctx, const float *lse_ctx, const int32_t *q_lens,
                          void *out, float *lse_out, relay_stream_t stream);

/* All three steps, queued on `stream` as two kernels, or three when the
 * tensor-core kernel runs in front (all of them fit in one CUDA graph):
 *  0. (D = 128, and more than 256 query rows per KV head counting the query
 *     heads of a group, where the system step is compute-bound; or requests
 *     of Lq * H / Hkv >= 64 rows per KV head, whose own contexts are as dense)
 *     a persistent tcgen05 kernel (one CTA per SM at most) computes the
 *     system partials -- items of one KV head, a pair of 128-row tiles and a
 *     range of system keys -- and the context partials of requests with
 *     several rows -- items of one request, a pair of its row tiles and one
 *     KV head, over its whole context; when the batch also has one-row
 *     requests, some of its SMs are left to step 1 from the start;
 *  1. a persistent grid (one CTA per SM), a programmatic dependent of step
 *     0 when that runs, works through system items (one KV head, a range of
 *     system keys, up to 64 query rows of the batch: the system KV is
 *     streamed once per batch) -- unless step 0 took them -- and context
 *     items (one request, one head or head group, a range of its paged
 *     context; those of several-row requests unless step 0 took them); each
 *     item writes an fp32 partial result and its log-sum-exp to the
 *     workspace;
 *  2. a merge kernel, launched as a programmatic dependent of step 1,
 *     combines each (row, head)'s partials -- the system ranges and the
 *     context splits -- into `out` (fp16) and `lse_out` (fp32 natural log,
 *     nullable): the relay fusion, over any number of parts. */
relay_status_t relay_attention_decode(const relay_dims_t *dims, const void *q,
                                      const void *sys_k, const void *sys_v,
                                      const void *k_cache, const void *v_cache,
                                      const int32_t *block_tables, const int32_t *ctx_lens,
                                      const int32_t *q_lens, void *out, float *lse_out,
                                      void *ws, size_t ws_bytes, relay_stream_t stream);

/* Relay fusion of K partial results of the same query rows, 1 <= K <= 16:
 * the convex combination of relay fusion (atyun.com RelayAttention article,
 * section "RelayAttention") generalised from two parts to K, for a tree of
 * shared prefixes (one part per shared level, e.g. a global system prompt
 * and a group prompt, plus the context, each from relay_sys_attn /
 * relay_ctx_attn):  out = sum_k w_k o_k, w_k = exp(lse_k) / sum_j exp(lse_j),
 * lse_out = log sum_k exp(lse_k).  A part whose lse is -inf for a row (an
 * empty segment, or rows relay_sys_attn left untouched after the caller
 * filled lse with -inf) contributes nothing; all K empty gives out = 0,
 * lse = -inf.  o_parts / lse_parts are HOST arrays of K device pointers to
 * [B, Lq, H, D] fp32 and [B, Lq, H] fp32; out [B, Lq, H, D] fp16, lse_out
 * nullable. */
relay_status_t relay_fuse_n(const relay_dims_t *dims, int K, const float *const *o_parts,
                            const float *const *lse_parts, const int32_t *q_lens, void *out,
                            float *lse_out, relay_stream_t stream);

/* Maximum number of shared prefix segments of relay_attention_decode_prefixes. */
#define RELAY_MAX_SEGMENTS 8

/* Bytes of workspace relay_attention_decode_prefixes needs for `dims` and
 * these segment lengths (seg_len: HOST array of n_seg token counts); 0 if
 * invalid.  Sized for the current device (its SM count sets the number of
 * key ranges per segment). */
size_t relay_workspace_size_prefixes(const relay_dims_t *dims, int n_seg, const int32_t *seg_len);

/* All three steps for a tree of shared prefixes in one queued unit (two
 * kernels): relay fusion generalised from one shared system prompt to
 * several shared segments -- e.g. a global system prompt seen by every
 * request and one group prompt per group of requests (the multi-level
 * prefix sharing that the works built on RelayAttention develop; the
 * fusion itself is the convex combination of the atyun.com RelayAttention
 * article, section "RelayAttention", over more than two parts).  Request b
 * attends over the segments s whose bit s is set in seg_mask[b], then its
 * own paged context; each segment's KV is read from memory once per batch,
 * by system items of the streaming kernel (never the tensor-core kernel:
 * for large batches with one prompt, relay_attention_decode is faster), and
 * the merge kernel fuses every segment's key ranges and the context splits
 * of each row by their log-sum-exps.  The result equals causal attention
 * over [the segments it sees, in any order; its context].
 *  - n_seg in [1, RELAY_MAX_SEGMENTS]; seg_k, seg_v, seg_len: HOST arrays of
 *    n_seg entries: device pointers to [seg_len[s], Hkv, D] fp16 (16-byte
 *    aligned; may be NULL when seg_len[s] == 0) and the token counts.
 *  - seg_mask: device [B] uint32 (nullable: every request sees every
 *    segment).  A row that sees no key at all gets out = 0, lse = -inf.
 *  - dims->Ls is not used; the other arguments, layouts and errors are
 *    those of relay_attention_decode, with the workspace sized by
 *    relay_workspace_size_prefixes. */
relay_status_t relay_attention_decode_prefixes(const relay_dims_t *dims, const void *q, int n_seg,
                                               const void *const *seg_k, const void *const *seg_v,
                                               const int32_t *seg_len, const uint32_t *seg_mask,
                                               const void *k_cache, const void *v_cache,
                                               const int32_t *block_tables, const int32_t *ctx_lens,
                                               const int32_t *q_lens, void *out, float *lse_out, void *ws,
                                               size_t ws_bytes, relay_stream_t stream);

/* KV append: the step's new keys and values into the paged context pool (the
 * cache write that precedes attention in every decode iteration; the
 * RelayAttention pages keep the request contexts in the paged cache and move
 * only the system prompt to a separate one, atyun.com RelayAttention article,
 * section "RelayAttention").  Row i < q_lens[b] of request b is context
 * position pos = ctx_lens[b] - q_lens[b] + i (ctx_lens already counts the
 * new tokens, as attention does); its row of every KV head hk is copied
 *     k_cache[blk][hk][pos % 16][:] = k_new[b][i][hk][:]   (and v alike),
 * blk = block_tables[b][pos / 16], bit for bit.  k_new, v_new: [B, Lq, Hkv,
 * D] fp16, 16-byte aligned; dims->num_blocks, max_blocks_per_seq, Hkv as for
 * attention (dims->Ls is not used).  A request whose q_len is outside
 * [0, Lq] or whose ctx_len is below its q_len or above
 * 16*max_blocks_per_seq is skipped, and so is a row whose block id is
 * outside [0, num_blocks); each raises its RELAY_FLAG_* in the workspace
 * (relay_device_status).  ws: at least 256 bytes (only the flag word is
 * used; a workspace sized by relay_workspace_size serves). */
relay_status_t relay_kv_append(const relay_dims_t *dims, const void *k_new, const void *v_new,
                               const int32_t *block_tables, const int32_t *ctx_lens,
                               const int32_t *q_lens, void *k_cache, void *v_cache,
                               void *ws, size_t ws_bytes, relay_stream_t stream);

/* Prefill attention of the system prompt: causal self-attention of its Ls
 * tokens, the attention step of filling the separate system cache offline,
 * once, before serving (atyun.com RelayAttention article, section
 * "RelayAttention": the system KVs are computed offline into their own
 * cache).  Row t (query q_sys[t][h]) attends to system keys 0..t of KV head
 * h / (H / Hkv); out[t][h] = softmax(scale * q K^T) V, lse[t][h] its natural-
 * log normaliser.  q_sys, out: [Ls, H, 128] fp16; sys_k, sys_v: [Ls, Hkv,
 * 128] fp16; lse_out: [Ls, H] fp32 or NULL.  Uses dims->H, D, Ls, Hkv,
 * scale; D must be 128 (it runs on the tcgen05 tensor-core kernel).  ws: at
 * least 256 bytes (flag word for RELAY_FLAG_WAIT_TIMEOUT). */
relay_status_t relay_sys_prefill(const relay_dims_t *dims, const void *q_sys, const void *sys_k,
                                 const void *sys_v, void *out, float *lse_out, void *ws,
                                 size_t ws_bytes, relay_stream_t stream);

/* Rotary position embedding of the step's new rows with the system-prompt
 * offset: the system KVs are computed offline, so the request tokens'
 * positions are shifted by the system prompt's length (atyun.com
 * RelayAttention article, section "RelayAttention").  Row i < q_lens[b] of
 * request b is at position p = Ls + ctx_lens[b] - q_lens[b] + i; q[b][i][h]
 * (every query head) and k_new[b][i][hk] (every KV head; k_new may be NULL)
 * are rotated in place, rotate-half form: for j < D/2 the pair
 * (x[j], x[j + D/2]) turns by the angle p * base^(-2j/D),
 *     x[j] <- x[j] cos - x[j+D/2] sin,   x[j+D/2] <- x[j+D/2] cos + x[j] sin.
 * Angles are computed in fp64, the rotation in fp32, results rounded to
 * fp16.  q: [B, Lq, H, D], k_new: [B, Lq, Hkv, D] fp16; base > 1 (10000 for
 * Llama).  A request with q_len outside [0, Lq] or ctx_len < q_len is skipped
 * and flagged.  ws: at least 256 bytes (flag word). */
relay_status_t relay_rope(const relay_dims_t *dims, void *q, void *k_new, const int32_t *ctx_lens,
                          const int32_t *q_lens, float base, void *ws, size_t ws_bytes,
                          relay_stream_t stream);

/* The non-relay formulation, as a paged-attention system with prefix sharing
 * runs it (atyun.com RelayAttention article, section "RelayAttention": the
 * system KVs are read from memory once per request).  The system prompt's KV
 * sits in the same pool as the contexts, in blocks sys_block_ids[0 ..
 * ceil(Ls/16)-1] (token s in block sys_block_ids[s/16], row s%16), and every
 * request attends over [those Ls tokens; its own context].  dims->Ls is the
 * system-prompt length and dims->num_blocks the size of the whole pool. */
relay_status_t relay_baseline_decode(const relay_dims_t *dims, const void *q,
                                     const void *k_pool, const void *v_pool,
                                     const int32_t *sys_block_ids,
                                     const int32_t *block_tables, const int32_t *ctx_lens,
                                     const int32_t *q_lens, void *out, float *lse_out,
                                     void *ws, size_t ws_bytes, relay_stream_t stream);

/* Maximum scratch of relay_attention_decode_noalloc, in bytes. */
#define RELAY_NOALLOC_SCRATCH_BYTES (32u << 20)

/* relay_attention_decode for callers that cannot allocate device memory at
 * the point of the call -- for example a serving process whose own pool
 * allocator owns all device memory and forbids outside allocations, or a
 * latency-critical decode loop that must not reach cudaMalloc (which can
 * synchronise the device).  The paper has no counterpart: this is a
 * packaging of the same computation.
 *
 * Same arguments as relay_attention_decode except the workspace: the
 * scratch (partials, schedule, queue counters) lives in one fixed buffer of
 * RELAY_NOALLOC_SCRATCH_BYTES compiled into the library, which every GPU that
 * loads the library keeps until the process exits.  Nothing is allocated or
 * freed, by the library or by any library it calls.
 *  - Shapes whose workspace (relay_workspace_size) exceeds the buffer are
 *    rejected with RELAY_ERR_WORKSPACE before anything is queued.
 *  - The first call on a device looks up the buffer's device address (with
 *    that device current); make that first call before any stream capture.
 *  - Every call queues a zero-fill of the buffer's counter header, then the
 *    two kernels.  All calls share the one buffer, which keeps the last
 *    call's contents: calls that may overlap on the GPU (other streams, other
 *    host threads) race and must be serialised by the caller.
 *  - Device-side check flags land in the shared buffer and are cleared by the
 *    next call: read them with relay_noalloc_device_status before that. */
relay_status_t relay_attention_decode_noalloc(const relay_dims_t *dims, const void *q,
                                              const void *sys_k, const void *sys_v,
                                              const void *k_cache, const void *v_cache,
                                              const int32_t *block_tables, const int32_t *ctx_lens,
                                              const int32_t *q_lens, void *out, float *lse_out,
                                              relay_stream_t stream);

/* Read and clear the device-side check flags that the last
 * relay_attention_decode_noalloc call on the current device raised (a block
 * id outside the pool, a q_lens or ctx_lens entry out of range, ...: the
 * kernels skip those accesses, and without this call the caller could not
 * tell).  SYNCHRONOUS: waits for `stream`, which must be ordered after that
 * call.  *flags_out (host pointer, nullable) receives the RELAY_FLAG_* mask.
 * Returns RELAY_ERR_DEVICE_CHECK if any flag was set.  Allocates nothing. */
relay_status_t relay_noalloc_device_status(uint32_t *flags_out, relay_stream_t stream);

/* Read and clear the device-side check flags of a workspace.  SYNCHRONOUS:
 * waits for `stream`.  *flags_out (host pointer, nullable) receives the
 * RELAY_FLAG_* mask.  Returns RELAY_ERR_DEVICE_CHECK if any flag was set. */
relay_status_t relay_device_status(void *ws, uint32_t *flags_out, relay_stream_t stream);

/* Static description of a status code. */
const char *relay_status_string(relay_status_t status);

#ifdef __cplusplus
}
#endif

#endif /* RELAY_H */
