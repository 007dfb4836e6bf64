// Device code of librelay: the persistent relay-attention kernel and the
// stand-alone fusion kernel, for sm_103a.
//
// One kernel, four modes:
//   MODE_FUSED     system items + context items, merged into fp16 out
//   MODE_SYS       system items only, merged into fp32 o_sys / lse_sys
//   MODE_CTX       context items only, merged into fp32 o_ctx / lse_ctx
//   MODE_BASELINE  context items over [system blocks; context] per request
//
// One CTA of 8 warps per SM works through two queues.
//
// Phase 1, row items.  The CTA's warps form two independent row teams of 4
// warps (each with half of the staging ring and its own named barrier); a
// team takes one item at a time:
//   system item  (KV head, key range, 64-row tile): 64 virtual rows of the
//                whole batch (query row x query head of the KV head's group)
//                against one range of system keys -- the matrix-matrix
//                product of the system-attention step (atyun.com RelayAttention
//                article, section "RelayAttention").  Each warp owns 16 rows;
//                when the rows fill fewer warps, the warps split each tile's
//                keys and combine their softmax states at the end.
//   multi-row context item (b, h, split, 64-row tile): the rows of one
//                request that carries several query tokens against a range of
//                its paged context, with the causal mask.
//   K/V tiles of 64 keys flow through a cp.async ring in XOR-swizzled shared
//   memory; S = Q K^T and O += P V run on mma.sync m16n8k16 (fp16 in, fp32
//   accumulate) with an online softmax in the log2 domain.  A team with no
//   row item left moves on to phase 2 at once.
//
// Phase 2, decode items (one warp per item, each warp independent):
//   (b, h, split): the one query row of a decode request against a range of
//   its paged context (the context-attention step).  A warp streams the
//   16-token pages of its items through a private cp.async ring, prefetching
//   the next item's pages while it finishes the current one.  Scores are
//   computed transposed, S^T = K q (keys on the MMA's M side), and the
//   output as O^T = V^T P, so a single query row wastes no MMA rows.
//
// Every item writes one fp32 partial result (normalised output and its
// log2-sum-exp) and moves on: no fence, no counter, no waiting.  A second,
// small kernel, launched as a programmatic dependent of the first, merges
// every row's partials: the relay fusion, generalised to any number of parts
// (system ranges and context splits), as a convex combination weighted by
// softmax mass.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace relay {

#ifndef RELAY_WARPS
#define RELAY_WARPS 8           // warps per CTA (one CTA per SM)
#endif
#ifndef RELAY_RING_KB
#define RELAY_RING_KB 192       // shared memory for K/V staging
#endif

constexpr int kBlock = 16;      // paged block size (tokens)
constexpr int kWarps = RELAY_WARPS;
constexpr int kThreads = kWarps * 32;
constexpr int kTileK = 64;      // keys per stage in phase 1
constexpr int kRowWarps = kWarps / 2;         // warps of a row team (phase-1 items); two teams per CTA
constexpr int kTeams = kWarps / kRowWarps;
constexpr int kRowThreads = kRowWarps * 32;
constexpr int kTileM = 16 * kRowWarps;        // query rows per phase-1 item
constexpr int kRingBytes = RELAY_RING_KB * 1024;
constexpr int kMaxB = 512;
constexpr int kMaxSegments = 8;   // shared prefix segments of one call

enum Mode : int { MODE_FUSED = 0, MODE_SYS = 1, MODE_CTX = 2, MODE_BASELINE = 3 };

enum : unsigned {
    FLAG_BAD_Q_LEN = 1u, FLAG_BAD_CTX_LEN = 2u, FLAG_BAD_BLOCK = 4u, FLAG_Q_TOTAL = 8u
};

// ctrl words in the workspace
enum { CTRL_FLAGS = 0, CTRL_ROW_ITEMS = 1, CTRL_DEC_ITEMS = 3, CTRL_TC_QUEUE = 4 /* and 5 */ };

struct Params {
    int B, Lq, H, Ls, num_blocks, max_blocks, max_q_total;
    int Hkv, G;                       // KV heads; query heads per KV head (query head h reads KV head h / G)
    int NG, HQ;                       // decode items per request and split: HQ = Hkv * NG head groups of up
                                      // to 8 query heads (NG = ceil(G / 8)) when G > 1, else HQ = H
    float scale_log2;                 // softmax scale * log2(e)
    const __half *q, *sys_k, *sys_v, *k_cache, *v_cache;
    const int *block_tables, *ctx_lens, *q_lens;
    const int *prefix_ids;            // baseline: system blocks in the pool
    int n_prefix;                     // baseline: system tokens ahead of each context
    __half *out;                      // fused / baseline output
    float *lse_out;                   // nullable
    float *o_f32, *lse_f32;           // sys-only / ctx-only outputs
    unsigned *ctrl;                   // see CTRL_*
    int *sched;                       // schedule handed to the merge kernel: [tps, qo[0..B], nctx[0..B-1]]
    float *part_o;                    // partial rows, D floats each (layout: see sys_slot)
    float *part_lse;                  // their log-sum-exps (log2 domain)
    int R_sys, sys_range, ctx_split;
    int tps_min, tps_max;             // pages per decode item: bounds of the adaptive choice
    int c_dec, c_mq;                  // context partial slots of a decode request / of a multi-row row
    int mq_split_min;                 // keys per split of a multi-row request: at least this
    long long dec_base, mq_base;      // first partial row of the decode and multi-row sections
    int skip_sys;                     // system partials come from the tensor-core kernel
    int skip_mq;                      // so do the multi-row requests' context partials (one split each)
    int dec_static;                   // static decode tickets per warp before the queue (0 or 3)
    int mode;
    // Shared prefix segments, each read once per batch: the system prompt
    // (one segment), or the levels of a tree of shared prefixes.  Request b
    // sees segment s when bit s of seg_mask[b] is set (seg_mask null: every
    // request sees every segment).  Segment s has seg_R[s] key ranges of
    // seg_range[s] keys, whose partials are system parts seg_part0[s] ...
    int n_seg;
    const __half *seg_k[kMaxSegments], *seg_v[kMaxSegments];
    int seg_len[kMaxSegments], seg_range[kMaxSegments], seg_R[kMaxSegments], seg_part0[kMaxSegments];
    const unsigned *seg_mask;
};

template <int D>
struct Smem {
    // row team t's ring is the t-th half of the staging memory, which holds
    // the decode rings of the team's own warps, so a team that moves on to
    // decode items never disturbs the other team's row item
    static constexpr int kStageC = kTileK * D * 2 * 2;        // bytes of one phase-1 stage (K + V)
    static constexpr int kRowRing = kRingBytes / kTeams;
    static constexpr int kStagesC = kRowRing / kStageC < 8 ? kRowRing / kStageC : 8;   // phase-1 ring depth
    static constexpr int kStageW = kBlock * D * 2 * 2;        // bytes of one page (K + V)
    static constexpr int kStagesW =
        kRingBytes / (kWarps * kStageW) < 6 ? kRingBytes / (kWarps * kStageW) : 6;   // per-warp ring depth
    alignas(128) unsigned char ring[kRingBytes];
    int qo[kMaxB + 1];        // exclusive prefix of query rows
    int mq[kMaxB + 1];        // exclusive prefix of multi-row context items
    int dec[kMaxB + 1];       // exclusive prefix of decode items over the decode order
    int nctx[kMaxB];          // context lengths (validated)
    unsigned segm[kMaxB];     // segments each request sees (bit s: segment s)
    short order[kMaxB];       // decode requests, longest item first
    signed char dcls[kMaxB];  // largest item of a decode request in pages (-1: not a decode request)
    int cls_cnt[33];
    int n_dec_req;
    int tps;                  // pages per decode item chosen for this launch
    int warp_tot[kWarps];
    int item[kTeams];
    int bad;

    __device__ __half *ck(int team, int st) { return reinterpret_cast<__half *>(ring + team * kRowRing + st * kStageC); }
    __device__ __half *cv(int team, int st) { return ck(team, st) + kTileK * D; }
    __device__ __half *wk(int w, int st) { return reinterpret_cast<__half *>(ring + (w * kStagesW + st) * kStageW); }
    __device__ __half *wv(int w, int st) { return wk(w, st) + kBlock * D; }
};

// ----------------------------------------------------------------------------- PTX helpers
__device__ __forceinline__ unsigned smem_u32(const void *p)
{
    return static_cast<unsigned>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void cp_async16(void *dst, const void *src, bool valid)
{
    int n = valid ? 16 : 0;   // n == 0: zero-fill, nothing read
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(smem_u32(dst)), "l"(src), "r"(n));
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;\n" ::); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;\n" ::"n"(N)); }

// wait until at most n groups are pending (n < 8)
__device__ __forceinline__ void cp_async_wait_dyn(int n)
{
    switch (n) {
    case 0: cp_async_wait<0>(); break;
    case 1: cp_async_wait<1>(); break;
    case 2: cp_async_wait<2>(); break;
    case 3: cp_async_wait<3>(); break;
    case 4: cp_async_wait<4>(); break;
    case 5: cp_async_wait<5>(); break;
    case 6: cp_async_wait<6>(); break;
    default: cp_async_wait<7>(); break;
    }
}

__device__ __forceinline__ void ldsm_x4(unsigned &r0, unsigned &r1, unsigned &r2, unsigned &r3, const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(p)));
}
__device__ __forceinline__ void ldsm_x4_t(unsigned &r0, unsigned &r1, unsigned &r2, unsigned &r3, const void *p)
{
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(smem_u32(p)));
}

// D(16x8 f32) += A(16x16 f16, row) * B(16x8 f16, col)
__device__ __forceinline__ void mma16816(float c[4], const unsigned a[4], unsigned b0, unsigned b1)
{
    asm volatile("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
                 "{%0,%1,%2,%3}, {%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
                 : "+f"(c[0]), "+f"(c[1]), "+f"(c[2]), "+f"(c[3])
                 : "r"(a[0]), "r"(a[1]), "r"(a[2]), "r"(a[3]), "r"(b0), "r"(b1));
}

__device__ __forceinline__ float ex2(float x)
{
    float y;
    asm("ex2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}
__device__ __forceinline__ float lg2(float x)
{
    float y;
    asm("lg2.approx.ftz.f32 %0, %1;\n" : "=f"(y) : "f"(x));
    return y;
}

__device__ __forceinline__ unsigned pack_half2(float lo, float hi)
{
    __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<unsigned *>(&h);
}

__device__ __forceinline__ unsigned ld_u32(const __half *p)
{
    return *reinterpret_cast<const unsigned *>(p);
}

#define kNegInf (-__int_as_float(0x7f800000))

// index of this thread's row team, and the team's barrier (named barrier
// 1 + team over the team's kRowThreads threads; the other team goes on)
__device__ __forceinline__ int team_of() { return (threadIdx.x >> 5) / kRowWarps; }
__device__ __forceinline__ void team_sync()
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(1 + team_of()), "n"(kRowThreads) : "memory");
}

// swizzled element offset of (row, 16-byte chunk) in a [rows][D] fp16 tile
template <int D>
__device__ __forceinline__ int swz(int row, int ch)
{
    return row * D + ((ch ^ (row & 7)) << 3);
}

// Largest b in [0, n) with a[b] <= x (a nondecreasing, a[0] <= x < a[n]).
__device__ __forceinline__ int find_owner(const int *a, int n, int x)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (a[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// ----------------------------------------------------------------------------- schedule
__device__ __forceinline__ bool has_sys(int mode) { return mode == MODE_FUSED || mode == MODE_SYS; }
__device__ __forceinline__ bool has_ctx(int mode) { return mode != MODE_SYS; }

// Context work of one request.
//   decode request (one query row): its key sequence is cut into pages --
//     ceil(n_prefix/16) prefix pages then ceil(n_ctx/16) context pages -- and
//     the pages into ns nearly equal splits of at most ctx_split/16 pages
//     (one warp item each; split j covers pages [j*pages/ns, (j+1)*pages/ns));
//   multi-row request: keys [0, n_prefix + n_ctx) in splits of `split` keys,
//     rows in tiles of kTileM (one CTA item per split and row tile).
struct ReqInfo {
    int ql, n_ctx;
    int pp;        // prefix pages (decode)
    int pages;     // total pages (decode)
    int tps;       // most pages per split (decode)
    int split;     // keys per split (multi-row)
    int ns;        // splits
    int mt;        // row tiles (multi-row), 1 for decode
};

__device__ __forceinline__ ReqInfo req_info(const Params &p, int n_ctx, int ql, int tps)
{
    ReqInfo r;
    r.ql = ql;
    r.n_ctx = n_ctx;
    r.pp = (p.n_prefix + kBlock - 1) / kBlock;
    r.pages = r.pp + (r.n_ctx + kBlock - 1) / kBlock;
    r.tps = tps;                 // at most 32: a decode item holds one page per lane
    if (ql <= 1) {
        r.split = p.ctx_split;
        r.ns = (r.pages + r.tps - 1) / r.tps;
        r.mt = 1;
    } else {
        // longer splits for multi-row requests keep the partial traffic small
        // next to the keys each item streams
        int want = ql * 64;
        r.split = max(((want + p.ctx_split - 1) / p.ctx_split) * p.ctx_split, p.mq_split_min);
        int nkeys = p.n_prefix + r.n_ctx;
        r.ns = (nkeys + r.split - 1) / r.split;
        r.mt = (ql + kTileM - 1) / kTileM;
    }
    if (r.ns < 1) r.ns = 1;
    return r;
}

// Inclusive prefix sum over the 32 lanes of a warp.
__device__ __forceinline__ int warp_incl_scan(int v)
{
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        const int t = __shfl_up_sync(0xffffffffu, v, off);
        if (lane >= off) v += t;
    }
    return v;
}

// Exclusive prefix sum over the batch of per-request values v[k] (request
// tid*PER + k), written to out[0..n] (out[n] = total).
template <int D, int PER>
__device__ __forceinline__ void block_scan(const int (&v)[PER], int *out, int n, Smem<D> &s)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int loc = 0;
#pragma unroll
    for (int k = 0; k < PER; k++) loc += v[k];
    int inc = loc;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int t = __shfl_up_sync(0xffffffffu, inc, off);
        if (lane >= off) inc += t;
    }
    if (lane == 31) s.warp_tot[warp] = inc;
    __syncthreads();
    int base = inc - loc;
    for (int j = 0; j < warp; j++) base += s.warp_tot[j];
#pragma unroll
    for (int k = 0; k < PER; k++) {
        int b = tid * PER + k;
        if (b < n) out[b] = base;
        base += v[k];
    }
    if (tid == kThreads - 1) out[n] = base;
    __syncthreads();
}

// The schedule of build_schedule (below) built by the whole CTA, PER
// requests per thread with block scans: for batches of more than 32
// requests, where one warp would need several dependent rounds.  Kept out of
// line: the kernel starts with its code cold (nothing of it in L2 after the
// other kernels of a model step), and this path inlined beside the one-warp
// build cost the 32-request step 2.5 us (measured).
template <int D>
__device__ __noinline__ void build_schedule_cta(const Params &p, Smem<D> &s)
{
    constexpr int PER = (kMaxB + kThreads - 1) / kThreads;
    constexpr int kClasses = 33;                  // item sizes 0..32 pages
    constexpr int kItemsPerWarp = 4;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int vq[PER], vm[PER], vp[PER], nn[PER];
    unsigned flags = 0;
    if (tid < kClasses) s.cls_cnt[tid] = 0;
    if (tid == 0) s.bad = 0;
    const int pp = (p.n_prefix + kBlock - 1) / kBlock;
#pragma unroll
    for (int k = 0; k < PER; k++) {
        const int b = tid * PER + k;
        int ql = 0, n = 0, m = 0, pg = 0;
        if (b < p.B) {
            ql = p.q_lens ? p.q_lens[b] : p.Lq;
            n = (has_ctx(p.mode) && p.ctx_lens) ? p.ctx_lens[b] : 0;
            s.segm[b] = p.seg_mask ? p.seg_mask[b] : ~0u;
            if (ql < 0 || ql > p.Lq) { flags |= FLAG_BAD_Q_LEN; ql = 0; }
            if (n < 0 || n > p.max_blocks * kBlock) { flags |= FLAG_BAD_CTX_LEN; ql = 0; n = 0; }
            if (has_ctx(p.mode) && ql > 1) {
                const ReqInfo r = req_info(p, n, ql, p.tps_max);
                m = p.H * r.ns * r.mt;
            }
            if (has_ctx(p.mode) && ql == 1) pg = p.HQ * (pp + (n + kBlock - 1) / kBlock);
        }
        vq[k] = ql;
        vm[k] = m;
        vp[k] = pg;
        nn[k] = n;
    }
    __syncthreads();
    if (flags) atomicOr(&s.bad, (int)flags);
    block_scan<D, PER>(vq, s.qo, p.B, s);
    block_scan<D, PER>(vm, s.mq, p.B, s);
    block_scan<D, PER>(vp, s.dec, p.B, s);        // s.dec[B]: decode pages over all heads
    if (tid == 0) {
        const long long want = (long long)gridDim.x * kWarps * kItemsPerWarp;
        int t = (int)((s.dec[p.B] + want - 1) / want);
        s.tps = max(p.tps_min, min(p.tps_max, t));
    }
    __syncthreads();
    const int tps = s.tps;
    // decode class of every request: its largest item in pages (-1: not decode)
#pragma unroll
    for (int k = 0; k < PER; k++) {
        const int b = tid * PER + k;
        if (b < p.B) {
            s.nctx[b] = nn[k];
            int c = -1;
            if (has_ctx(p.mode) && vq[k] == 1) {
                const ReqInfo r = req_info(p, nn[k], 1, tps);
                c = (r.pages + r.ns - 1) / r.ns;
                atomicAdd(&s.cls_cnt[c], 1);
            }
            s.dcls[b] = (signed char)c;
        }
    }
    __syncthreads();
    // counting sort of decode requests: class descending, request index ascending
    if (warp == 0) {
        // start position of classes 32..1 (lanes 0..31), then class 0
        const int v = kClasses - 1 - lane;
        const int cnt = s.cls_cnt[v];
        int inc = cnt;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int t = __shfl_up_sync(0xffffffffu, inc, off);
            if (lane >= off) inc += t;
        }
        const int c0 = s.cls_cnt[0];
        __syncwarp();
        s.cls_cnt[v] = inc - cnt;
        if (lane == 31) {
            s.cls_cnt[0] = inc;
            s.n_dec_req = inc + c0;
        }
        __syncwarp();
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            const int c = b < p.B ? s.dcls[b] : -1;
            const unsigned same = __match_any_sync(0xffffffffu, c);
            const int base = c >= 0 ? s.cls_cnt[c] : 0;
            if (c >= 0) s.order[base + __popc(same & ((1u << lane) - 1u))] = (short)b;
            __syncwarp();
            if (c >= 0 && lane == __ffs(same) - 1) s.cls_cnt[c] = base + __popc(same);
            __syncwarp();
        }
    }
    __syncthreads();
    // decode items per sorted position
    int dv[PER];
#pragma unroll
    for (int k = 0; k < PER; k++) {
        const int pos = tid * PER + k;
        dv[k] = 0;
        if (pos < s.n_dec_req) dv[k] = p.HQ * req_info(p, s.nctx[s.order[pos]], 1, tps).ns;
    }
    block_scan<D, PER>(dv, s.dec, s.n_dec_req, s);
    if (tid == 0 && s.qo[p.B] > p.max_q_total) s.bad |= FLAG_Q_TOTAL;
    __syncthreads();
}

// Per-CTA schedule over the batch (B <= kMaxB): row prefix qo, multi-row
// item prefix mq, and the decode queue.  Up to 32 requests it is built by
// warp 0 alone with warp shuffles (no block-wide barrier until the end);
// larger batches use the block-wide build above.
//   * Pages per decode item: between tps_min and tps_max, chosen so that the
//     decode queue holds about kItemsPerWarp items per warp of the grid (fine
//     enough for the dynamic queue to balance, coarse enough to keep the
//     per-item cost small).
//   * Decode requests are ordered longest item first (their largest split in
//     pages, descending; ties by request index), so the queue ends with the
//     shortest items and the warps finish together.
// Every CTA computes the same schedule from the same inputs.
template <int D>
__device__ void build_schedule(const Params &p, Smem<D> &s)
{
    constexpr int kClasses = 33;                  // item sizes 0..32 pages
    constexpr int kItemsPerWarp = 4;
    const int lane = threadIdx.x & 31;
    if (p.B > 32) {
        build_schedule_cta<D>(p, s);
        return;
    }
    if ((threadIdx.x >> 5) == 0) {
        const int pp = (p.n_prefix + kBlock - 1) / kBlock;
        unsigned flags = 0;
        int run_q = 0, run_m = 0, pages = 0;
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            int ql = 0, n = 0, m = 0, pg = 0;
            if (b < p.B) {
                ql = p.q_lens ? p.q_lens[b] : p.Lq;
                n = (has_ctx(p.mode) && p.ctx_lens) ? p.ctx_lens[b] : 0;
                s.segm[b] = p.seg_mask ? p.seg_mask[b] : ~0u;
                if (ql < 0 || ql > p.Lq) { flags |= FLAG_BAD_Q_LEN; ql = 0; }
                if (n < 0 || n > p.max_blocks * kBlock) { flags |= FLAG_BAD_CTX_LEN; ql = 0; n = 0; }
                if (has_ctx(p.mode) && ql > 1) {
                    const ReqInfo r = req_info(p, n, ql, p.tps_max);
                    m = p.H * r.ns * r.mt;
                }
                if (has_ctx(p.mode) && ql == 1) pg = p.HQ * (pp + (n + kBlock - 1) / kBlock);
                s.nctx[b] = n;
                s.dcls[b] = (signed char)(has_ctx(p.mode) && ql == 1 ? 0 : -1);   // decode request (class below)
            }
            const int iq = warp_incl_scan(ql), im = warp_incl_scan(m);
            if (b < p.B) {
                s.qo[b] = run_q + iq - ql;
                s.mq[b] = run_m + im - m;
            }
            run_q += __shfl_sync(0xffffffffu, iq, 31);
            run_m += __shfl_sync(0xffffffffu, im, 31);
            pages += __reduce_add_sync(0xffffffffu, pg);
        }
        flags = __reduce_or_sync(0xffffffffu, flags);
        if (run_q > p.max_q_total) flags |= FLAG_Q_TOTAL;
        const long long want = (long long)gridDim.x * kWarps * kItemsPerWarp;
        const int tps = max(p.tps_min, min(p.tps_max, (int)((pages + want - 1) / want)));
        if (lane == 0) {
            s.qo[p.B] = run_q;
            s.mq[p.B] = run_m;
            s.tps = tps;
            s.bad = (int)flags;
        }
        // decode class of every request (its largest item in pages), counted per class
        s.cls_cnt[lane] = 0;
        if (lane == 0) s.cls_cnt[32] = 0;
        __syncwarp();
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            int c = -1;
            if (b < p.B && s.dcls[b] == 0) {
                const ReqInfo r = req_info(p, s.nctx[b], 1, tps);
                c = (r.pages + r.ns - 1) / r.ns;
                s.dcls[b] = (signed char)c;
            }
            const unsigned same = __match_any_sync(0xffffffffu, c);
            if (c >= 0 && lane == __ffs(same) - 1) s.cls_cnt[c] += __popc(same);
            __syncwarp();
        }
        // counting sort of decode requests: class descending, request index ascending.
        // Start position of classes 32..1 (lanes 0..31), then class 0.
        {
            const int v = kClasses - 1 - lane;
            const int cnt = s.cls_cnt[v];
            const int inc = warp_incl_scan(cnt);
            const int c0 = s.cls_cnt[0];
            __syncwarp();
            s.cls_cnt[v] = inc - cnt;
            if (lane == 31) {
                s.cls_cnt[0] = inc;
                s.n_dec_req = inc + c0;
            }
            __syncwarp();
        }
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            const int c = b < p.B ? s.dcls[b] : -1;
            const unsigned same = __match_any_sync(0xffffffffu, c);
            const int base = c >= 0 ? s.cls_cnt[c] : 0;
            if (c >= 0) s.order[base + __popc(same & ((1u << lane) - 1u))] = (short)b;
            __syncwarp();
            if (c >= 0 && lane == __ffs(same) - 1) s.cls_cnt[c] = base + __popc(same);
            __syncwarp();
        }
        // decode items per sorted position: exclusive prefix into s.dec
        const int n_dec_req = s.n_dec_req;
        int run_d = 0;
        for (int q0 = 0; q0 < n_dec_req; q0 += 32) {
            const int pos = q0 + lane;
            const int dv = pos < n_dec_req ? p.HQ * req_info(p, s.nctx[s.order[pos]], 1, tps).ns : 0;
            const int id = warp_incl_scan(dv);
            if (pos < n_dec_req) s.dec[pos] = run_d + id - dv;
            run_d += __shfl_sync(0xffffffffu, id, 31);
        }
        if (lane == 0) s.dec[n_dec_req] = run_d;
    }
    __syncthreads();
}

// ----------------------------------------------------------------------------- merge (relay fusion)
// Partial rows in the workspace (index into part_lse, and in units of D
// floats into part_o):
//   system part k (key range) of compact row r, head h:  (k * max_q_total + r) * H + h
//   context part k of the decode request b (one row):     dec_base + (k * B + b) * H + h
//   context part k of compact row r of a multi-row request:  mq_base + (k * max_q_total + r) * H + h
// so a decode row reserves context slots once per request, not once per row
// of the max_q_total bound.
__device__ __forceinline__ size_t sys_slot(const Params &p, int k, int r, int h)
{
    return ((size_t)k * p.max_q_total + r) * p.H + h;
}
__device__ __forceinline__ size_t dec_slot(const Params &p, int k, int b, int h)
{
    return (size_t)p.dec_base + ((size_t)k * p.B + b) * p.H + h;
}
__device__ __forceinline__ size_t mq_slot(const Params &p, int k, int r, int h)
{
    return (size_t)p.mq_base + ((size_t)k * p.max_q_total + r) * p.H + h;
}
// part j of a row: the n_sys system ranges first, then the context splits
__device__ __forceinline__ size_t part_slot(const Params &p, int j, int n_sys, bool dec, int r, int b, int h)
{
    return j < n_sys ? sys_slot(p, j, r, h) : dec ? dec_slot(p, j - n_sys, b, h) : mq_slot(p, j - n_sys, r, h);
}

// Merge the partials of one output row (compact row r = row i of request b,
// head h) into the output: the convex combination of the parts weighted by
// their softmax mass.  One warp; lane k loads the log-sum-exp of part k and
// every lane the first CH parts' output rows, all in one round trip; further
// parts follow CH at a time with all CH loads in flight together.  Lane t
// handles D/32 adjacent elements.
template <int D, int CH = 16>   // CH: partial rows in flight per lane (one round for up to CH partials)
__device__ void merge_row(const Params &p, int r, int b, int i, int h, int n_sys, int n_ctx, bool dec,
                          bool have_lk0 = false, float lk0 = 0.f)
{
    constexpr int V = D / 32;
    constexpr float kLn2 = 0.69314718055994531f;
    const int lane = threadIdx.x & 31;
    const int n = n_sys + n_ctx;
    const int d0 = lane * V;
    // part j's slot: first + j * stride within its section (system parts,
    // then context parts)
    const size_t sys0 = sys_slot(p, 0, r, h), ctx0 = dec ? dec_slot(p, 0, b, h) : mq_slot(p, 0, r, h);
    const size_t sys_st = (size_t)p.max_q_total * p.H, ctx_st = dec ? (size_t)p.B * p.H : sys_st;
    auto slot = [&](int j) { return j < n_sys ? sys0 + (size_t)j * sys_st : ctx0 + (size_t)(j - n_sys) * ctx_st; };
    float M = kNegInf, W = 0.f, acc[V];
#pragma unroll
    for (int v = 0; v < V; v++) acc[v] = 0.f;
    // CH partial rows of parts j0 + c0 .. into x (zeros past cnt)
    auto load_parts = [&](float (&x)[CH][V], int j0, int c0, int cnt) {
#pragma unroll
        for (int k = 0; k < CH; k++) {
            if (c0 + k < cnt) {
                const float *src = p.part_o + slot(j0 + c0 + k) * D + d0;
                if constexpr (V == 4) {
                    const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
                    x[k][0] = t.x; x[k][1] = t.y; x[k][2] = t.z; x[k][3] = t.w;
                } else {
                    const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
                    x[k][0] = t.x; x[k][1] = t.y;
                }
            } else {
#pragma unroll
                for (int v = 0; v < V; v++) x[k][v] = 0.f;
            }
        }
    };
    for (int j0 = 0; j0 < n; j0 += 32) {
        const int cnt = min(32, n - j0);
        // the first CH partial rows of the chunk are requested together with
        // its log-sum-exps (the rows do not depend on them, only their
        // weights do): one round trip for a row of at most CH parts
        float x[CH][V];
        load_parts(x, j0, 0, cnt);
        float lk = kNegInf;      // lane k: log-sum-exp of part j0 + k
        if (j0 == 0 && have_lk0) {
            lk = lane < cnt ? lk0 : kNegInf;
        } else if (lane < cnt) {
            lk = __ldcg(p.part_lse + slot(j0 + lane));
        }
        float mk = lk;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) mk = fmaxf(mk, __shfl_xor_sync(0xffffffffu, mk, off));
        if (mk == kNegInf) continue;
        const float Mn = fmaxf(M, mk);
        const float sc = ex2(M - Mn);          // rescale what was merged so far
        W *= sc;
#pragma unroll
        for (int v = 0; v < V; v++) acc[v] *= sc;
        M = Mn;
        const float wk = ex2(lk - M);
        for (int c0 = 0; c0 < cnt; c0 += CH) {
            if (c0 > 0) load_parts(x, j0, c0, cnt);
#pragma unroll
            for (int k = 0; k < CH; k++) {
                const float w = __shfl_sync(0xffffffffu, wk, (c0 + k) & 31);
                if (c0 + k < cnt) {
                    W += w;
#pragma unroll
                    for (int v = 0; v < V; v++) acc[v] += w * x[k][v];
                }
            }
        }
    }
    const float inv = W > 0.f ? 1.f / W : 0.f;
    const float lse = W > 0.f ? (M + lg2(W)) * kLn2 : kNegInf;
    const size_t orow = ((size_t)b * p.Lq + i) * p.H + h;
    if (p.mode == MODE_FUSED || p.mode == MODE_BASELINE) {
        __half *dst = p.out + orow * D + d0;
        if constexpr (V == 4) {
            *reinterpret_cast<uint2 *>(dst) =
                make_uint2(pack_half2(acc[0] * inv, acc[1] * inv), pack_half2(acc[2] * inv, acc[3] * inv));
        } else {
            *reinterpret_cast<unsigned *>(dst) = pack_half2(acc[0] * inv, acc[1] * inv);
        }
        if (p.lse_out && lane == 0) p.lse_out[orow] = lse;
    } else {
        float *dst = p.o_f32 + orow * D + d0;
#pragma unroll
        for (int v = 0; v < V; v++) dst[v] = acc[v] * inv;
        if (lane == 0) p.lse_f32[orow] = lse;
    }
}

// ============================================================================= phase 1: row items
struct KeySrc {
    const __half *k, *v;
    const int *table;       // this request's block table row (paged) or nullptr (system cache)
    const int *prefix;      // baseline: system blocks
    int n_prefix;
    int H, h, num_blocks;   // KV heads of the cache and the KV head read
};

// Element offset of key t's row; false (and a flag) for an out-of-range block.
__device__ __forceinline__ bool key_offset(const KeySrc &s, int t, size_t &off, unsigned *flags, int D)
{
    if (s.table == nullptr) {
        off = ((size_t)t * s.H + s.h) * D;
        return true;
    }
    int blk, slot;
    if (t < s.n_prefix) {
        blk = s.prefix[t / kBlock];
        slot = t % kBlock;
    } else {
        int u = t - s.n_prefix;
        blk = s.table[u / kBlock];
        slot = u % kBlock;
    }
    if (blk < 0 || blk >= s.num_blocks) {
        atomicOr(flags, FLAG_BAD_BLOCK);
        return false;
    }
    off = (((size_t)blk * s.H + s.h) * kBlock + slot) * D;
    return true;
}

// Stage keys [key0, key0 + kTileK) of K and V into ring slot `st`; keys at or
// beyond key_end are zero-filled (never read from memory).
template <int D>
__device__ __forceinline__ void load_tile(Smem<D> &s, int st, const KeySrc &src, int key0, int key_end,
                                          unsigned *flags)
{
    constexpr int CPR = D / 8;                      // 16-byte chunks per row
    constexpr int PER = kTileK * CPR / kRowThreads; // chunks per team thread
    const int tid = threadIdx.x % kRowThreads;
    __half *K = s.ck(team_of(), st), *V = s.cv(team_of(), st);
#pragma unroll
    for (int k = 0; k < PER; k++) {
        int c = tid + k * kRowThreads;
        int key = c / CPR, ch = c % CPR;
        int t = key0 + key;
        size_t off = 0;
        bool valid = t < key_end;
        if (valid) valid = key_offset(src, t, off, flags, D);
        int dst = swz<D>(key, ch);
        cp_async16(K + dst, valid ? src.k + off + ch * 8 : src.k, valid);
        cp_async16(V + dst, valid ? src.v + off + ch * 8 : src.v, valid);
    }
}

template <int D>
struct RowState {
    float o[D / 8][4];
    float m[2], l[2];
};

// One warp: 16 query rows (A fragments in qf) against keys [kb, kb + 8*NT)
// of a staged tile.  Lane state: rows g and g+8.
template <int D, int NT>
__device__ __forceinline__ void row_tile(const __half *K, const __half *V, int kb, const unsigned (&qf)[D / 16][4],
                                         RowState<D> &ws, int key_tile0, int end0, int end1, float scale_log2)
{
    static_assert(NT % 2 == 0 || NT == 1, "key sub-range of 8, 16, 32 or 64 keys");
    const int lane = threadIdx.x & 31;
    float sc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; n++)
#pragma unroll
        for (int e = 0; e < 4; e++) sc[n][e] = 0.f;

    if constexpr (NT == 1) {
#pragma unroll
        for (int kp = 0; kp < D / 32; kp++) {
            // four 8x8 blocks: keys kb..kb+7, d-chunks 4kp .. 4kp+3
            int row = kb + (lane & 7);
            int ch = 4 * kp + (lane >> 3);
            unsigned b0, b1, b2, b3;
            ldsm_x4(b0, b1, b2, b3, K + swz<D>(row, ch));
            mma16816(sc[0], qf[2 * kp], b0, b1);
            mma16816(sc[0], qf[2 * kp + 1], b2, b3);
        }
    } else {
#pragma unroll
        for (int kt = 0; kt < D / 16; kt++) {
#pragma unroll
            for (int np = 0; np < NT / 2; np++) {
                int row = kb + np * 16 + (lane & 7) + ((lane >> 4) << 3);
                int ch = 2 * kt + ((lane >> 3) & 1);
                unsigned b0, b1, b2, b3;
                ldsm_x4(b0, b1, b2, b3, K + swz<D>(row, ch));
                mma16816(sc[2 * np], qf[kt], b0, b1);
                mma16816(sc[2 * np + 1], qf[kt], b2, b3);
            }
        }
    }

    const int tig = lane & 3;
    float mx0 = kNegInf, mx1 = kNegInf;
#pragma unroll
    for (int n = 0; n < NT; n++) {
#pragma unroll
        for (int e = 0; e < 4; e++) {
            int key = key_tile0 + kb + n * 8 + 2 * tig + (e & 1);
            int end = (e < 2) ? end0 : end1;
            float v = sc[n][e] * scale_log2;
            sc[n][e] = (key < end) ? v : kNegInf;
        }
        mx0 = fmaxf(mx0, fmaxf(sc[n][0], sc[n][1]));
        mx1 = fmaxf(mx1, fmaxf(sc[n][2], sc[n][3]));
    }
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 1));
    mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, 2));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 1));
    mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, 2));
    float mn0 = fmaxf(ws.m[0], mx0), mn1 = fmaxf(ws.m[1], mx1);
    float mu0 = (mn0 == kNegInf) ? 0.f : mn0;
    float mu1 = (mn1 == kNegInf) ? 0.f : mn1;
    float al0 = ex2(ws.m[0] - mu0), al1 = ex2(ws.m[1] - mu1);
    ws.m[0] = mn0;
    ws.m[1] = mn1;
    float rs0 = 0.f, rs1 = 0.f;
#pragma unroll
    for (int n = 0; n < NT; n++) {
        sc[n][0] = ex2(sc[n][0] - mu0);
        sc[n][1] = ex2(sc[n][1] - mu0);
        sc[n][2] = ex2(sc[n][2] - mu1);
        sc[n][3] = ex2(sc[n][3] - mu1);
        rs0 += sc[n][0] + sc[n][1];
        rs1 += sc[n][2] + sc[n][3];
    }
    ws.l[0] = ws.l[0] * al0 + rs0;
    ws.l[1] = ws.l[1] * al1 + rs1;
#pragma unroll
    for (int d = 0; d < D / 8; d++) {
        ws.o[d][0] *= al0; ws.o[d][1] *= al0;
        ws.o[d][2] *= al1; ws.o[d][3] *= al1;
    }

    if constexpr (NT == 1) {
        // one k-step of 16 keys whose upper 8 weights are zero; the V rows
        // of those 8 keys are read (they lie inside the staged tile) but
        // multiplied by zero, and they are finite (zero-filled or real data)
        unsigned pa[4];
        pa[0] = pack_half2(sc[0][0], sc[0][1]);
        pa[1] = pack_half2(sc[0][2], sc[0][3]);
        pa[2] = 0u;
        pa[3] = 0u;
        const int kb16 = kb & ~15;
        const int hi = kb & 8;     // our 8 keys are rows kb16+hi .. +7 of the 16-key step
        if (hi) {                  // move our weights to the upper half of the step
            pa[2] = pa[0]; pa[3] = pa[1]; pa[0] = 0u; pa[1] = 0u;
        }
#pragma unroll
        for (int dp = 0; dp < D / 16; dp++) {
            int row = kb16 + (lane & 7) + (((lane >> 3) & 1) << 3);
            int ch = 2 * dp + (lane >> 4);
            unsigned b0, b1, b2, b3;
            ldsm_x4_t(b0, b1, b2, b3, V + swz<D>(row, ch));
            mma16816(ws.o[2 * dp], pa, b0, b1);
            mma16816(ws.o[2 * dp + 1], pa, b2, b3);
        }
    } else {
#pragma unroll
        for (int ks = 0; ks < NT / 2; ks++) {
            unsigned pa[4];
            pa[0] = pack_half2(sc[2 * ks][0], sc[2 * ks][1]);
            pa[1] = pack_half2(sc[2 * ks][2], sc[2 * ks][3]);
            pa[2] = pack_half2(sc[2 * ks + 1][0], sc[2 * ks + 1][1]);
            pa[3] = pack_half2(sc[2 * ks + 1][2], sc[2 * ks + 1][3]);
#pragma unroll
            for (int dp = 0; dp < D / 16; dp++) {
                int row = kb + ks * 16 + (lane & 7) + (((lane >> 3) & 1) << 3);
                int ch = 2 * dp + (lane >> 4);
                unsigned b0, b1, b2, b3;
                ldsm_x4_t(b0, b1, b2, b3, V + swz<D>(row, ch));
                mma16816(ws.o[2 * dp], pa, b0, b1);
                mma16816(ws.o[2 * dp + 1], pa, b2, b3);
            }
        }
    }
}

// Key-tile pipeline of a row item over [key0, key_hi): each warp owns 16 rows
// and keys [kb, kb + 8*NT) of every tile.  Warps without valid rows only help
// load.
template <int D, int NT>
__device__ __forceinline__ void row_pipeline(Smem<D> &s, const KeySrc &src, int key0, int key_hi, int kb,
                                             const unsigned (&qf)[D / 16][4], RowState<D> &ws, int end0,
                                             int end1, bool active, float scale_log2, unsigned *flags)
{
    constexpr int S = Smem<D>::kStagesC;
    const int n_tiles = (key_hi > key0) ? (key_hi - key0 + kTileK - 1) / kTileK : 0;
    for (int j = 0; j < n_tiles; j++) {
        cp_async_wait<S - 2>();
        team_sync();
        int jn = j + S - 1;
        if (jn < n_tiles) load_tile<D>(s, jn % S, src, key0 + jn * kTileK, key_hi, flags);
        cp_async_commit();
        if (active)
            row_tile<D, NT>(s.ck(team_of(), j % S), s.cv(team_of(), j % S), kb, qf, ws, key0 + j * kTileK, end0, end1,
                            scale_log2);
    }
    cp_async_wait<0>();
    team_sync();
}

template <int D>
__device__ __forceinline__ void row_prologue(Smem<D> &s, const KeySrc &src, int key0, int key_hi, unsigned *flags)
{
    constexpr int S = Smem<D>::kStagesC;
    const int n_tiles = (key_hi > key0) ? (key_hi - key0 + kTileK - 1) / kTileK : 0;
#pragma unroll
    for (int j = 0; j < S - 1; j++) {
        if (j < n_tiles) load_tile<D>(s, j, src, key0 + j * kTileK, key_hi, flags);
        cp_async_commit();
    }
}

template <int D>
__device__ __forceinline__ void load_q_rows(unsigned (&qf)[D / 16][4], const __half *qa, const __half *qb)
{
    const int tig = threadIdx.x & 3;
#pragma unroll
    for (int kt = 0; kt < D / 16; kt++) {
        int c = kt * 16 + 2 * tig;
        qf[kt][0] = qa ? ld_u32(qa + c) : 0u;
        qf[kt][1] = qb ? ld_u32(qb + c) : 0u;
        qf[kt][2] = qa ? ld_u32(qa + c + 8) : 0u;
        qf[kt][3] = qb ? ld_u32(qb + c + 8) : 0u;
    }
}

// Write one warp's partial rows (normalised output, log2-sum-exp).
// (system part k when !mq, else context part k of a multi-row request)
template <int D>
__device__ __forceinline__ void write_row_partials(const Params &p, const RowState<D> &ws, bool mq, int k, int hA,
                                                   int rA, bool vA, int hB, int rB, bool vB)
{
    const int tig = threadIdx.x & 3;
    float l0 = ws.l[0], l1 = ws.l[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
#pragma unroll
    for (int half = 0; half < 2; half++) {
        if (!(half ? vB : vA)) continue;
        float l = half ? l1 : l0, m = ws.m[half];
        float inv = l > 0.f ? 1.f / l : 0.f;
        const int r = half ? rB : rA, h = half ? hB : hA;
        const size_t pr = mq ? mq_slot(p, k, r, h) : sys_slot(p, k, r, h);
        float *po = p.part_o + pr * D;
#pragma unroll
        for (int n = 0; n < D / 8; n++)
            __stcg(reinterpret_cast<float2 *>(po + n * 8 + 2 * tig),
                   make_float2(ws.o[n][2 * half] * inv, ws.o[n][2 * half + 1] * inv));
        if (tig == 0) __stcg(p.part_lse + pr, l > 0.f ? m + lg2(l) : kNegInf);
    }
}

// Warp roles of a row item with `rows` valid rows: RG groups of 16 rows, and
// when the rows fill fewer than all warps, KG groups that split each tile's
// 64 keys (their softmax states are combined at the end of the item).
struct RowRoles {
    int KG, RGp, rg, kg;
    bool active;
};

__device__ __forceinline__ RowRoles row_roles(int rows)
{
    RowRoles r;
    const int RG = (rows + 15) / 16;
    int np2 = 1;
    while (np2 < RG) np2 <<= 1;
    r.KG = min(kRowWarps / np2, kTileK / 8);
    r.RGp = kRowWarps / r.KG;
    const int warp = (threadIdx.x >> 5) % kRowWarps;
    r.rg = warp % r.RGp;
    r.kg = warp / r.RGp;
    r.active = r.rg < RG && r.kg < r.KG;
    return r;
}

// KGF: 0 = any key-group count (chosen per item); else the only count this
// kernel instance meets (the host knows it), so that only that pipeline is
// compiled in.
template <int D, int KGF>
__device__ __forceinline__ void run_rows(Smem<D> &s, const KeySrc &src, int key0, int key_hi, const RowRoles &rr,
                                         const unsigned (&qf)[D / 16][4], RowState<D> &ws, int end0, int end1,
                                         float scale_log2, unsigned *flags)
{
    const int kpk = kTileK / rr.KG;          // keys per key group
    const int kb = rr.kg * kpk;
    if constexpr (KGF > 0) {
        row_pipeline<D, 8 / KGF>(s, src, key0, key_hi, kb, qf, ws, end0, end1, rr.active, scale_log2, flags);
    } else {
        switch (rr.KG) {
        case 1: row_pipeline<D, 8>(s, src, key0, key_hi, kb, qf, ws, end0, end1, rr.active, scale_log2, flags); break;
        case 2: row_pipeline<D, 4>(s, src, key0, key_hi, kb, qf, ws, end0, end1, rr.active, scale_log2, flags); break;
        case 4: row_pipeline<D, 2>(s, src, key0, key_hi, kb, qf, ws, end0, end1, rr.active, scale_log2, flags); break;
        default: row_pipeline<D, 1>(s, src, key0, key_hi, kb, qf, ws, end0, end1, rr.active, scale_log2, flags); break;
        }
    }
    if (rr.KG == 1) return;
    // combine the key groups' states into the kg == 0 warps (ring is idle now)
    constexpr int PL = D / 2 + 4;            // floats per lane
    float *red = reinterpret_cast<float *>(s.ring + team_of() * Smem<D>::kRowRing);
    const int lane = threadIdx.x & 31, warp = (threadIdx.x >> 5) % kRowWarps;
    if (rr.active && rr.kg > 0) {
        float *mine = red + warp * PL * 32;
#pragma unroll
        for (int n = 0; n < D / 8; n++)
#pragma unroll
            for (int e = 0; e < 4; e++) mine[(n * 4 + e) * 32 + lane] = ws.o[n][e];
        mine[(D / 2 + 0) * 32 + lane] = ws.m[0];
        mine[(D / 2 + 1) * 32 + lane] = ws.m[1];
        mine[(D / 2 + 2) * 32 + lane] = ws.l[0];
        mine[(D / 2 + 3) * 32 + lane] = ws.l[1];
    }
    team_sync();
    if (rr.active && rr.kg == 0) {
        for (int k = 1; k < rr.KG; k++) {
            const float *oth = red + (warp + k * rr.RGp) * PL * 32;
#pragma unroll
            for (int half = 0; half < 2; half++) {
                const float mo = oth[(D / 2 + half) * 32 + lane];
                const float lo = oth[(D / 2 + 2 + half) * 32 + lane];
                const float M = fmaxf(ws.m[half], mo);
                const float mu = (M == kNegInf) ? 0.f : M;
                const float a = ex2(ws.m[half] - mu), c = ex2(mo - mu);
                ws.l[half] = ws.l[half] * a + lo * c;
                ws.m[half] = M;
#pragma unroll
                for (int n = 0; n < D / 8; n++) {
                    ws.o[n][2 * half] = ws.o[n][2 * half] * a + oth[(n * 4 + 2 * half) * 32 + lane] * c;
                    ws.o[n][2 * half + 1] = ws.o[n][2 * half + 1] * a + oth[(n * 4 + 2 * half + 1) * 32 + lane] * c;
                }
            }
        }
    }
    team_sync();
}

// System items run over the virtual rows v = r * G + c of one KV head hk:
// query row r of the batch with query head hk * G + c, so a KV head's
// system keys are read once per 64 virtual rows whatever the head grouping
// (multi-head: G = 1, v = r).  Items of a shared prefix segment: every KV
// head, row tile and key range of it; rows of requests that do not see the
// segment get no key (their partial has lse = -inf and counts for nothing).
template <int D, int KGF>
__device__ void sys_item(const Params &p, Smem<D> &s, int item, int Mtot)
{
    // KV heads vary fastest: CTAs that run concurrently read whole [Hkv, D]
    // rows of the segment together instead of one head's slivers
    const int Mv = Mtot * p.G;
    const int T = (Mv + kTileM - 1) / kTileM;
    int seg = 0;
    if (p.n_seg > 1)
        while (seg + 1 < p.n_seg && item >= p.Hkv * T * p.seg_R[seg]) item -= p.Hkv * T * p.seg_R[seg++];
    const bool all_see = p.seg_mask == nullptr;
    const int hk = item % p.Hkv;
    const int tau = (item / p.Hkv) % T;
    const int rho = item / (p.Hkv * T);
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;

    KeySrc src{p.seg_k[seg], p.seg_v[seg], nullptr, nullptr, 0, p.Hkv, hk, 0};
    const int key0 = rho * p.seg_range[seg];
    const int key_hi = min(key0 + p.seg_range[seg], p.seg_len[seg]);

    const RowRoles rr = row_roles(min(kTileM, Mv - tau * kTileM));
    const int vW = tau * kTileM + rr.rg * 16;
    const int vA = vW + g, vB = vA + 8;
    const int rA = vA / p.G, hA = hk * p.G + vA % p.G;
    const int rB = vB / p.G, hB = hk * p.G + vB % p.G;
    const __half *qa = nullptr, *qb = nullptr;
    int endA = key0, endB = key0;     // keys the rows see: none unless their request sees the segment
    if (vA < Mv) {
        int b = find_owner(s.qo, p.B, rA);
        qa = p.q + (((size_t)b * p.Lq + (rA - s.qo[b])) * p.H + hA) * D;
        if (all_see || ((s.segm[b] >> seg) & 1u)) endA = key_hi;
    }
    if (vB < Mv) {
        int b = find_owner(s.qo, p.B, rB);
        qb = p.q + (((size_t)b * p.Lq + (rB - s.qo[b])) * p.H + hB) * D;
        if (all_see || ((s.segm[b] >> seg) & 1u)) endB = key_hi;
    }
    unsigned qf[D / 16][4];
    load_q_rows<D>(qf, qa, qb);     // the query rows are requested before the item's tiles
    row_prologue<D>(s, src, key0, key_hi, p.ctrl);
    RowState<D> ws;
#pragma unroll
    for (int d = 0; d < D / 8; d++)
#pragma unroll
        for (int e = 0; e < 4; e++) ws.o[d][e] = 0.f;
    ws.m[0] = ws.m[1] = kNegInf;
    ws.l[0] = ws.l[1] = 0.f;
    run_rows<D, KGF>(s, src, key0, key_hi, rr, qf, ws, endA, endB, p.scale_log2, p.ctrl);
    if (rr.active && rr.kg == 0)
        write_row_partials<D>(p, ws, false, p.seg_part0[seg] + rho, hA, rA, vA < Mv, hB, rB, vB < Mv);
}

// Context item of a request with several query rows (causal within the context).
template <int D>
__device__ void mq_item(const Params &p, Smem<D> &s, int local)
{
    const int b = find_owner(s.mq, p.B, local);
    const int ql = s.qo[b + 1] - s.qo[b];
    const ReqInfo ri = req_info(p, s.nctx[b], ql, s.tps);
    int j = local - s.mq[b];
    const int mtile = j % ri.mt;
    j /= ri.mt;
    const int split = j % ri.ns;
    const int h = j / ri.ns;
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2;
    const int n_ctx = ri.n_ctx;

    KeySrc src{p.k_cache, p.v_cache, p.block_tables + (size_t)b * p.max_blocks, p.prefix_ids, p.n_prefix,
               p.Hkv, h / p.G, p.num_blocks};
    auto vis = [&](int i) {   // keys row i may see: prefix + max(0, n - ql + 1 + i)
        int v = n_ctx - ql + 1 + i;
        v = v < 0 ? 0 : (v > n_ctx ? n_ctx : v);
        return p.n_prefix + v;
    };
    const int key0 = split * ri.split;
    const int last_row = min(ql, (mtile + 1) * kTileM) - 1;
    const int key_hi = min(key0 + ri.split, vis(last_row));

    const RowRoles rr = row_roles(min(kTileM, ql - mtile * kTileM));
    const int iW = mtile * kTileM + rr.rg * 16;
    const int iA = iW + g, iB = iA + 8;
    const __half *qa = iA < ql ? p.q + (((size_t)b * p.Lq + iA) * p.H + h) * D : nullptr;
    const __half *qb = iB < ql ? p.q + (((size_t)b * p.Lq + iB) * p.H + h) * D : nullptr;
    unsigned qf[D / 16][4];
    load_q_rows<D>(qf, qa, qb);     // the query rows are requested before the item's tiles
    row_prologue<D>(s, src, key0, key_hi, p.ctrl);
    const int endA = iA < ql ? min(key0 + ri.split, vis(iA)) : 0;
    const int endB = iB < ql ? min(key0 + ri.split, vis(iB)) : 0;
    RowState<D> ws;
#pragma unroll
    for (int d = 0; d < D / 8; d++)
#pragma unroll
        for (int e = 0; e < 4; e++) ws.o[d][e] = 0.f;
    ws.m[0] = ws.m[1] = kNegInf;
    ws.l[0] = ws.l[1] = 0.f;
    run_rows<D, 0>(s, src, key0, key_hi, rr, qf, ws, endA, endB, p.scale_log2, p.ctrl);
    if (rr.active && rr.kg == 0)
        write_row_partials<D>(p, ws, true, split, h, s.qo[b] + iA, iA < ql, h, s.qo[b] + iB, iB < ql);
}

// ============================================================================= phase 2: decode items
// A decode item, decoded by every lane of the warp.  Lane j also holds the
// physical block of the item's page j (fetched when the item is decoded, so
// the page loads never wait on a block-table lookup) and the lanes hold the
// query rows as the B operand of S^T = K q: multi-head, one query head in
// column 0 (lanes 0..3); grouped-query (GRP), the item's nh <= 8 query heads
// h .. h+nh-1, all reading KV head hk, in columns 0..nh-1 (lanes 4c..4c+3),
// so one pass over the pages serves the whole head group.
template <int D>
struct DecItem {
    int id;          // queue index, or -1 when the queue is exhausted
    int b, h, split;
    int hk, nh;      // KV head; query heads in the item
    int p0, np;      // first page and page count of the item
    int pp;          // prefix pages of the request's key sequence
    int n_ctx;
    int blk;         // lane j: block of page p0 + j
    unsigned qb[D / 16][2];
};

template <int D, bool GRP>
__device__ __forceinline__ void dec_item(const Params &p, const Smem<D> &s, int id, int n_dec, DecItem<D> &it)
{
    const int lane = threadIdx.x & 31;
    it.id = -1;
    it.np = 0;
    if (id >= n_dec) return;
    it.id = id;
    const int pos = find_owner(s.dec, s.n_dec_req, id);
    it.b = s.order[pos];
    it.n_ctx = s.nctx[it.b];
    const ReqInfo ri = req_info(p, it.n_ctx, 1, s.tps);
    const int j = id - s.dec[pos];
    it.split = j % ri.ns;
    const int hq = j / ri.ns;
    if (GRP) {
        const int sub = hq % p.NG;
        it.hk = hq / p.NG;
        it.h = it.hk * p.G + 8 * sub;
        it.nh = min(8, p.G - 8 * sub);
    } else {
        it.h = it.hk = hq;
        it.nh = 1;
    }
    it.p0 = it.split * ri.pages / ri.ns;
    it.np = (it.split + 1) * ri.pages / ri.ns - it.p0;
    it.pp = ri.pp;
    it.blk = -1;
    if (lane < it.np) {
        const int pg = it.p0 + lane;
        it.blk = pg < it.pp ? p.prefix_ids[pg] : p.block_tables[(size_t)it.b * p.max_blocks + (pg - it.pp)];
    }
    // column n of the B operand (lanes 4n..4n+3): rows k = 2*tig, 2*tig+1 (b0) and +8 (b1)
    const int n = lane >> 2;
    const bool has = n < it.nh;
    const __half *q = p.q + ((size_t)it.b * p.Lq * p.H + it.h + (has ? n : 0)) * D;
#pragma unroll
    for (int kt = 0; kt < D / 16; kt++) {
        const int c = kt * 16 + 2 * (lane & 3);
        it.qb[kt][0] = has ? ld_u32(q + c) : 0u;
        it.qb[kt][1] = has ? ld_u32(q + c + 8) : 0u;
    }
}

__device__ __forceinline__ int page_rows(const Params &p, int pp, int n_ctx, int pg)
{
    return pg < pp ? min(kBlock, p.n_prefix - pg * kBlock) : min(kBlock, n_ctx - (pg - pp) * kBlock);
}

// One lane's share of staging page j of the item (16 rows of K and V) into a
// ring slot; rows past the page's valid rows, or a bad block, are zero-filled.
template <int D>
__device__ __forceinline__ void load_page(const Params &p, __half *K, __half *V, const DecItem<D> &it, int j,
                                          int lane)
{
    constexpr int CPR = D / 8;
    constexpr int PER = kBlock * CPR / 32;
    const int blk = __shfl_sync(0xffffffffu, it.blk, j);
    const int rows = page_rows(p, it.pp, it.n_ctx, it.p0 + j);
    const bool ok = blk >= 0 && blk < p.num_blocks;
    if (!ok && lane == 0) atomicOr(&p.ctrl[CTRL_FLAGS], FLAG_BAD_BLOCK);
    const size_t base = (((size_t)(ok ? blk : 0) * p.Hkv + it.hk) * kBlock) * D;
#pragma unroll
    for (int k = 0; k < PER; k++) {
        int c = lane + k * 32;
        int row = c / CPR, ch = c % CPR;
        bool valid = ok && row < rows;
        size_t off = base + (size_t)row * D + ch * 8;
        int dst = swz<D>(row, ch);
        cp_async16(K + dst, valid ? p.k_cache + off : p.k_cache, valid);
        cp_async16(V + dst, valid ? p.v_cache + off : p.v_cache, valid);
    }
}

template <int D>
struct DecState {
    float o[D / 16][4];   // O^T accumulators: lane (g, tig=0) holds d = 16*mt + g (c0) and +8 (c2)
    float m;              // running max (log2 domain), uniform across the warp
    float l;              // lane partial of the normaliser
};

// One warp, one page: S^T = K q (16 keys on M, the query in column 0 of N),
// online softmax, O^T += V^T P.
template <int D>
__device__ __forceinline__ void dec_page(const __half *K, const __half *V, const unsigned (&qb)[D / 16][2],
                                         DecState<D> &st, int valid_rows, float scale_log2)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kt = 0; kt < D / 16; kt++) {
        unsigned a[4];
        int row = (lane & 7) + (((lane >> 3) & 1) << 3);
        int ch = 2 * kt + (lane >> 4);
        ldsm_x4(a[0], a[1], a[2], a[3], K + swz<D>(row, ch));
        mma16816(acc, a, qb[kt][0], qb[kt][1]);
    }
    // column 0 of S^T lives in lanes with tig == 0: key g in acc[0], key g+8 in acc[2]
    float s0 = (tig == 0 && g < valid_rows) ? acc[0] * scale_log2 : kNegInf;
    float s1 = (tig == 0 && g + 8 < valid_rows) ? acc[2] * scale_log2 : kNegInf;
    float mx = fmaxf(s0, s1);
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
    mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
    mx = __shfl_sync(0xffffffffu, mx, 0);
    const float mn = fmaxf(st.m, mx);
    const float mu = (mn == kNegInf) ? 0.f : mn;
    if (mn != st.m) {     // warp-uniform: rescale only when the running max moves
        const float al = ex2(st.m - mu);
        st.l *= al;
#pragma unroll
        for (int mt = 0; mt < D / 16; mt++)
#pragma unroll
            for (int e = 0; e < 4; e++) st.o[mt][e] *= al;
        st.m = mn;
    }
    const float p0 = ex2(s0 - mu), p1 = ex2(s1 - mu);
    st.l += p0 + p1;
    // B operand P[16 keys x 8]: lanes 0..3 (column 0) need keys 2t, 2t+1 (b0)
    // and 2t+8, 2t+9 (b1); key k's weight sits in lane 4*(k%8), p0 or p1.
    const unsigned pk = pack_half2(p0, p1);
    const unsigned x = __shfl_sync(0xffffffffu, pk, (lane & 3) * 8);
    const unsigned y = __shfl_sync(0xffffffffu, pk, (lane & 3) * 8 + 4);
    unsigned b0 = __byte_perm(x, y, 0x5410);     // (x.lo, y.lo)
    unsigned b1 = __byte_perm(x, y, 0x7632);     // (x.hi, y.hi)
    if (g != 0) b0 = b1 = 0u;
#pragma unroll
    for (int mt = 0; mt < D / 16; mt++) {
        unsigned a[4];
        int row = (lane & 7) + ((lane >> 4) << 3);
        int ch = 2 * mt + ((lane >> 3) & 1);
        ldsm_x4_t(a[0], a[1], a[2], a[3], V + swz<D>(row, ch));
        mma16816(st.o[mt], a, b0, b1);
    }
}

// Finish a decode item: write its partial (normalised output, log2-sum-exp).
template <int D>
__device__ void dec_epilogue(const Params &p, const Smem<D> &s, const DecItem<D> &it, DecState<D> &st)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    float L = st.l;
    L += __shfl_xor_sync(0xffffffffu, L, 4);
    L += __shfl_xor_sync(0xffffffffu, L, 8);
    L += __shfl_xor_sync(0xffffffffu, L, 16);
    L = __shfl_sync(0xffffffffu, L, 0);
    const float inv = L > 0.f ? 1.f / L : 0.f;
    const size_t pr = dec_slot(p, it.split, it.b, it.h);
    if (tig == 0) {
        float *po = p.part_o + pr * D;
#pragma unroll
        for (int mt = 0; mt < D / 16; mt++) {
            __stcg(po + 16 * mt + g, st.o[mt][0] * inv);
            __stcg(po + 16 * mt + g + 8, st.o[mt][2] * inv);
        }
    }
    if (lane == 0) __stcg(p.part_lse + pr, L > 0.f ? st.m + lg2(L) : kNegInf);
}

// 8x8 transpose of a b16 matrix held in the accumulator fragment layout
// (lane 4r + c: row r, columns 2c, 2c+1): the same lane then holds row r of
// the transpose.
__device__ __forceinline__ unsigned movmatrix_t(unsigned x)
{
    unsigned y;
    asm volatile("movmatrix.sync.aligned.m8n8.trans.b16 %0, %1;\n" : "=r"(y) : "r"(x));
    return y;
}

// Grouped-query state: lane (g, tig) owns columns 2*tig and 2*tig+1 (query
// heads h + 2*tig + e) of O^T and their softmax statistics.
template <int D>
struct DecStateG {
    float o[D / 16][4];   // O^T: d = 16*mt + g (c0: col 2tig, c1: col 2tig+1), d + 8 (c2, c3)
    float m[2];           // running max per owned column (log2 domain)
    float l[2];           // lane partials of the normalisers
};

// One warp, one page, up to 8 query heads of one KV head: S^T = K Q (16 keys
// on M, the heads on N), an online softmax per column, O^T += V^T P.  P moves
// from the accumulator layout of S^T into the B-operand layout with two 8x8
// transposes (keys 0-7 and 8-15).
template <int D>
__device__ __forceinline__ void dec_page_grp(const __half *K, const __half *V, const unsigned (&qb)[D / 16][2],
                                             DecStateG<D> &st, int valid_rows, int nh, float scale_log2)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    float acc[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int kt = 0; kt < D / 16; kt++) {
        unsigned a[4];
        int row = (lane & 7) + (((lane >> 3) & 1) << 3);
        int ch = 2 * kt + (lane >> 4);
        ldsm_x4(a[0], a[1], a[2], a[3], K + swz<D>(row, ch));
        mma16816(acc, a, qb[kt][0], qb[kt][1]);
    }
    // lane (g, tig): acc[0..1] = key g, columns 2tig, 2tig+1; acc[2..3] = key g+8
    const bool c0 = 2 * tig < nh, c1 = 2 * tig + 1 < nh;
    const bool r0 = g < valid_rows, r1 = g + 8 < valid_rows;
    const float s00 = (c0 && r0) ? acc[0] * scale_log2 : kNegInf;
    const float s01 = (c1 && r0) ? acc[1] * scale_log2 : kNegInf;
    const float s10 = (c0 && r1) ? acc[2] * scale_log2 : kNegInf;
    const float s11 = (c1 && r1) ? acc[3] * scale_log2 : kNegInf;
    float mx0 = fmaxf(s00, s10), mx1 = fmaxf(s01, s11);
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {      // over the 8 key rows g, for each column
        mx0 = fmaxf(mx0, __shfl_xor_sync(0xffffffffu, mx0, off));
        mx1 = fmaxf(mx1, __shfl_xor_sync(0xffffffffu, mx1, off));
    }
    const float mn0 = fmaxf(st.m[0], mx0), mn1 = fmaxf(st.m[1], mx1);
    const float mu0 = (mn0 == kNegInf) ? 0.f : mn0, mu1 = (mn1 == kNegInf) ? 0.f : mn1;
    if (__any_sync(0xffffffffu, mn0 != st.m[0] || mn1 != st.m[1])) {
        const float al0 = ex2(st.m[0] - mu0), al1 = ex2(st.m[1] - mu1);
        st.l[0] *= al0;
        st.l[1] *= al1;
#pragma unroll
        for (int mt = 0; mt < D / 16; mt++) {
            st.o[mt][0] *= al0;
            st.o[mt][2] *= al0;
            st.o[mt][1] *= al1;
            st.o[mt][3] *= al1;
        }
        st.m[0] = mn0;
        st.m[1] = mn1;
    }
    const float p00 = ex2(s00 - mu0), p01 = ex2(s01 - mu1), p10 = ex2(s10 - mu0), p11 = ex2(s11 - mu1);
    st.l[0] += p00 + p10;
    st.l[1] += p01 + p11;
    // B operand P[16 keys x 8 heads]: lane (g, tig) needs keys 2tig, 2tig+1 of
    // head g (b0) and keys 2tig+8, 2tig+9 (b1): the transposes of the lane's
    // (key g, heads 2tig..2tig+1) and (key g+8, ...) pairs.
    const unsigned b0 = movmatrix_t(pack_half2(p00, p01));
    const unsigned b1 = movmatrix_t(pack_half2(p10, p11));
#pragma unroll
    for (int mt = 0; mt < D / 16; mt++) {
        unsigned a[4];
        int row = (lane & 7) + ((lane >> 4) << 3);
        int ch = 2 * mt + ((lane >> 3) & 1);
        ldsm_x4_t(a[0], a[1], a[2], a[3], V + swz<D>(row, ch));
        mma16816(st.o[mt], a, b0, b1);
    }
}

// Finish a grouped decode item: one partial (normalised output, log2-sum-exp)
// per query head of the group.
template <int D>
__device__ void dec_epilogue_grp(const Params &p, const Smem<D> &s, const DecItem<D> &it, DecStateG<D> &st)
{
    const int lane = threadIdx.x & 31;
    const int g = lane >> 2, tig = lane & 3;
    float L[2] = {st.l[0], st.l[1]};
#pragma unroll
    for (int e = 0; e < 2; e++)
#pragma unroll
        for (int off = 4; off < 32; off <<= 1) L[e] += __shfl_xor_sync(0xffffffffu, L[e], off);
#pragma unroll
    for (int e = 0; e < 2; e++) {
        const int c = 2 * tig + e;
        if (c >= it.nh) continue;
        const float inv = L[e] > 0.f ? 1.f / L[e] : 0.f;
        const size_t pr = dec_slot(p, it.split, it.b, it.h + c);
        float *po = p.part_o + pr * D;
#pragma unroll
        for (int mt = 0; mt < D / 16; mt++) {
            __stcg(po + 16 * mt + g, st.o[mt][e] * inv);
            __stcg(po + 16 * mt + g + 8, st.o[mt][2 + e] * inv);
        }
        if (g == 0) __stcg(p.part_lse + pr, L[e] > 0.f ? st.m[e] + lg2(L[e]) : kNegInf);
    }
}

// Phase 2 for one warp: pull decode items until the queue is empty, streaming
// pages through the warp's ring and prefetching across item boundaries.  The
// item after the current one is decoded (block ids and query loads issued)
// as soon as the current one starts, and the queue ticket after that is
// requested at the same time, so no item start waits on memory.
template <int D, bool GRP>
__device__ void decode_phase(const Params &p, Smem<D> &s, int n_dec)
{
    constexpr int S = Smem<D>::kStagesW;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    // Small batches (dec_static = 3): the first three tickets of every warp
    // are static, in snake order over the longest-first queue (warp w takes
    // items w, 2 n_w - 1 - w and 2 n_w + w), so the static rounds give every
    // warp a similar load and no warp touches the queue counter before its
    // first item is done (1216 warps incrementing one address at the same
    // instant hold up the requests behind them).  Large batches, and a grid
    // whose CTAs start at different times (beside the tensor-core grid),
    // take every ticket from the queue (dec_static = 0), so that the longest
    // items go first to whichever warps run.  Queue tickets are requested
    // one item ahead.
    const unsigned n_w = gridDim.x * kWarps;
    const unsigned wid = blockIdx.x * kWarps + warp;
    const int n_static = p.dec_static;
    unsigned ticket = wid;
    if (n_static == 0 && lane == 0) ticket = atomicAdd(&p.ctrl[CTRL_DEC_ITEMS], 1u);
    int taken = 0;
    auto request = [&]() {      // ask for a ticket; its value is read later
        if (lane == 0) ticket = n_static * n_w + atomicAdd(&p.ctrl[CTRL_DEC_ITEMS], 1u);
    };
    auto take = [&](DecItem<D> &it) {
        int id = __shfl_sync(0xffffffffu, (int)ticket, 0);
        dec_item<D, GRP>(p, s, id, n_dec, it);
        ++taken;
        if (taken < n_static) ticket = (taken & 1) ? (taken + 1) * n_w - 1 - wid : taken * n_w + wid;
        else if (it.id >= 0) request();
    };

    // the first item's first pages are requested before the second item is
    // decoded
    DecItem<D> cur, nxt;
    nxt.id = -1;
    nxt.np = 0;
    take(cur);
    if (cur.id < 0) return;
    bool load_on_nxt = false;     // the loader has moved on to `nxt`
    int load_pg = 0;              // next page (relative) of the item being loaded
    int issued = 0, computed = 0;

    auto fill = [&]() {
        while (issued - computed < S - 1) {
            if (!load_on_nxt) {
                if (load_pg < cur.np) {
                    const int st = issued % S;
                    load_page<D>(p, s.wk(warp, st), s.wv(warp, st), cur, load_pg, lane);
                    cp_async_commit();
                    load_pg++;
                    issued++;
                    continue;
                }
                if (nxt.id < 0) break;
                load_on_nxt = true;
                load_pg = 0;
            }
            if (load_pg >= nxt.np) break;
            const int st = issued % S;
            load_page<D>(p, s.wk(warp, st), s.wv(warp, st), nxt, load_pg, lane);
            cp_async_commit();
            load_pg++;
            issued++;
        }
    };

    fill();
    take(nxt);
    fill();
    for (;;) {
        DecState<D> st;        // multi-head
        DecStateG<D> stg_;     // grouped-query
        if (GRP) {
#pragma unroll
            for (int mt = 0; mt < D / 16; mt++)
#pragma unroll
                for (int e = 0; e < 4; e++) stg_.o[mt][e] = 0.f;
            stg_.m[0] = stg_.m[1] = kNegInf;
            stg_.l[0] = stg_.l[1] = 0.f;
        } else {
#pragma unroll
            for (int mt = 0; mt < D / 16; mt++)
#pragma unroll
                for (int e = 0; e < 4; e++) st.o[mt][e] = 0.f;
            st.m = kNegInf;
            st.l = 0.f;
        }
        for (int j = 0; j < cur.np; j++) {
            cp_async_wait_dyn(issued - computed - 1);
            __syncwarp();
            const int stg = computed % S;
            const int rows = page_rows(p, cur.pp, cur.n_ctx, cur.p0 + j);
            if (GRP)
                dec_page_grp<D>(s.wk(warp, stg), s.wv(warp, stg), cur.qb, stg_, rows, cur.nh, p.scale_log2);
            else
                dec_page<D>(s.wk(warp, stg), s.wv(warp, stg), cur.qb, st, rows, p.scale_log2);
            __syncwarp();
            computed++;
            fill();
        }
        if (GRP)
            dec_epilogue_grp<D>(p, s, cur, stg_);
        else
            dec_epilogue<D>(p, s, cur, st);
        if (nxt.id < 0) break;
        // nxt becomes current (its pages already issued stay in flight), and
        // the item after it is decoded now
        if (!load_on_nxt) load_pg = 0;
        load_on_nxt = false;
        cur = nxt;
        take(nxt);
        fill();
    }
    cp_async_wait<0>();
    __syncwarp();
}

// ============================================================================= persistent kernel
// GRP: decode items serve a group of query heads sharing one KV head (G > 1).
// ROWS: the row items this instance handles.  -1: any (system items of any
// row count, multi-row context items).  0: none (no system items on this
// kernel, no multi-row request).  1, 2, 4: system items only, all split into
// that many key groups (the host knows it from the shape when every request
// has one query row).  The kernel starts with its code cold, and every
// pipeline compiled into it costs start-up time whether it runs or not
// (3.5 us of a 70 us step, measured), hence the instances.
template <int D, bool GRP, int ROWS>
__device__ __forceinline__ void relay_body(const Params &p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<D> &s = *reinterpret_cast<Smem<D> *>(smem_raw);

    build_schedule<D>(p, s);
    if (blockIdx.x == 0) {
        // hand the schedule to the merge kernel; tps < 0 tells it to do nothing
        for (int k = threadIdx.x; k <= p.B; k += kThreads) p.sched[1 + k] = s.qo[k];
        for (int k = threadIdx.x; k < p.B; k += kThreads) p.sched[2 + p.B + k] = s.nctx[k];
        if (threadIdx.x == 0) p.sched[0] = s.bad ? -1 : s.tps;
    }
    if (s.bad) {
        if (threadIdx.x == 0) atomicOr(&p.ctrl[CTRL_FLAGS], (unsigned)s.bad);
        return;    // counters untouched: nothing was scheduled
    }
    const int Mtot = s.qo[p.B];
    const int T = (Mtot * p.G + kTileM - 1) / kTileM;     // tiles of virtual rows per KV head
    int n_sys = 0;                                         // system items of every segment
    if (has_sys(p.mode) && !p.skip_sys)
        for (int sg = 0; sg < p.n_seg; sg++) n_sys += p.Hkv * T * p.seg_R[sg];
    const int n_rows = n_sys + (p.skip_mq ? 0 : s.mq[p.B]);
    const int n_dec = s.dec[s.n_dec_req];

    // phase 1: row items, two independent row teams per CTA (first items
    // static); a team with no row item starts on decode items at once
    if constexpr (ROWS != 0) {
        const int team = team_of();
        const bool leader = (threadIdx.x % kRowThreads) == 0;
        for (int item = blockIdx.x + team * gridDim.x; item < n_rows;) {
            if constexpr (ROWS > 0) {
                sys_item<D, ROWS>(p, s, item, Mtot);
            } else {
                if (item < n_sys) sys_item<D, 0>(p, s, item, Mtot);
                else mq_item<D>(p, s, item - n_sys);
            }
            if (leader) s.item[team] = (int)(kTeams * gridDim.x + atomicAdd(&p.ctrl[CTRL_ROW_ITEMS], 1u));
            team_sync();
            item = s.item[team];
            team_sync();
        }
    }
    // phase 2: decode items, each warp on its own
    if (n_dec > 0) decode_phase<D, GRP>(p, s, n_dec);
    __syncthreads();
    // this CTA's partials are written: the merge kernel may be launched
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <int D, bool GRP, int ROWS>
__global__ void __launch_bounds__(kThreads, 1) relay_kernel(const Params p)
{
    relay_body<D, GRP, ROWS>(p);
    // Behind the tensor-core grid this grid is a programmatic dependent: it
    // starts on the SMs that grid's last wave frees (nothing here reads what
    // that grid writes) and leaves only once that grid has completed, so
    // that its own completion, which the merge waits for, covers both.
    // Without a primary grid the wait returns at once.
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

// ============================================================================= merge kernel
// One warp per (row, head): combines the row's system partials and context
// partials.  Launched as a programmatic dependent of relay_kernel: it waits
// for that grid (and its memory) before reading anything it wrote.  SPEC
// (small batches without q_lens, where the merge is one L2 round trip after
// another): the first candidate partial rows are requested together with
// their log-sum-exps.  Otherwise (many rows: the merge is latency-bound by
// the warps resident) 8 partial rows in flight per lane and three CTAs per
// SM (four spill registers).
template <int D, bool SPEC>
__global__ void __launch_bounds__(kThreads, SPEC ? 1 : 3) merge_kernel(const Params p)
{
    __shared__ int qo[kMaxB + 1];
    __shared__ int nctx[kMaxB];
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
    // the streaming grid has finished: its queue counters go back to zero
    // for the next call (stream order puts that call's kernels after this one)
    if (blockIdx.x == 0 && threadIdx.x == 0) {
        p.ctrl[CTRL_ROW_ITEMS] = 0u;
        p.ctrl[CTRL_DEC_ITEMS] = 0u;
    }
    if (p.q_lens == nullptr) {
        // every request has Lq rows: row r is row r % Lq of request r / Lq, so
        // no schedule table is needed; the request's context length, the
        // split size and the log-sum-exps of the first 32 slots the row may
        // use are loaded together (one round trip).  Lane k's slot is part k
        // of the row whatever its context turns out to be (system ranges
        // first, then context splits), which is what merge_row reads for its
        // first 32 parts; slots past the row's own parts are inside the
        // workspace and masked there.
        const int lane = threadIdx.x & 31;
        const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
        const int r = w / p.H, h = w % p.H;
        if (r >= p.B * p.Lq) return;
        const int b = r / p.Lq;
        const int n_sys = has_sys(p.mode) ? p.R_sys : 0;
        const bool dec = p.Lq == 1;
        const int ncand = n_sys + (has_ctx(p.mode) ? (dec ? p.c_dec : p.c_mq) : 0);
        // The output rows of the first kSpec candidate parts are requested in
        // the same round trip too (slot k is part k whatever the row's part
        // count turns out to be), so a row of at most kSpec parts is merged
        // after one round trip; rows with more take the general path.
        constexpr int V = D / 32, kSpec = SPEC ? 16 : 0;
        const int d0 = lane * V;
        float x[kSpec > 0 ? kSpec : 1][V];
#pragma unroll
        for (int k = 0; k < kSpec; k++) {
            if (k < ncand) {
                const float *src = p.part_o + part_slot(p, k, n_sys, dec, r, b, h) * D + d0;
                if constexpr (V == 4) {
                    const float4 t = __ldcg(reinterpret_cast<const float4 *>(src));
                    x[k][0] = t.x; x[k][1] = t.y; x[k][2] = t.z; x[k][3] = t.w;
                } else {
                    const float2 t = __ldcg(reinterpret_cast<const float2 *>(src));
                    x[k][0] = t.x; x[k][1] = t.y;
                }
            }
        }
        float lk = kNegInf;
        if (lane < ncand) lk = __ldcg(p.part_lse + part_slot(p, lane, n_sys, dec, r, b, h));
        const int tps = __ldcg(p.sched);
        const int nc = has_ctx(p.mode) ? __ldg(p.ctx_lens + b) : 0;
        if (tps < 0) return;
        const int n_ctx = has_ctx(p.mode) ? req_info(p, nc, p.Lq, tps).ns : 0;
        const int n = n_sys + n_ctx;
        if (!SPEC || n > kSpec) {
            merge_row<D, SPEC ? 16 : 8>(p, r, b, r % p.Lq, h, n_sys, n_ctx, dec, true, lk);
            return;
        }
        constexpr float kLn2 = 0.69314718055994531f;
        if (lane >= n) lk = kNegInf;
        float M = lk;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) M = fmaxf(M, __shfl_xor_sync(0xffffffffu, M, off));
        float acc[V], W = 0.f;
#pragma unroll
        for (int v = 0; v < V; v++) acc[v] = 0.f;
        if (M != kNegInf) {
            const float wl = ex2(lk - M);      // lane k: weight of part k (0 past the row's parts)
#pragma unroll
            for (int k = 0; k < kSpec; k++) {
                const float w = __shfl_sync(0xffffffffu, wl, k);
                if (k < n && w > 0.f) {
                    W += w;
#pragma unroll
                    for (int v = 0; v < V; v++) acc[v] += w * x[k][v];
                }
            }
        }
        const float inv = W > 0.f ? 1.f / W : 0.f;
        const float lse = W > 0.f ? (M + lg2(W)) * kLn2 : kNegInf;
        const size_t orow = (size_t)r * p.H + h;        // row r = b * Lq + i
        if (p.mode == MODE_FUSED || p.mode == MODE_BASELINE) {
            __half *dst = p.out + orow * D + d0;
            if constexpr (V == 4) {
                *reinterpret_cast<uint2 *>(dst) =
                    make_uint2(pack_half2(acc[0] * inv, acc[1] * inv), pack_half2(acc[2] * inv, acc[3] * inv));
            } else {
                *reinterpret_cast<unsigned *>(dst) = pack_half2(acc[0] * inv, acc[1] * inv);
            }
            if (p.lse_out && lane == 0) p.lse_out[orow] = lse;
        } else {
            float *dst = p.o_f32 + orow * D + d0;
#pragma unroll
            for (int v = 0; v < V; v++) dst[v] = acc[v] * inv;
            if (lane == 0) p.lse_f32[orow] = lse;
        }
        return;
    }
    const int tps = p.sched[0];
    if (tps < 0) return;                 // the producer rejected its inputs
    for (int k = threadIdx.x; k <= p.B; k += blockDim.x) qo[k] = p.sched[1 + k];
    for (int k = threadIdx.x; k < p.B; k += blockDim.x) nctx[k] = p.sched[2 + p.B + k];
    __syncthreads();
    const int w = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    const int r = w / p.H, h = w % p.H;
    if (r >= qo[p.B]) return;
    const int b = find_owner(qo, p.B, r);
    const int ql = qo[b + 1] - qo[b];
    const int n_sys = has_sys(p.mode) ? p.R_sys : 0;
    const int n_ctx = has_ctx(p.mode) ? req_info(p, nctx[b], ql, tps).ns : 0;
    merge_row<D, 8>(p, r, b, r - qo[b], h, n_sys, n_ctx, ql == 1);
}

// ============================================================================= KV append
// The step's new keys and values into the paged pool (the cache write that
// precedes attention): one warp per (row slot b * Lq + i, KV head); lanes
// 0..D/8-1 copy the K row and lanes 16..16+D/8-1 the V row, 16 bytes each.
struct KvAppend {
    int B, Lq, Hkv, D, num_blocks, max_blocks;
    const __half *k_new, *v_new;      // [B, Lq, Hkv, D]
    const int *block_tables, *ctx_lens, *q_lens;
    __half *k_cache, *v_cache;        // [num_blocks, Hkv, 16, D]
    unsigned *flags;
};

__global__ void __launch_bounds__(256) kv_append_kernel(const KvAppend a)
{
    const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    if (w >= (long long)a.B * a.Lq * a.Hkv) return;
    const int hk = (int)(w % a.Hkv);
    const long long bi = w / a.Hkv;
    const int b = (int)(bi / a.Lq), i = (int)(bi % a.Lq);
    const int ql = a.q_lens ? a.q_lens[b] : a.Lq;
    if (ql < 0 || ql > a.Lq) {
        if (lane == 0 && i == 0 && hk == 0) atomicOr(a.flags, FLAG_BAD_Q_LEN);
        return;
    }
    if (i >= ql) return;
    const int n = a.ctx_lens[b];
    if (n < ql || n > a.max_blocks * kBlock) {      // the new tokens are the last ql of the context
        if (lane == 0 && i == 0 && hk == 0) atomicOr(a.flags, FLAG_BAD_CTX_LEN);
        return;
    }
    const int pos = n - ql + i;
    const int blk = a.block_tables[(size_t)b * a.max_blocks + pos / kBlock];
    if (blk < 0 || blk >= a.num_blocks) {
        if (lane == 0) atomicOr(a.flags, FLAG_BAD_BLOCK);
        return;
    }
    const int half = lane >> 4, c = lane & 15;
    if (c >= a.D / 8) return;
    const size_t src = ((size_t)bi * a.Hkv + hk) * a.D + c * 8;
    const size_t dst = (((size_t)blk * a.Hkv + hk) * kBlock + pos % kBlock) * a.D + c * 8;
    const __half *from = half ? a.v_new : a.k_new;
    __half *to = half ? a.v_cache : a.k_cache;
    *reinterpret_cast<uint4 *>(to + dst) = __ldg(reinterpret_cast<const uint4 *>(from + src));
}

// ============================================================================= rotary positions
// Rotary position embedding of the step's new rows with the system-prompt
// offset: row i of request b sits at position Ls + ctx_lens[b] - q_lens[b] + i
// (the request tokens follow the Ls system tokens).  Rotate-half pairs
// (j, j + D/2) turn by the angle pos * base^(-2j/D).  The angle reaches tens
// of thousands of radians, so it is formed and reduced modulo 2 pi in fp64
// (inv_freq[j] = base^(-2j/D) comes from the host in fp64); sine and cosine
// of the reduced angle, and the rotation, are fp32.  One warp per (row slot,
// head); q heads first, then the KV heads of k_new.
constexpr int kMaxRopePairs = 64;
struct Rope {
    int B, Lq, H, Hkv, D, Ls;
    double inv_freq[kMaxRopePairs];
    __half *q, *k;                    // [B, Lq, H, D], [B, Lq, Hkv, D] (k nullable)
    const int *ctx_lens, *q_lens;
    unsigned *flags;
};

__global__ void __launch_bounds__(256) rope_kernel(const Rope a)
{
    const long long w = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int lane = threadIdx.x & 31;
    const int nh = a.H + (a.k ? a.Hkv : 0);
    if (w >= (long long)a.B * a.Lq * nh) return;
    const int head = (int)(w % nh);
    const long long bi = w / nh;
    const int b = (int)(bi / a.Lq), i = (int)(bi % a.Lq);
    const int ql = a.q_lens ? a.q_lens[b] : a.Lq;
    const int n = a.ctx_lens[b];
    if (ql < 0 || ql > a.Lq || n < ql) {
        if (lane == 0 && i == 0 && head == 0) atomicOr(a.flags, (ql < 0 || ql > a.Lq) ? FLAG_BAD_Q_LEN : FLAG_BAD_CTX_LEN);
        return;
    }
    if (i >= ql) return;
    const double pos = (double)a.Ls + (double)(n - ql + i);
    __half *x = head < a.H ? a.q + ((size_t)bi * a.H + head) * a.D : a.k + ((size_t)bi * a.Hkv + (head - a.H)) * a.D;
    const int half = a.D / 2;
    constexpr double kTwoPi = 6.283185307179586476925286766559;
    for (int j = lane; j < half; j += 32) {
        const double ang = pos * a.inv_freq[j];
        const float red = (float)(ang - kTwoPi * rint(ang * (1.0 / kTwoPi)));   // in [-pi, pi]
        float s, c;
        sincosf(red, &s, &c);
        const float x0 = __half2float(x[j]), x1 = __half2float(x[j + half]);
        x[j] = __float2half_rn(x0 * c - x1 * s);
        x[j + half] = __float2half_rn(x1 * c + x0 * s);
    }
}

// ============================================================================= stand-alone relay fusion
// out = a*o_sys + (1-a)*o_ctx, a = e^lse_sys / (e^lse_sys + e^lse_ctx).
template <int D>
__global__ void __launch_bounds__(256) fuse_kernel(int B, int Lq, int H, const float *__restrict__ o_sys,
                                                   const float *__restrict__ lse_sys,
                                                   const float *__restrict__ o_ctx,
                                                   const float *__restrict__ lse_ctx,
                                                   const int *__restrict__ q_lens, __half *__restrict__ out,
                                                   float *__restrict__ lse_out)
{
    constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.69314718055994531f;
    const size_t rows = (size_t)B * Lq * H;
    constexpr int V = 4;   // elements per thread
    const size_t n = rows * (D / V);
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (size_t)gridDim.x * blockDim.x) {
        size_t row = idx / (D / V);
        int d = (int)(idx % (D / V)) * V;
        int b = (int)(row / ((size_t)Lq * H));
        int i = (int)((row / H) % Lq);
        int ql = q_lens ? q_lens[b] : Lq;
        if (i >= ql) continue;
        float ls = lse_sys[row] * kLog2e, lc = lse_ctx[row] * kLog2e;
        float M = fmaxf(ls, lc);
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        float lse2 = kNegInf;
        if (M != kNegInf) {
            float ws = ex2(ls - M), wc = ex2(lc - M);
            float inv = 1.f / (ws + wc);
            float a = ws * inv, c = wc * inv;
            float4 x = *reinterpret_cast<const float4 *>(o_sys + row * D + d);
            float4 y = *reinterpret_cast<const float4 *>(o_ctx + row * D + d);
            r = make_float4(a * x.x + c * y.x, a * x.y + c * y.y, a * x.z + c * y.z, a * x.w + c * y.w);
            lse2 = M + lg2(ws + wc);
        }
        uint2 pk = make_uint2(pack_half2(r.x, r.y), pack_half2(r.z, r.w));
        *reinterpret_cast<uint2 *>(out + row * D + d) = pk;
        if (lse_out && d == 0) lse_out[row] = lse2 * kLn2;
    }
}

// ============================================================================= relay fusion of K parts
// The relay fusion generalised from two parts to K (a tree of shared
// prefixes: one part per shared level plus the context): out = sum_k w_k o_k,
// w_k = e^lse_k / sum_j e^lse_j, lse = log sum_k e^lse_k.  A part with
// lse = -inf for a row contributes nothing to it.
constexpr int kMaxFuseParts = 16;
struct FuseN {
    int B, Lq, H, K;
    const float *o[kMaxFuseParts];      // [B, Lq, H, D] fp32
    const float *lse[kMaxFuseParts];    // [B, Lq, H] natural log
    const int *q_lens;
    __half *out;
    float *lse_out;
};

template <int D>
__global__ void __launch_bounds__(256) fuse_n_kernel(const FuseN f)
{
    constexpr float kLog2e = 1.4426950408889634f, kLn2 = 0.69314718055994531f;
    constexpr int V = 4;   // elements per thread
    const size_t rows = (size_t)f.B * f.Lq * f.H;
    const size_t n = rows * (D / V);
    for (size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x; idx < n; idx += (size_t)gridDim.x * blockDim.x) {
        const size_t row = idx / (D / V);
        const int d = (int)(idx % (D / V)) * V;
        const int b = (int)(row / ((size_t)f.Lq * f.H));
        const int i = (int)((row / f.H) % f.Lq);
        const int ql = f.q_lens ? f.q_lens[b] : f.Lq;
        if (i >= ql) continue;
        float M = kNegInf;
        for (int k = 0; k < f.K; k++) M = fmaxf(M, f.lse[k][row] * kLog2e);
        float4 r = make_float4(0.f, 0.f, 0.f, 0.f);
        float lse2 = kNegInf;
        if (M != kNegInf) {
            float W = 0.f;
            for (int k = 0; k < f.K; k++) {
                const float w = ex2(f.lse[k][row] * kLog2e - M);
                if (w == 0.f) continue;                  // an empty part: its o is never read
                const float4 x = *reinterpret_cast<const float4 *>(f.o[k] + row * D + d);
                r.x += w * x.x;
                r.y += w * x.y;
                r.z += w * x.z;
                r.w += w * x.w;
                W += w;
            }
            const float inv = 1.f / W;
            r = make_float4(r.x * inv, r.y * inv, r.z * inv, r.w * inv);
            lse2 = M + lg2(W);
        }
        *reinterpret_cast<uint2 *>(f.out + row * D + d) = make_uint2(pack_half2(r.x, r.y), pack_half2(r.z, r.w));
        if (f.lse_out && d == 0) f.lse_out[row] = lse2 * kLn2;
    }
}

}  // namespace relay
