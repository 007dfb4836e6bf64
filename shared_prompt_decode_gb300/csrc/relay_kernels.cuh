// Device code of librelay: the persistent relay-attention kernel and the
// stand-alone fusion kernel, for sm_103a.
//
// One kernel, four modes:
//   MODE_FUSED     system items + context items, merged into fp16 out
//   MODE_SYS       system items only, merged into fp32 o_sys / lse_sys
//   MODE_CTX       context items only, merged into fp32 o_ctx / lse_ctx
//   MODE_BASELINE  context items over [system blocks; context] per request
//
// Work items (scheduled dynamically by an atomic counter over a persistent
// grid, largest items first):
//   system item  (h, key range rho, row tile tau): 64 query rows of the whole
//                batch against one range of system keys.  This is the
//                matrix-matrix product of the system-attention step
//                (atyun.com RelayAttention article, section "RelayAttention").
//   multi-row context item (b, h, split, row tile): up to 64 query rows of one
//                request against a range of its paged context, causal mask.
//   decode context item (b, h, split): the single query row of a decode
//                request against a range of its paged context; the four
//                warps split the keys of each tile.
// Every item computes with mma.sync m16n8k16 (fp16 in, fp32 accumulate)
// over K/V tiles of 64 keys staged through a 3-deep cp.async ring in
// XOR-swizzled shared memory, keeps an online softmax in the log2 domain,
// and writes one fp32 partial (normalised output + log2-sum-exp).  The item
// that brings a (request, head) counter to its target merges all partials of
// that pair -- the relay fusion, generalised to any number of parts.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace relay {

constexpr int kBlock = 16;      // paged block size (tokens)
constexpr int kWarps = 4;
constexpr int kThreads = kWarps * 32;
constexpr int kTileK = 64;      // keys per pipeline stage
constexpr int kTileM = 64;      // query rows per row-tile item (16 per warp)
constexpr int kStages = 3;
constexpr int kMaxB = 512;

enum Mode : int { MODE_FUSED = 0, MODE_SYS = 1, MODE_CTX = 2, MODE_BASELINE = 3 };

enum : unsigned {
    FLAG_BAD_Q_LEN = 1u, FLAG_BAD_CTX_LEN = 2u, FLAG_BAD_BLOCK = 4u, FLAG_Q_TOTAL = 8u
};

struct Params {
    int B, Lq, H, Ls, num_blocks, max_blocks, max_q_total;
    float scale_log2;                 // softmax scale * log2(e)
    const __half *q, *sys_k, *sys_v, *k_cache, *v_cache;
    const int *block_tables, *ctx_lens, *q_lens;
    const int *prefix_ids;            // baseline: system blocks in the pool
    int n_prefix;                     // baseline: system tokens ahead of each context
    __half *out;                      // fused / baseline output
    float *lse_out;                   // nullable
    float *o_f32, *lse_f32;           // sys-only / ctx-only outputs
    unsigned *ctrl;                   // [0] flags, [1] work counter, [2] finished CTAs
    unsigned *arrive;                 // [B*H] arrival counters
    float *part_o;                    // [n_parts][max_q_total][H][D]
    float *part_lse;                  // [n_parts][max_q_total][H]  (log2 domain)
    int R_sys, sys_range, ctx_split, ctx_base;   // ctx_base: first partial slot of context parts
    int mode;
};

template <int D>
struct Smem {
    __half k[kStages][kTileK * D];
    __half v[kStages][kTileK * D];
    float red_o[kWarps][D];
    float red_m[kWarps];
    float red_l[kWarps];
    int qo[kMaxB + 1];        // exclusive prefix of query rows
    int mq[kMaxB + 1];        // exclusive prefix of multi-row context items
    int dec[kMaxB + 1];       // exclusive prefix of decode context items
    int warp_tot[3][kWarps];
    int item;
    int bad;
    int n_merge;
    int merge_b[kTileM + kThreads];
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
struct ReqInfo {
    int ql;       // query rows
    int nkeys;    // keys of the context sequence (prefix + context)
    int split;    // keys per context item
    int ns;       // context items along the keys
    int mt;       // row tiles (1 for decode rows)
};

__device__ __forceinline__ ReqInfo req_info(const Params &p, int b, int ql)
{
    ReqInfo r;
    r.ql = ql;
    r.nkeys = p.n_prefix + p.ctx_lens[b];
    if (ql <= 1) {
        r.split = p.ctx_split;
    } else {
        // Longer splits for multi-row requests keep the partial traffic small
        // next to the keys each item streams.
        int want = ql * 64;
        r.split = ((want + p.ctx_split - 1) / p.ctx_split) * p.ctx_split;
        if (r.split < p.ctx_split) r.split = p.ctx_split;
    }
    r.ns = (r.nkeys + r.split - 1) / r.split;
    if (r.ns < 1) r.ns = 1;
    r.mt = (ql + kTileM - 1) / kTileM;
    return r;
}

__device__ __forceinline__ bool has_sys(int mode) { return mode == MODE_FUSED || mode == MODE_SYS; }
__device__ __forceinline__ bool has_ctx(int mode) { return mode != MODE_SYS; }

// Per-CTA prefix sums over the batch (B <= kMaxB, four entries per thread).
template <int D>
__device__ void build_schedule(const Params &p, Smem<D> &s)
{
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int cnt[3][4];
    int loc[3] = {0, 0, 0};
    unsigned flags = 0;
    for (int k = 0; k < 4; k++) {
        int b = tid * 4 + k;
        int c0 = 0, c1 = 0, c2 = 0;
        if (b < p.B) {
            int ql = p.q_lens ? p.q_lens[b] : p.Lq;
            int n = p.ctx_lens ? p.ctx_lens[b] : 0;
            if (ql < 0 || ql > p.Lq) { flags |= FLAG_BAD_Q_LEN; ql = 0; }
            if (has_ctx(p.mode) && (n < 0 || n > p.max_blocks * kBlock)) { flags |= FLAG_BAD_CTX_LEN; ql = 0; }
            c0 = ql;
            if (has_ctx(p.mode) && ql > 0) {
                ReqInfo r = req_info(p, b, ql);
                if (ql > 1) c1 = p.H * r.ns * r.mt; else c2 = p.H * r.ns;
            }
        }
        cnt[0][k] = c0; cnt[1][k] = c1; cnt[2][k] = c2;
        loc[0] += c0; loc[1] += c1; loc[2] += c2;
    }
    // warp-level inclusive scan of the per-thread totals
    int inc[3] = {loc[0], loc[1], loc[2]};
    for (int off = 1; off < 32; off <<= 1) {
        for (int a = 0; a < 3; a++) {
            int v = __shfl_up_sync(0xffffffffu, inc[a], off);
            if (lane >= off) inc[a] += v;
        }
    }
    if (lane == 31)
        for (int a = 0; a < 3; a++) s.warp_tot[a][warp] = inc[a];
    if (tid == 0) s.bad = 0;
    __syncthreads();
    if (flags) atomicOr(&s.bad, (int)flags);
    int base[3];
    for (int a = 0; a < 3; a++) {
        int w = 0;
        for (int j = 0; j < warp; j++) w += s.warp_tot[a][j];
        base[a] = w + inc[a] - loc[a];
    }
    int *arr[3] = {s.qo, s.mq, s.dec};
    for (int k = 0; k < 4; k++) {
        int b = tid * 4 + k;
        if (b < p.B)
            for (int a = 0; a < 3; a++) {
                arr[a][b] = base[a];
                base[a] += cnt[a][k];
            }
    }
    if (tid == kThreads - 1)    // the last thread's running sums are the totals
        for (int a = 0; a < 3; a++) arr[a][p.B] = base[a];
    __syncthreads();
    if (tid == 0 && s.qo[p.B] > p.max_q_total) s.bad |= FLAG_Q_TOTAL;
    __syncthreads();
}

// ----------------------------------------------------------------------------- key sources
struct KeySrc {
    const __half *k, *v;
    const int *table;       // this request's block table row (paged) or nullptr (system cache)
    const int *prefix;      // baseline: system blocks
    int n_prefix;
    int H, h, num_blocks;
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
    constexpr int PER = kTileK * CPR / kThreads;    // chunks per thread
    const int tid = threadIdx.x;
#pragma unroll
    for (int k = 0; k < PER; k++) {
        int c = tid + k * kThreads;
        int key = c / CPR, ch = c % CPR;
        int t = key0 + key;
        size_t off = 0;
        bool valid = t < key_end;
        if (valid) valid = key_offset(src, t, off, flags, D);
        int dst = key * D + ((ch ^ (key & 7)) << 3);
        cp_async16(&s.k[st][dst], valid ? src.k + off + ch * 8 : src.k, valid);
        cp_async16(&s.v[st][dst], valid ? src.v + off + ch * 8 : src.v, valid);
    }
}

// ----------------------------------------------------------------------------- warp attention core
// One warp: 16 query rows (A fragments in qf) against NT*8 keys of the staged
// tile starting at tile row kb.  Online softmax state per lane: rows g, g+8.
template <int D, int NT>
struct WarpState {
    float o[D / 8][4];
    float m[2], l[2];
};

template <int D, int NT>
__device__ __forceinline__ void warp_tile(const Smem<D> &s, int st, int kb, const unsigned (&qf)[D / 16][4],
                                          WarpState<D, NT> &ws, int key_tile0, int end0, int end1,
                                          float scale_log2)
{
    const int lane = threadIdx.x & 31;
    const __half *K = s.k[st];
    const __half *V = s.v[st];
    float sc[NT][4];
#pragma unroll
    for (int n = 0; n < NT; n++)
#pragma unroll
        for (int e = 0; e < 4; e++) sc[n][e] = 0.f;

    // S = Q K^T
#pragma unroll
    for (int kt = 0; kt < D / 16; kt++) {
#pragma unroll
        for (int np = 0; np < NT / 2; np++) {
            int row = kb + np * 16 + (lane & 7) + ((lane >> 4) << 3);
            int ch = 2 * kt + ((lane >> 3) & 1);
            unsigned b0, b1, b2, b3;
            ldsm_x4(b0, b1, b2, b3, K + row * D + ((ch ^ (row & 7)) << 3));
            mma16816(sc[2 * np], qf[kt], b0, b1);
            mma16816(sc[2 * np + 1], qf[kt], b2, b3);
        }
    }

    // scale, mask, online softmax (log2 domain)
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

    // O += P V
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
            ldsm_x4_t(b0, b1, b2, b3, V + row * D + ((ch ^ (row & 7)) << 3));
            mma16816(ws.o[2 * dp], pa, b0, b1);
            mma16816(ws.o[2 * dp + 1], pa, b2, b3);
        }
    }
}

template <int D, int NT>
__device__ __forceinline__ void warp_state_init(WarpState<D, NT> &ws)
{
#pragma unroll
    for (int d = 0; d < D / 8; d++)
#pragma unroll
        for (int e = 0; e < 4; e++) ws.o[d][e] = 0.f;
    ws.m[0] = ws.m[1] = kNegInf;
    ws.l[0] = ws.l[1] = 0.f;
}

// Run the key-tile pipeline over [key0, key_hi) for this CTA's warps.
// ROWS: each warp owns 16 rows and all 64 keys of a tile (NT = 8);
// otherwise the warps share one padded row block and split each tile's keys
// (NT = 2, warp w takes keys 16w..16w+15).
template <int D, bool ROWS>
__device__ __forceinline__ void run_pipeline(Smem<D> &s, const KeySrc &src, int key0, int key_hi,
                                             const unsigned (&qf)[D / 16][4],
                                             WarpState<D, ROWS ? 8 : 2> &ws, int end0, int end1,
                                             float scale_log2, unsigned *flags)
{
    constexpr int NT = ROWS ? 8 : 2;
    const int warp = threadIdx.x >> 5;
    int n_tiles = (key_hi > key0) ? (key_hi - key0 + kTileK - 1) / kTileK : 0;
    // prologue was issued by the caller (so that Q loads overlap it)
    for (int j = 0; j < n_tiles; j++) {
        cp_async_wait<kStages - 2>();
        __syncthreads();
        int jn = j + kStages - 1;
        if (jn < n_tiles) load_tile<D>(s, jn % kStages, src, key0 + jn * kTileK, key_hi, flags);
        cp_async_commit();
        warp_tile<D, NT>(s, j % kStages, ROWS ? 0 : warp * 16, qf, ws, key0 + j * kTileK, end0, end1, scale_log2);
    }
    cp_async_wait<0>();
    __syncthreads();
}

template <int D>
__device__ __forceinline__ void issue_prologue(Smem<D> &s, const KeySrc &src, int key0, int key_hi, unsigned *flags)
{
    int n_tiles = (key_hi > key0) ? (key_hi - key0 + kTileK - 1) / kTileK : 0;
#pragma unroll
    for (int j = 0; j < kStages - 1; j++) {
        if (j < n_tiles) load_tile<D>(s, j, src, key0 + j * kTileK, key_hi, flags);
        cp_async_commit();
    }
}

// ----------------------------------------------------------------------------- merge (relay fusion)
__device__ __forceinline__ size_t part_row(const Params &p, int part, int r, int h)
{
    return ((size_t)part * p.max_q_total + r) * p.H + h;
}

// Merge every partial of (b, h) into the output: the convex combination of
// the parts weighted by their softmax mass.  Called by all threads of the CTA
// that completed the pair.
template <int D>
__device__ void merge_pair(const Params &p, const Smem<D> &s, int b, int h)
{
    const int r0 = s.qo[b], r1 = s.qo[b + 1];
    const int ql = r1 - r0;
    const int n_sys = has_sys(p.mode) ? p.R_sys : 0;
    int n_ctx = 0;
    if (has_ctx(p.mode)) n_ctx = req_info(p, b, ql).ns;
    constexpr int RPP = kThreads / D;    // rows per pass (1 for D=128, 2 for D=64)
    const int d = threadIdx.x % D;
    for (int rr = threadIdx.x / D; rr < ql; rr += RPP) {
        int r = r0 + rr;
        float M = kNegInf;
        for (int j = 0; j < n_sys + n_ctx; j++) {
            int part = j < n_sys ? j : p.ctx_base + (j - n_sys);
            M = fmaxf(M, __ldcg(p.part_lse + part_row(p, part, r, h)));
        }
        float W = 0.f, acc = 0.f;
        if (M != kNegInf) {
            for (int j = 0; j < n_sys + n_ctx; j++) {
                int part = j < n_sys ? j : p.ctx_base + (j - n_sys);
                size_t pr = part_row(p, part, r, h);
                float w = ex2(__ldcg(p.part_lse + pr) - M);
                W += w;
                acc += w * __ldcg(p.part_o + pr * D + d);
            }
        }
        float o = (W > 0.f) ? acc / W : 0.f;
        float lse2 = (W > 0.f) ? M + lg2(W) : kNegInf;
        size_t orow = ((size_t)b * p.Lq + rr) * p.H + h;
        if (p.mode == MODE_FUSED || p.mode == MODE_BASELINE) {
            p.out[orow * D + d] = __float2half_rn(o);
            if (p.lse_out && d == 0) p.lse_out[orow] = lse2 * 0.69314718055994531f;
        } else {
            p.o_f32[orow * D + d] = o;
            if (d == 0) p.lse_f32[orow] = lse2 * 0.69314718055994531f;
        }
    }
}

// Count the item's arrival for (b, h); returns true to the one thread whose
// increment completed the pair.
__device__ __forceinline__ bool arrive(const Params &p, int b, int h, int target)
{
    unsigned old = atomicAdd(&p.arrive[b * p.H + h], 1u);
    if ((int)old + 1 == target) {
        p.arrive[b * p.H + h] = 0;   // every arrival is in: reset for the next call
        return true;
    }
    return false;
}

template <int D>
__device__ __forceinline__ int pair_target(const Params &p, const Smem<D> &s, int b)
{
    const int r0 = s.qo[b], r1 = s.qo[b + 1];
    int t = 0;
    if (r1 <= r0) return 0;
    if (has_sys(p.mode)) t += p.R_sys * ((r1 - 1) / kTileM - r0 / kTileM + 1);
    if (has_ctx(p.mode)) {
        ReqInfo ri = req_info(p, b, r1 - r0);
        t += ri.ns * ri.mt;
    }
    return t;
}

// ----------------------------------------------------------------------------- items
template <int D>
__device__ void sys_item(const Params &p, Smem<D> &s, int item, int Mtot)
{
    const int T = (Mtot + kTileM - 1) / kTileM;
    const int tau = item % T;
    const int rho = (item / T) % p.R_sys;
    const int h = item / (T * p.R_sys);
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, tig = lane & 3;

    KeySrc src{p.sys_k, p.sys_v, nullptr, nullptr, 0, p.H, h, 0};
    const int key0 = rho * p.sys_range;
    int key_hi = key0 + p.sys_range;
    if (key_hi > p.Ls) key_hi = p.Ls;
    issue_prologue<D>(s, src, key0, key_hi, p.ctrl);

    // Q fragments: rows tau*64 + 16*warp + {g, g+8}
    const int rA = tau * kTileM + warp * 16 + g, rB = rA + 8;
    const __half *qa = nullptr, *qb = nullptr;
    if (rA < Mtot) {
        int b = find_owner(s.qo, p.B, rA);
        qa = p.q + (((size_t)b * p.Lq + (rA - s.qo[b])) * p.H + h) * D;
    }
    if (rB < Mtot) {
        int b = find_owner(s.qo, p.B, rB);
        qb = p.q + (((size_t)b * p.Lq + (rB - s.qo[b])) * p.H + h) * D;
    }
    unsigned qf[D / 16][4];
#pragma unroll
    for (int kt = 0; kt < D / 16; kt++) {
        int c = kt * 16 + 2 * tig;
        qf[kt][0] = qa ? ld_u32(qa + c) : 0u;
        qf[kt][1] = qb ? ld_u32(qb + c) : 0u;
        qf[kt][2] = qa ? ld_u32(qa + c + 8) : 0u;
        qf[kt][3] = qb ? ld_u32(qb + c + 8) : 0u;
    }
    WarpState<D, 8> ws;
    warp_state_init(ws);
    run_pipeline<D, true>(s, src, key0, key_hi, qf, ws, key_hi, key_hi, p.scale_log2, p.ctrl);

    // partial for rows rA, rB
    float l0 = ws.l[0], l1 = ws.l[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const int part = rho;
#pragma unroll
    for (int half = 0; half < 2; half++) {
        int r = half ? rB : rA;
        if (r >= Mtot) continue;
        float l = half ? l1 : l0, m = ws.m[half];
        float inv = l > 0.f ? 1.f / l : 0.f;
        size_t pr = part_row(p, part, r, h);
        float *po = p.part_o + pr * D;
#pragma unroll
        for (int n = 0; n < D / 8; n++) {
            float2 v = make_float2(ws.o[n][2 * half] * inv, ws.o[n][2 * half + 1] * inv);
            __stcg(reinterpret_cast<float2 *>(po + n * 8 + 2 * tig), v);
        }
        if (tig == 0) __stcg(p.part_lse + pr, l > 0.f ? m + lg2(l) : kNegInf);
    }
    __threadfence();
    __syncthreads();

    // arrivals for every request with rows in this tile
    const int r0 = tau * kTileM;
    const int r1 = min(Mtot, r0 + kTileM);
    const int bf = find_owner(s.qo, p.B, r0), bl = find_owner(s.qo, p.B, r1 - 1);
    if (threadIdx.x == 0) s.n_merge = 0;
    __syncthreads();
    for (int b = bf + threadIdx.x; b <= bl; b += kThreads) {
        if (s.qo[b + 1] > s.qo[b] && arrive(p, b, h, pair_target(p, s, b))) {
            int k = atomicAdd(&s.n_merge, 1);
            s.merge_b[k] = b;
        }
    }
    __syncthreads();
    if (s.n_merge > 0) {
        __threadfence();
        for (int k = 0; k < s.n_merge; k++) merge_pair<D>(p, s, s.merge_b[k], h);
    }
    __syncthreads();
}

// Context item for a request with several query rows (causal within the context).
template <int D>
__device__ void mq_item(const Params &p, Smem<D> &s, int local)
{
    const int b = find_owner(s.mq, p.B, local);
    const int ql = s.qo[b + 1] - s.qo[b];
    ReqInfo ri = req_info(p, b, ql);
    int j = local - s.mq[b];
    const int mtile = j % ri.mt;
    j /= ri.mt;
    const int split = j % ri.ns;
    const int h = j / ri.ns;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, tig = lane & 3;
    const int n_ctx = p.ctx_lens[b];

    KeySrc src{p.k_cache, p.v_cache, p.block_tables + (size_t)b * p.max_blocks, p.prefix_ids, p.n_prefix,
               p.H, h, p.num_blocks};
    // visible keys of row i: prefix + max(0, n - ql + 1 + i)
    auto vis = [&](int i) {
        int v = n_ctx - ql + 1 + i;
        v = v < 0 ? 0 : (v > n_ctx ? n_ctx : v);
        return p.n_prefix + v;
    };
    const int key0 = split * ri.split;
    const int last_row = min(ql, (mtile + 1) * kTileM) - 1;
    int key_hi = min(key0 + ri.split, vis(last_row));
    issue_prologue<D>(s, src, key0, key_hi, p.ctrl);

    const int iA = mtile * kTileM + warp * 16 + g, iB = iA + 8;
    const __half *qa = iA < ql ? p.q + (((size_t)b * p.Lq + iA) * p.H + h) * D : nullptr;
    const __half *qb = iB < ql ? p.q + (((size_t)b * p.Lq + iB) * p.H + h) * D : nullptr;
    unsigned qf[D / 16][4];
#pragma unroll
    for (int kt = 0; kt < D / 16; kt++) {
        int c = kt * 16 + 2 * tig;
        qf[kt][0] = qa ? ld_u32(qa + c) : 0u;
        qf[kt][1] = qb ? ld_u32(qb + c) : 0u;
        qf[kt][2] = qa ? ld_u32(qa + c + 8) : 0u;
        qf[kt][3] = qb ? ld_u32(qb + c + 8) : 0u;
    }
    const int endA = iA < ql ? min(key0 + ri.split, vis(iA)) : 0;
    const int endB = iB < ql ? min(key0 + ri.split, vis(iB)) : 0;
    WarpState<D, 8> ws;
    warp_state_init(ws);
    run_pipeline<D, true>(s, src, key0, key_hi, qf, ws, endA, endB, p.scale_log2, p.ctrl);

    float l0 = ws.l[0], l1 = ws.l[1];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 1);
    l1 += __shfl_xor_sync(0xffffffffu, l1, 2);
    const int part = p.ctx_base + split;
#pragma unroll
    for (int half = 0; half < 2; half++) {
        int i = half ? iB : iA;
        if (i >= ql) continue;
        float l = half ? l1 : l0, m = ws.m[half];
        float inv = l > 0.f ? 1.f / l : 0.f;
        size_t pr = part_row(p, part, s.qo[b] + i, h);
        float *po = p.part_o + pr * D;
#pragma unroll
        for (int n = 0; n < D / 8; n++) {
            float2 v = make_float2(ws.o[n][2 * half] * inv, ws.o[n][2 * half + 1] * inv);
            __stcg(reinterpret_cast<float2 *>(po + n * 8 + 2 * tig), v);
        }
        if (tig == 0) __stcg(p.part_lse + pr, l > 0.f ? m + lg2(l) : kNegInf);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s.n_merge = arrive(p, b, h, pair_target(p, s, b)) ? 1 : 0;
    __syncthreads();
    if (s.n_merge) {
        __threadfence();
        merge_pair<D>(p, s, b, h);
    }
    __syncthreads();
}

// Context item for a decode request (one query row).
template <int D>
__device__ void dec_item(const Params &p, Smem<D> &s, int local)
{
    const int b = find_owner(s.dec, p.B, local);
    ReqInfo ri = req_info(p, b, 1);
    const int j = local - s.dec[b];
    const int split = j % ri.ns;
    const int h = j / ri.ns;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, tig = lane & 3;

    KeySrc src{p.k_cache, p.v_cache, p.block_tables + (size_t)b * p.max_blocks, p.prefix_ids, p.n_prefix,
               p.H, h, p.num_blocks};
    const int key0 = split * ri.split;
    const int key_hi = min(key0 + ri.split, ri.nkeys);
    issue_prologue<D>(s, src, key0, key_hi, p.ctrl);

    // the one real query row sits in row 0 of the padded 16-row block
    const __half *qrow = p.q + ((size_t)b * p.Lq * p.H + h) * D;
    unsigned qf[D / 16][4];
#pragma unroll
    for (int kt = 0; kt < D / 16; kt++) {
        int c = kt * 16 + 2 * tig;
        qf[kt][0] = (g == 0) ? ld_u32(qrow + c) : 0u;
        qf[kt][1] = 0u;
        qf[kt][2] = (g == 0) ? ld_u32(qrow + c + 8) : 0u;
        qf[kt][3] = 0u;
    }
    WarpState<D, 2> ws;
    warp_state_init(ws);
    run_pipeline<D, false>(s, src, key0, key_hi, qf, ws, key_hi, key_hi, p.scale_log2, p.ctrl);

    // combine the four warps' states of row 0
    float l0 = ws.l[0];
    l0 += __shfl_xor_sync(0xffffffffu, l0, 1);
    l0 += __shfl_xor_sync(0xffffffffu, l0, 2);
    if (g == 0) {
#pragma unroll
        for (int n = 0; n < D / 8; n++) {
            s.red_o[warp][n * 8 + 2 * tig] = ws.o[n][0];
            s.red_o[warp][n * 8 + 2 * tig + 1] = ws.o[n][1];
        }
        if (tig == 0) {
            s.red_m[warp] = ws.m[0];
            s.red_l[warp] = l0;
        }
    }
    __syncthreads();
    const int part = p.ctx_base + split;
    const size_t pr = part_row(p, part, s.qo[b], h);
    if (threadIdx.x < D) {
        const int d = threadIdx.x;
        float M = kNegInf;
#pragma unroll
        for (int w = 0; w < kWarps; w++) M = fmaxf(M, s.red_m[w]);
        float L = 0.f, acc = 0.f;
        if (M != kNegInf) {
#pragma unroll
            for (int w = 0; w < kWarps; w++) {
                float c = ex2(s.red_m[w] - M);
                L += c * s.red_l[w];
                acc += c * s.red_o[w][d];
            }
        }
        __stcg(p.part_o + pr * D + d, L > 0.f ? acc / L : 0.f);
        if (d == 0) __stcg(p.part_lse + pr, L > 0.f ? M + lg2(L) : kNegInf);
    }
    __threadfence();
    __syncthreads();
    if (threadIdx.x == 0) s.n_merge = arrive(p, b, h, pair_target(p, s, b)) ? 1 : 0;
    __syncthreads();
    if (s.n_merge) {
        __threadfence();
        merge_pair<D>(p, s, b, h);
    }
    __syncthreads();
}

// ----------------------------------------------------------------------------- persistent kernel
template <int D>
__global__ void __launch_bounds__(kThreads, 2) relay_kernel(const Params p)
{
    extern __shared__ __align__(128) unsigned char smem_raw[];
    Smem<D> &s = *reinterpret_cast<Smem<D> *>(smem_raw);

    build_schedule<D>(p, s);
    if (s.bad) {
        if (threadIdx.x == 0) atomicOr(&p.ctrl[0], (unsigned)s.bad);
        return;    // counters untouched: nothing was scheduled
    }
    const int Mtot = s.qo[p.B];
    const int T = (Mtot + kTileM - 1) / kTileM;
    const int n_sys = has_sys(p.mode) ? p.H * p.R_sys * T : 0;
    const int n_mq = s.mq[p.B];
    const int n_dec = s.dec[p.B];
    const int total = n_sys + n_mq + n_dec;

    for (;;) {
        if (threadIdx.x == 0) s.item = (int)atomicAdd(&p.ctrl[1], 1u);
        __syncthreads();
        const int item = s.item;
        __syncthreads();
        if (item >= total) break;
        if (item < n_sys) sys_item<D>(p, s, item, Mtot);
        else if (item < n_sys + n_mq) mq_item<D>(p, s, item - n_sys);
        else dec_item<D>(p, s, item - n_sys - n_mq);
    }
    // the last CTA out resets the work counters for the next launch
    if (threadIdx.x == 0) {
        __threadfence();
        unsigned done = atomicAdd(&p.ctrl[2], 1u);
        if (done == gridDim.x - 1) {
            p.ctrl[1] = 0u;
            p.ctrl[2] = 0u;
            __threadfence();
        }
    }
}

// ----------------------------------------------------------------------------- stand-alone relay fusion
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
        __half2 h0 = __floats2half2_rn(r.x, r.y), h1 = __floats2half2_rn(r.z, r.w);
        uint2 pk;
        pk.x = *reinterpret_cast<unsigned *>(&h0);
        pk.y = *reinterpret_cast<unsigned *>(&h1);
        *reinterpret_cast<uint2 *>(out + row * D + d) = pk;
        if (lse_out && d == 0) lse_out[row] = lse2 * kLn2;
    }
}

}  // namespace relay
