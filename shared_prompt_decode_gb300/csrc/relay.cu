// librelay: host side of the C ABI declared in include/relay.h.
//
// Host work is argument checking, the workspace layout, the choice of work
// item sizes, and one launch per call.  No allocation, no synchronisation
// (relay_device_status excepted), no state beyond a per-device cache of the
// SM count and the kernels' occupancy.
#include <cuda_runtime.h>
#include <cudaTypedefs.h>

#include <algorithm>
#include <climits>
#include <cmath>
#include <cstdint>
#include <mutex>

#include "relay.h"
#include "relay_kernels.cuh"
#include "sys_tc.cuh"

namespace {

using namespace relay;

constexpr int kMaxDevices = 64;
constexpr int kAutoCtxSplit = 512;
constexpr int kMaxMqParts = 8;         // context splits of a multi-row request, at most
static_assert(RELAY_MAX_SEGMENTS == kMaxSegments, "segment limit of the header and the kernels");
static_assert(tc::kPageTC == kBlock, "page size of the tensor-core context path");
static_assert(tc::kMaxBatchTC == kMaxB, "batch limit of the tensor-core kernel");

struct DevInfo {
    bool ready = false;
    int sms = 0;
    int occ64 = 0, occ128 = 0;
};

// Streaming-kernel instances: D = 128 has one per row-item class (ROWS =
// -1: any; 0: none; 1, 2, 4: system items only, in that many key groups), in
// the multi-head and grouped-query flavours; D = 64 has the general one.
template <int D, bool GRP, int ROWS>
cudaError_t prepare_one(int *occ)
{
    cudaError_t e = cudaFuncSetAttribute(relay_kernel<D, GRP, ROWS>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sizeof(Smem<D>));
    int o = 0;
    if (e == cudaSuccess)
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&o, relay_kernel<D, GRP, ROWS>, kThreads, sizeof(Smem<D>));
    *occ = std::min(*occ, o);
    return e;
}

// Batches with more query rows per head than this run the system step on the
// tensor cores (tcgen05), where it is compute-bound; below it the step stays
// inside the streaming kernel, where it is memory-bound and overlaps context.
constexpr int kTcMinRows = 256;
constexpr int kTcCtxMinRows = 64;      // rows of a request per KV head (Lq G) for its context on tcgen05
constexpr int kTcYieldPct = 24;        // most SMs that stream decode contexts beside the tensor cores, %
DevInfo g_dev[kMaxDevices];
std::mutex g_mu;

template <int D>
cudaError_t prepare_kernel(int *occ)
{
    *occ = 1 << 30;
    cudaError_t e = prepare_one<D, false, -1>(occ);
    if (e == cudaSuccess) e = prepare_one<D, true, -1>(occ);
    if constexpr (D == 128) {
        if (e == cudaSuccess) e = prepare_one<D, false, 0>(occ);
        if (e == cudaSuccess) e = prepare_one<D, true, 0>(occ);
        if (e == cudaSuccess) e = prepare_one<D, false, 1>(occ);
        if (e == cudaSuccess) e = prepare_one<D, true, 1>(occ);
        if (e == cudaSuccess) e = prepare_one<D, false, 2>(occ);
        if (e == cudaSuccess) e = prepare_one<D, true, 2>(occ);
        if (e == cudaSuccess) e = prepare_one<D, false, 4>(occ);
        if (e == cudaSuccess) e = prepare_one<D, true, 4>(occ);
    }
    return e;
}


relay_status_t device_info(const DevInfo **out)
{
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return RELAY_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    DevInfo &d = g_dev[dev];
    if (!d.ready) {
        if (cudaDeviceGetAttribute(&d.sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
            prepare_kernel<64>(&d.occ64) != cudaSuccess || prepare_kernel<128>(&d.occ128) != cudaSuccess) {
            cudaGetLastError();
            return RELAY_ERR_CUDA;
        }
        if (d.occ64 < 1 || d.occ128 < 1) return RELAY_ERR_CUDA;
        if (cudaFuncSetAttribute(tc::sys_tc_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc::kSmemTC) != cudaSuccess ||
            cudaFuncSetAttribute(tc::sys_tc_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 tc::kSmemTC) != cudaSuccess) {
            cudaGetLastError();
            return RELAY_ERR_CUDA;
        }
        // the tensor-core kernel's warpgroups re-split the registers it is
        // launched with: never launch it with fewer than the split needs (the
        // raising warpgroups would wait for registers that never come)
        cudaFuncAttributes fa0{}, fa1{};
        if (cudaFuncGetAttributes(&fa0, tc::sys_tc_kernel<false>) != cudaSuccess ||
            cudaFuncGetAttributes(&fa1, tc::sys_tc_kernel<true>) != cudaSuccess) {
            cudaGetLastError();
            return RELAY_ERR_CUDA;
        }
        if (fa0.numRegs * tc::kThreadsTC < tc::kRegSplit || fa1.numRegs * tc::kThreadsTC < tc::kRegSplit)
            return RELAY_ERR_CUDA;
        d.ready = true;
    }
    *out = &d;
    return RELAY_OK;
}

// KV heads of the caches (0 in the dims means multi-head: H)
int kv_heads(const relay_dims_t *d) { return d->Hkv > 0 ? d->Hkv : d->H; }

relay_status_t check_dims(const relay_dims_t *d)
{
    if (!d) return RELAY_ERR_INVALID_ARG;
    if (d->B < 0 || d->Lq < 1 || d->H < 1 || d->D < 1 || d->Ls < 0 || d->block_size < 1 ||
        d->num_blocks < 0 || d->max_blocks_per_seq < 0 || d->max_q_total < 0 || d->ctx_split < 0 ||
        d->sys_range < 0 || !(d->scale == d->scale))
        return RELAY_ERR_INVALID_ARG;
    if (d->ctx_split % kTileK || d->sys_range % kTileK) return RELAY_ERR_INVALID_ARG;
    if (d->Hkv < 0 || (d->Hkv > 0 && d->H % d->Hkv != 0)) return RELAY_ERR_INVALID_ARG;
    if (d->D != 64 && d->D != 128) return RELAY_ERR_UNSUPPORTED;
    if (d->block_size != kBlock) return RELAY_ERR_UNSUPPORTED;
    if (d->B > kMaxB) return RELAY_ERR_UNSUPPORTED;
    // 32-bit item and row counters on the device
    if ((int64_t)d->B * d->Lq > INT_MAX / 2 || (int64_t)d->B * d->H > INT_MAX / 2 ||
        (int64_t)d->B * d->Lq * d->H > INT_MAX / 2 ||     // virtual rows of the system step
        (int64_t)d->max_blocks_per_seq * kBlock + d->Ls > INT_MAX / 2)
        return RELAY_ERR_UNSUPPORTED;
    return RELAY_OK;
}

int tc_pairs(int Mtot) { return ((Mtot + tc::kRowsTC - 1) / tc::kRowsTC + 1) / 2; }

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (the library links only the CUDA runtime).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder()
{
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *f = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
        cudaGetLastError();
    });
    return fn;
}

// sys_k or sys_v, [Ls][H][128] fp16, as a 3-D tensor (d, head, key) read in
// {64, 1, 128} boxes with 128-byte swizzle; keys past Ls read as zero.
bool encode_sys_map(CUtensorMap *m, const void *base, int H, int Ls)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)Ls};
    const cuuint64_t strides[2] = {128 * sizeof(__half), (cuuint64_t)H * 128 * sizeof(__half)};
    const cuuint32_t box[3] = {64, 1, (cuuint32_t)tc::kKeysTC};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Prefill output, [Ls][H][128] fp16, as a 3-D tensor (d, head, position)
// written in {64, G, 128 / G} boxes with 128-byte swizzle: one d-half of a
// 128-row tile of virtual rows (position t, head hk G + c: row t G + c), the
// box's rows in that order; rows past Ls are not written.
bool encode_out_map(CUtensorMap *m, void *base, int H, int Ls, int G)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc || G < 1 || tc::kRowsTC % G) return false;
    const cuuint64_t dims[3] = {128, (cuuint64_t)H, (cuuint64_t)Ls};
    const cuuint64_t strides[2] = {128 * sizeof(__half), (cuuint64_t)H * 128 * sizeof(__half)};
    const cuuint32_t box[3] = {64, (cuuint32_t)G, (cuuint32_t)(tc::kRowsTC / G)};
    const cuuint32_t estr[3] = {1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
               CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_NONE,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// The paged pool k_cache or v_cache, [num_blocks][Hkv][16][128] fp16, as a
// 4-D tensor (d, token, head, page) read in {64, 16, 1, 1} boxes (one d-half
// of one page of one head) with 128-byte swizzle; pages past num_blocks read
// as zero.
bool encode_pool_map(CUtensorMap *m, const void *base, int Hkv, int num_blocks)
{
    PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
    if (!enc) return false;
    const cuuint64_t dims[4] = {128, (cuuint64_t)kBlock, (cuuint64_t)Hkv, (cuuint64_t)num_blocks};
    const cuuint64_t strides[3] = {128 * sizeof(__half), (cuuint64_t)kBlock * 128 * sizeof(__half),
                                   (cuuint64_t)Hkv * kBlock * 128 * sizeof(__half)};
    const cuuint32_t box[4] = {64, (cuuint32_t)kBlock, 1, 1};
    const cuuint32_t estr[4] = {1, 1, 1, 1};
    return enc(m, CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 4, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Shared prefix segments of a call: the system prompt alone (one segment of
// dims->Ls tokens), or the levels of a tree of shared prefixes.
struct Segments {
    int n = 0;
    int len[kMaxSegments] = {};
    const void *k[kMaxSegments] = {}, *v[kMaxSegments] = {};
};

Segments one_segment(const relay_dims_t *d, const void *k, const void *v)
{
    Segments sg;
    sg.n = 1;
    sg.len[0] = d->Ls;
    sg.k[0] = k;
    sg.v[0] = v;
    return sg;
}

struct Plan {
    int Mtot = 0;
    int R_sys = 0, sys_range = kTileK, ctx_split = kAutoCtxSplit;
    int seg_R[kMaxSegments] = {}, seg_range[kMaxSegments] = {}, seg_part0[kMaxSegments] = {};
    int c_dec = 0, c_mq = 0, mq_split_min = 0, n_prefix = 0;
    int tps_min = 32, tps_max = 32;
    bool tc = false;          // system step on the tensor-core kernel
    bool ctx_tc = false;      // multi-row requests' own contexts on the tensor-core kernel too
    int ctx_pairs = 0;        // tile pairs of a request of Lq rows
    long long n_tc_sys = 0, n_tc_ctx = 0;   // CTAs of the tensor-core grid: system, then context
    size_t dec_base = 0, mq_base = 0, rows = 0;   // partial rows: [system | decode | multi-row] sections
    size_t off_sched = 0, off_part_o = 0, off_part_lse = 0, total = 0;
};

int round_up(int x, int m) { return (x + m - 1) / m * m; }

// Work-item sizes and workspace layout for one mode, for a GPU of `sms` SMs
// (one streaming CTA per SM; the number of system key ranges depends on it).
// `seg`: several shared prefix segments (never on the tensor-core kernel);
// null: the one system prompt of dims->Ls tokens.
Plan make_plan(const relay_dims_t *d, int mode, int sms, const Segments *seg = nullptr)
{
    Plan pl;
    pl.Mtot = d->max_q_total > 0 ? d->max_q_total : d->B * d->Lq;
    const bool sys = mode == MODE_FUSED || mode == MODE_SYS;
    const bool ctx = mode != MODE_SYS;
    pl.n_prefix = mode == MODE_BASELINE ? d->Ls : 0;
    const int G = d->H / kv_heads(d);            // query heads per KV head
    const long long Mv = (long long)pl.Mtot * G;   // rows of the system step per KV head
    pl.tc = !seg && sys && d->D == 128 && d->Ls > 0 && Mv > kTcMinRows;
    if (pl.tc) {
        // (head, tile pair, key range) items, one CTA each.  The number of
        // ranges R minimises the makespan in waves of one CTA per SM times
        // keys per range, ceil(n R / SMs) / R, among ranges of at least
        // 2048 keys (so the partials stay small); the smallest R within 2%
        // of the best wins.
        const long long n = (long long)tc_pairs((int)Mv) * kv_heads(d);
        const int r_cap = std::max(1, d->Ls / 2048);
        double best = 1e30;
        int r_best = 1;
        for (int r = 1; r <= r_cap; r++) {
            const double cost = (double)((n * r + sms - 1) / sms) / r;
            if (cost < best) best = cost;
        }
        for (int r = 1; r <= r_cap; r++) {
            if ((double)((n * r + sms - 1) / sms) / r <= best * 1.02) {
                r_best = r;
                break;
            }
        }
        int range = d->sys_range > 0 ? d->sys_range : round_up((d->Ls + r_best - 1) / r_best, tc::kKeysTC);
        pl.sys_range = range;
        pl.R_sys = (d->Ls + range - 1) / range;
        pl.seg_range[0] = range;
        pl.seg_R[0] = pl.R_sys;
        pl.n_tc_sys = n * pl.R_sys;
    } else if (sys) {
        const Segments one = one_segment(d, nullptr, nullptr);
        const Segments &sg = seg ? *seg : one;
        long long total = 0;
        for (int i = 0; i < sg.n; i++) total += sg.len[i];
        pl.R_sys = 0;
        for (int i = 0; i < sg.n; i++) {
            const int L = sg.len[i];
            int range = kTileK, R = 0;
            if (L > 0) {
                range = d->sys_range;
                if (range == 0) {
                    // Enough system items to spread over the GPU (segments
                    // share it by length), but long enough ranges that each
                    // range's partial results stay small next to the keys it
                    // streams.
                    const int tiles = (int)((Mv + kTileM - 1) / kTileM);
                    const int hkv = kv_heads(d);
                    const long long share = std::max<long long>(1, (long long)sms * L / std::max<long long>(1, total));
                    int r_want = (int)((share + (long long)hkv * tiles - 1) / ((long long)hkv * tiles));
                    // cap on the ranges from the query rows per head (not the
                    // virtual rows of a head group), so the items stay short
                    int r_cap = L / std::max(256, 16 * pl.Mtot);
                    int r = std::max(1, std::min(r_want, r_cap));
                    range = round_up((L + r - 1) / r, kTileK);
                }
                R = (L + range - 1) / range;
            } else if (mode == MODE_SYS && sg.n == 1) {
                R = 1;   // one empty range still reports lse = -inf for sys-only output
            }
            pl.seg_range[i] = range;
            pl.seg_R[i] = R;
            pl.seg_part0[i] = pl.R_sys;
            pl.R_sys += R;
        }
        pl.sys_range = pl.seg_range[0];
    }
    if (ctx) {
        // Context splits per request.  A decode request's pages (prefix
        // pages + context pages) go to items of tps pages, tps chosen on the
        // device in [tps_min, tps_max] (fixed when ctx_split is given);
        // tps_min keeps a request at <= kMaxCtxParts partials.  A multi-row
        // request uses splits of at least ctx_split keys, and at least
        // mq_split_min, so that it has at most kMaxMqParts of them.
        constexpr int kMaxCtxParts = 32;
        pl.ctx_split = d->ctx_split > 0 ? d->ctx_split : kAutoCtxSplit;
        const int max_pages = (pl.n_prefix + kBlock - 1) / kBlock + d->max_blocks_per_seq;
        pl.tps_max = std::min(pl.ctx_split / kBlock, 32);    // a decode item holds <= 32 pages
        pl.tps_min = d->ctx_split > 0 ? pl.tps_max
                                      : std::min(pl.tps_max, std::max(2, (max_pages + kMaxCtxParts - 1) / kMaxCtxParts));
        pl.c_dec = std::max(1, (max_pages + pl.tps_min - 1) / pl.tps_min);
        const long long max_keys = (long long)pl.n_prefix + (long long)d->max_blocks_per_seq * kBlock;
        pl.mq_split_min = (int)((max_keys + kMaxMqParts - 1) / kMaxMqParts);
        // Requests of at least kTcCtxMinRows virtual rows per KV head take
        // their own context on the tensor cores, one split over all of it,
        // in the same grid as the system step (after its CTAs).
        pl.ctx_tc = d->D == 128 && pl.n_prefix == 0 && d->Lq > 1 && (long long)d->Lq * G >= kTcCtxMinRows &&
                    d->num_blocks > 0 && d->max_blocks_per_seq > 0 && d->max_blocks_per_seq <= tc::kMaxPagesTC;
        if (pl.ctx_tc) {
            pl.mq_split_min = (int)max_keys;
            pl.ctx_pairs = tc_pairs(d->Lq * G);
            // items (request, tile pair): a request of q > 1 rows holds
            // ceil(q G / 256) < q G / 256 + 1 pairs, and at most
            // min(B, max_q_total / 2) requests have more than one row
            const long long n_mr = std::min<long long>(d->B, pl.Mtot / 2);
            const long long items =
                std::min((long long)d->B * pl.ctx_pairs, n_mr + ((long long)pl.Mtot * G + 255) / 256);
            pl.n_tc_ctx = items * kv_heads(d);
        }
        pl.mq_split_min = round_up(std::max(pl.mq_split_min, 1), pl.ctx_split);
        // multi-row requests exist only when a request may carry several rows
        pl.c_mq = d->Lq > 1 ? std::max(1, (int)((max_keys + pl.mq_split_min - 1) / pl.mq_split_min)) : 0;
        if (pl.ctx_tc) pl.c_mq = 1;
    }
    const size_t sys_rows = (size_t)(sys ? pl.R_sys : 0) * pl.Mtot * d->H;
    const size_t dec_rows = (size_t)(ctx ? pl.c_dec : 0) * d->B * d->H;
    const size_t mq_rows = (size_t)(ctx ? pl.c_mq : 0) * pl.Mtot * d->H;
    pl.dec_base = sys_rows;
    pl.mq_base = sys_rows + dec_rows;
    pl.rows = sys_rows + dec_rows + mq_rows;
    pl.off_sched = 256;
    size_t sched_bytes = ((size_t)(2 * d->B + 2) * sizeof(int) + 255) / 256 * 256;
    pl.off_part_o = pl.off_sched + sched_bytes;
    pl.off_part_lse = pl.off_part_o + (pl.rows * d->D * sizeof(float) + 255) / 256 * 256;
    pl.total = pl.off_part_lse + (pl.rows * sizeof(float) + 255) / 256 * 256;
    return pl;
}

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

float scale_log2_of(const relay_dims_t *d)
{
    float sc = d->scale > 0.f ? d->scale : 1.0f / std::sqrt((float)d->D);
    return sc * 1.4426950408889634f;
}

// Key groups of a system tile with `rows` virtual rows (the device's row_roles).
int key_groups(int rows)
{
    const int rg = (rows + 15) / 16;
    int np2 = 1;
    while (np2 < rg) np2 <<= 1;
    return std::min(kRowWarps / np2, kTileK / 8);
}

// The row-item class of a launch (the ROWS of relay_kernel), -1 unless the
// shape fixes it: every request has its Lq = 1 row (no q_lens), so there is
// no multi-row item, and every system tile has the same number of key groups.
int row_class(const relay_dims_t *d, const Plan &pl, int mode, int G, bool have_q_lens)
{
    if (d->D != 128) return -1;
    const bool sys_items = (mode == MODE_FUSED || mode == MODE_SYS) && !pl.tc && pl.R_sys > 0;
    // multi-row context items: requests of several rows whose contexts are
    // not on the tensor cores
    const bool mq_items = mode != MODE_SYS && d->Lq > 1 && !pl.ctx_tc;
    if (!sys_items && !mq_items) return 0;
    if (have_q_lens || d->Lq != 1) return -1;
    const int Mv = d->B * G;                          // virtual rows per KV head
    const int T = (Mv + kTileM - 1) / kTileM;
    const int kg_last = key_groups(Mv - (T - 1) * kTileM);
    if (T > 1 && kg_last != key_groups(kTileM)) return -1;
    return kg_last;
}

// Shared prefix segments from the caller's host arrays: 1..kMaxSegments
// segments of >= 0 tokens, [len, Hkv, D] fp16 each, 16-byte aligned.
relay_status_t make_segments(int n_seg, const void *const *k, const void *const *v, const int32_t *len,
                             Segments *out)
{
    if (n_seg < 1 || n_seg > kMaxSegments || !len) return RELAY_ERR_INVALID_ARG;
    long long total = 0;
    out->n = n_seg;
    for (int i = 0; i < n_seg; i++) {
        if (len[i] < 0) return RELAY_ERR_INVALID_ARG;
        total += len[i];
        out->len[i] = len[i];
        out->k[i] = k ? k[i] : nullptr;
        out->v[i] = v ? v[i] : nullptr;
        if (len[i] > 0 && (!out->k[i] || !out->v[i] || !aligned(out->k[i], 16) || !aligned(out->v[i], 16)))
            return RELAY_ERR_INVALID_ARG;
    }
    if (total > INT_MAX / 2) return RELAY_ERR_UNSUPPORTED;
    return RELAY_OK;
}

relay_status_t launch_relay(const relay_dims_t *d, int mode, Params p, void *ws, size_t ws_bytes,
                            relay_stream_t stream, const Segments *seg = nullptr)
{
    if (!ws) return RELAY_ERR_WORKSPACE;
    if (!aligned(ws, 256)) return RELAY_ERR_INVALID_ARG;
    // host checks first: a workspace too small for any device, and (without
    // q_lens every request has Lq rows, and the partial slots are laid out
    // for max_q_total rows) a bound below B * Lq; with q_lens the kernel
    // checks their sum on the device
    if (ws_bytes < make_plan(d, mode, 1, seg).total) return RELAY_ERR_WORKSPACE;
    if (!p.q_lens && (long long)d->B * d->Lq > make_plan(d, mode, 1, seg).Mtot) return RELAY_ERR_INVALID_ARG;
    const DevInfo *dev = nullptr;
    relay_status_t st = device_info(&dev);
    if (st != RELAY_OK) return st;
    Plan pl = make_plan(d, mode, dev->sms, seg);
    if (ws_bytes < pl.total) return RELAY_ERR_WORKSPACE;

    unsigned char *base = static_cast<unsigned char *>(ws);
    p.B = d->B;
    p.Lq = d->Lq;
    p.H = d->H;
    p.Hkv = kv_heads(d);
    p.G = d->H / p.Hkv;
    p.NG = (p.G + 7) / 8;
    p.HQ = p.G > 1 ? p.Hkv * p.NG : d->H;
    p.Ls = d->Ls;
    p.num_blocks = d->num_blocks;
    p.max_blocks = d->max_blocks_per_seq;
    p.max_q_total = pl.Mtot;
    p.scale_log2 = scale_log2_of(d);
    p.n_prefix = pl.n_prefix;
    p.ctrl = reinterpret_cast<unsigned *>(base);
    p.sched = reinterpret_cast<int *>(base + pl.off_sched);
    p.part_o = reinterpret_cast<float *>(base + pl.off_part_o);
    p.part_lse = reinterpret_cast<float *>(base + pl.off_part_lse);
    p.R_sys = pl.R_sys;
    p.sys_range = pl.sys_range;
    p.ctx_split = pl.ctx_split;
    p.tps_min = pl.tps_min;
    p.tps_max = pl.tps_max;
    p.c_dec = pl.c_dec;
    p.c_mq = pl.c_mq;
    p.mq_split_min = pl.mq_split_min;
    p.dec_base = (long long)pl.dec_base;
    p.mq_base = (long long)pl.mq_base;
    p.skip_sys = pl.tc ? 1 : 0;
    p.skip_mq = pl.ctx_tc ? 1 : 0;
    p.dec_static = (pl.n_tc_sys + pl.n_tc_ctx > 0 || d->B > 32) ? 0 : 3;
    p.mode = mode;
    {
        const Segments one = one_segment(d, p.sys_k, p.sys_v);
        const Segments &sg = seg ? *seg : one;
        p.n_seg = sg.n;
        for (int i = 0; i < sg.n; i++) {
            p.seg_k[i] = static_cast<const __half *>(sg.k[i]);
            p.seg_v[i] = static_cast<const __half *>(sg.v[i]);
            p.seg_len[i] = sg.len[i];
            p.seg_range[i] = pl.seg_range[i];
            p.seg_R[i] = pl.seg_R[i];
            p.seg_part0[i] = pl.seg_part0[i];
        }
    }

    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (pl.n_tc_sys + pl.n_tc_ctx > 0) {
        // tensor cores: system partials, one CTA per (range, head, tile
        // pair), then the multi-row requests' context partials, one CTA per
        // (request, tile pair, head)
        tc::TcParams t{};
        t.B = d->B;
        t.Lq = d->Lq;
        t.H = d->H;
        t.G = p.G;
        t.Hkv = p.Hkv;
        t.Ls = d->Ls;
        t.max_q_total = pl.Mtot;
        t.scale_log2 = p.scale_log2;
        t.q = p.q;
        t.q_lens = p.q_lens;
        t.flags = p.ctrl;
        t.part_o = p.part_o;
        t.part_lse = p.part_lse;
        t.R = pl.R_sys;
        t.range = pl.sys_range;
        t.pairs = tc_pairs(pl.Mtot * p.G);
        t.n_sys = (int)pl.n_tc_sys;
        t.ctx_pairs = pl.ctx_pairs;
        t.ctx_lens = mode == MODE_SYS ? nullptr : p.ctx_lens;
        t.block_tables = p.block_tables;
        t.max_blocks = d->max_blocks_per_seq;
        t.num_blocks = d->num_blocks;
        t.mq_base = (long long)pl.mq_base;
        t.queue = p.ctrl + CTRL_TC_QUEUE;
        CUtensorMap tmK{}, tmV{}, tmKc{}, tmVc{};
        if (pl.tc && (!encode_sys_map(&tmK, p.sys_k, p.Hkv, d->Ls) || !encode_sys_map(&tmV, p.sys_v, p.Hkv, d->Ls)))
            return RELAY_ERR_CUDA;
        if (pl.ctx_tc) {
            if (!p.k_cache || !p.v_cache || !p.block_tables || !p.ctx_lens) return RELAY_ERR_INVALID_ARG;
            if (!encode_pool_map(&tmKc, p.k_cache, p.Hkv, d->num_blocks) ||
                !encode_pool_map(&tmVc, p.v_cache, p.Hkv, d->num_blocks))
                return RELAY_ERR_CUDA;
        }
        // persistent: one CTA per SM at most
        const long long tc_grid = std::min<long long>(pl.n_tc_sys + pl.n_tc_ctx, dev->sms);
        t.n_yield = (dev->sms * kTcYieldPct + 50) / 100;
        t.sms = dev->sms;
        t.sys_stages = (float)pl.n_tc_sys * (float)((pl.sys_range + tc::kKeysTC - 1) / tc::kKeysTC);
        tc::sys_tc_kernel<false><<<(unsigned)tc_grid, tc::kThreadsTC, tc::kSmemTC, s>>>(tmK, tmV, tmKc, tmVc, t);
        if (cudaGetLastError() != cudaSuccess) return RELAY_ERR_CUDA;
    }
    {
        // the streaming kernel's instance for this shape
        void (*fn)(const Params) = nullptr;
        unsigned grid = 0;
        size_t smem = 0;
        const bool grp = p.G > 1;
        if (d->D == 128) {
            grid = dev->sms * dev->occ128;
            smem = sizeof(Smem<128>);
            switch (row_class(d, pl, mode, p.G, p.q_lens != nullptr)) {
            case 0: fn = grp ? relay_kernel<128, true, 0> : relay_kernel<128, false, 0>; break;
            case 1: fn = grp ? relay_kernel<128, true, 1> : relay_kernel<128, false, 1>; break;
            case 2: fn = grp ? relay_kernel<128, true, 2> : relay_kernel<128, false, 2>; break;
            case 4: fn = grp ? relay_kernel<128, true, 4> : relay_kernel<128, false, 4>; break;
            default: fn = grp ? relay_kernel<128, true, -1> : relay_kernel<128, false, -1>; break;
            }
        } else {
            grid = dev->sms * dev->occ64;
            smem = sizeof(Smem<64>);
            fn = grp ? relay_kernel<64, true, -1> : relay_kernel<64, false, -1>;
        }
        // behind the tensor-core grid, a programmatic dependent of it: it
        // starts on the SMs that grid's last wave frees
        cudaLaunchConfig_t cfg = {};
        cudaLaunchAttribute attr[1];
        cfg.gridDim = dim3(grid);
        cfg.blockDim = dim3(kThreads);
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        if (pl.n_tc_sys + pl.n_tc_ctx > 0) {
            attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
            attr[0].val.programmaticStreamSerializationAllowed = 1;
            cfg.attrs = attr;
            cfg.numAttrs = 1;
        }
        if (cudaLaunchKernelEx(&cfg, fn, p) != cudaSuccess) {
            cudaGetLastError();
            return RELAY_ERR_CUDA;
        }
    }

    // merge kernel: one warp per (row, head), launched as a programmatic
    // dependent so that its launch overlaps the first kernel's tail
    const long long warps = (long long)pl.Mtot * d->H;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)((warps + kWarps - 1) / kWarps));
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    // speculative partial-row loads only where the merge is latency-bound:
    // at most 1024 (row, head) pairs (the extra rows cost L2 bandwidth above)
    const bool spec = !p.q_lens && warps <= 1024;
    cudaError_t e;
    if (d->D == 128) e = spec ? cudaLaunchKernelEx(&cfg, merge_kernel<128, true>, p)
                              : cudaLaunchKernelEx(&cfg, merge_kernel<128, false>, p);
    else e = cudaLaunchKernelEx(&cfg, merge_kernel<64, false>, p);
    if (e != cudaSuccess) {
        cudaGetLastError();
        return RELAY_ERR_CUDA;
    }
    return RELAY_OK;
}

Params blank_params()
{
    Params p{};
    return p;
}

}  // namespace

extern "C" {

size_t relay_workspace_size(const relay_dims_t *dims)
{
    if (check_dims(dims) != RELAY_OK) return 0;
    // for the current device (its SM count sets the number of system key
    // ranges); without a usable device, for as many ranges as any device
    // would use (an unbounded SM count)
    const DevInfo *dev = nullptr;
    const int sms = device_info(&dev) == RELAY_OK ? dev->sms : INT_MAX / 4;
    size_t m = 0;
    for (int mode : {MODE_FUSED, MODE_SYS, MODE_CTX, MODE_BASELINE}) m = std::max(m, make_plan(dims, mode, sms).total);
    return m;
}

relay_status_t relay_workspace_init(void *ws, size_t ws_bytes, relay_stream_t stream)
{
    if (!ws || ws_bytes < 256) return RELAY_ERR_WORKSPACE;
    if (cudaMemsetAsync(ws, 0, ws_bytes, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return RELAY_ERR_CUDA;
    }
    return RELAY_OK;
}

relay_status_t relay_sys_attn(const relay_dims_t *dims, const void *q, const void *sys_k, const void *sys_v,
                              const int32_t *q_lens, float *o_sys, float *lse_sys, void *ws, size_t ws_bytes,
                              relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    if (!q || !o_sys || !lse_sys || (dims->Ls > 0 && (!sys_k || !sys_v))) return RELAY_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(sys_k, 16) || !aligned(sys_v, 16) || !aligned(o_sys, 16) ||
        !aligned(lse_sys, 4) || !aligned(q_lens, 4))
        return RELAY_ERR_INVALID_ARG;
    if (dims->B == 0) return RELAY_OK;
    Params p = blank_params();
    p.q = static_cast<const __half *>(q);
    p.sys_k = static_cast<const __half *>(sys_k);
    p.sys_v = static_cast<const __half *>(sys_v);
    p.q_lens = q_lens;
    p.o_f32 = o_sys;
    p.lse_f32 = lse_sys;
    return launch_relay(dims, MODE_SYS, p, ws, ws_bytes, stream);
}

relay_status_t relay_ctx_attn(const relay_dims_t *dims, const void *q, const void *k_cache, const void *v_cache,
                              const int32_t *block_tables, const int32_t *ctx_lens, const int32_t *q_lens,
                              float *o_ctx, float *lse_ctx, void *ws, size_t ws_bytes, relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    if (!q || !o_ctx || !lse_ctx || !ctx_lens || (dims->max_blocks_per_seq > 0 && !block_tables) ||
        (dims->num_blocks > 0 && (!k_cache || !v_cache)))
        return RELAY_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(o_ctx, 16) ||
        !aligned(lse_ctx, 4) || !aligned(block_tables, 4) || !aligned(ctx_lens, 4) || !aligned(q_lens, 4))
        return RELAY_ERR_INVALID_ARG;
    if (dims->B == 0) return RELAY_OK;
    Params p = blank_params();
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const __half *>(k_cache);
    p.v_cache = static_cast<const __half *>(v_cache);
    p.block_tables = block_tables;
    p.ctx_lens = ctx_lens;
    p.q_lens = q_lens;
    p.o_f32 = o_ctx;
    p.lse_f32 = lse_ctx;
    return launch_relay(dims, MODE_CTX, p, ws, ws_bytes, stream);
}

relay_status_t relay_fuse(const relay_dims_t *dims, const float *o_sys, const float *lse_sys, const float *o_ctx,
                          const float *lse_ctx, const int32_t *q_lens, void *out, float *lse_out,
                          relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    if (!o_sys || !lse_sys || !o_ctx || !lse_ctx || !out) return RELAY_ERR_INVALID_ARG;
    if (!aligned(o_sys, 16) || !aligned(o_ctx, 16) || !aligned(out, 16) || !aligned(lse_sys, 4) ||
        !aligned(lse_ctx, 4) || !aligned(lse_out, 4) || !aligned(q_lens, 4))
        return RELAY_ERR_INVALID_ARG;
    if (dims->B == 0) return RELAY_OK;
    const DevInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != RELAY_OK) return st;
    size_t n = (size_t)dims->B * dims->Lq * dims->H * (dims->D / 4);
    size_t blocks = (n + 255) / 256;
    size_t cap = (size_t)dev->sms * 8;
    int grid = (int)std::max<size_t>(1, std::min(blocks, cap));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    __half *o = static_cast<__half *>(out);
    if (dims->D == 128)
        fuse_kernel<128><<<grid, 256, 0, s>>>(dims->B, dims->Lq, dims->H, o_sys, lse_sys, o_ctx, lse_ctx, q_lens, o,
                                              lse_out);
    else
        fuse_kernel<64><<<grid, 256, 0, s>>>(dims->B, dims->Lq, dims->H, o_sys, lse_sys, o_ctx, lse_ctx, q_lens, o,
                                             lse_out);
    if (cudaGetLastError() != cudaSuccess) return RELAY_ERR_CUDA;
    return RELAY_OK;
}

relay_status_t relay_fuse_n(const relay_dims_t *dims, int K, const float *const *o_parts,
                            const float *const *lse_parts, const int32_t *q_lens, void *out, float *lse_out,
                            relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    if (K < 1 || K > kMaxFuseParts || !o_parts || !lse_parts || !out) return RELAY_ERR_INVALID_ARG;
    FuseN f{};
    for (int k = 0; k < K; k++) {
        if (!o_parts[k] || !lse_parts[k] || !aligned(o_parts[k], 16) || !aligned(lse_parts[k], 4))
            return RELAY_ERR_INVALID_ARG;
        f.o[k] = o_parts[k];
        f.lse[k] = lse_parts[k];
    }
    if (!aligned(out, 16) || !aligned(lse_out, 4) || !aligned(q_lens, 4)) return RELAY_ERR_INVALID_ARG;
    if (dims->B == 0) return RELAY_OK;
    const DevInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != RELAY_OK) return st;
    f.B = dims->B;
    f.Lq = dims->Lq;
    f.H = dims->H;
    f.K = K;
    f.q_lens = q_lens;
    f.out = static_cast<__half *>(out);
    f.lse_out = lse_out;
    const size_t n = (size_t)dims->B * dims->Lq * dims->H * (dims->D / 4);
    const int grid = (int)std::max<size_t>(1, std::min((n + 255) / 256, (size_t)dev->sms * 8));
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    if (dims->D == 128)
        fuse_n_kernel<128><<<grid, 256, 0, s>>>(f);
    else
        fuse_n_kernel<64><<<grid, 256, 0, s>>>(f);
    return cudaGetLastError() == cudaSuccess ? RELAY_OK : RELAY_ERR_CUDA;
}

relay_status_t relay_attention_decode(const relay_dims_t *dims, const void *q, const void *sys_k, const void *sys_v,
                                      const void *k_cache, const void *v_cache, const int32_t *block_tables,
                                      const int32_t *ctx_lens, const int32_t *q_lens, void *out, float *lse_out,
                                      void *ws, size_t ws_bytes, relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    if (!q || !out || !ctx_lens || (dims->Ls > 0 && (!sys_k || !sys_v)) ||
        (dims->max_blocks_per_seq > 0 && !block_tables) || (dims->num_blocks > 0 && (!k_cache || !v_cache)))
        return RELAY_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(sys_k, 16) || !aligned(sys_v, 16) || !aligned(k_cache, 16) ||
        !aligned(v_cache, 16) || !aligned(out, 16) || !aligned(lse_out, 4) || !aligned(block_tables, 4) ||
        !aligned(ctx_lens, 4) || !aligned(q_lens, 4))
        return RELAY_ERR_INVALID_ARG;
    if (dims->B == 0) return RELAY_OK;
    Params p = blank_params();
    p.q = static_cast<const __half *>(q);
    p.sys_k = static_cast<const __half *>(sys_k);
    p.sys_v = static_cast<const __half *>(sys_v);
    p.k_cache = static_cast<const __half *>(k_cache);
    p.v_cache = static_cast<const __half *>(v_cache);
    p.block_tables = block_tables;
    p.ctx_lens = ctx_lens;
    p.q_lens = q_lens;
    p.out = static_cast<__half *>(out);
    p.lse_out = lse_out;
    return launch_relay(dims, MODE_FUSED, p, ws, ws_bytes, stream);
}

size_t relay_workspace_size_prefixes(const relay_dims_t *dims, int n_seg, const int32_t *seg_len)
{
    if (check_dims(dims) != RELAY_OK) return 0;
    Segments sg;
    if (n_seg < 1 || n_seg > kMaxSegments || !seg_len) return 0;
    for (int i = 0; i < n_seg; i++) {
        if (seg_len[i] < 0) return 0;
        sg.len[i] = seg_len[i];
    }
    sg.n = n_seg;
    const DevInfo *dev = nullptr;
    const int sms = device_info(&dev) == RELAY_OK ? dev->sms : INT_MAX / 4;
    return make_plan(dims, MODE_FUSED, sms, &sg).total;
}

relay_status_t relay_attention_decode_prefixes(const relay_dims_t *dims, const void *q, int n_seg,
                                               const void *const *seg_k, const void *const *seg_v,
                                               const int32_t *seg_len, const uint32_t *seg_mask,
                                               const void *k_cache, const void *v_cache,
                                               const int32_t *block_tables, const int32_t *ctx_lens,
                                               const int32_t *q_lens, void *out, float *lse_out, void *ws,
                                               size_t ws_bytes, relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    Segments sg;
    st = make_segments(n_seg, seg_k, seg_v, seg_len, &sg);
    if (st != RELAY_OK) return st;
    if (!q || !out || !ctx_lens || (dims->max_blocks_per_seq > 0 && !block_tables) ||
        (dims->num_blocks > 0 && (!k_cache || !v_cache)))
        return RELAY_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(out, 16) ||
        !aligned(lse_out, 4) || !aligned(block_tables, 4) || !aligned(ctx_lens, 4) || !aligned(q_lens, 4) ||
        !aligned(seg_mask, 4))
        return RELAY_ERR_INVALID_ARG;
    if (dims->B == 0) return RELAY_OK;
    Params p = blank_params();
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const __half *>(k_cache);
    p.v_cache = static_cast<const __half *>(v_cache);
    p.block_tables = block_tables;
    p.ctx_lens = ctx_lens;
    p.q_lens = q_lens;
    p.seg_mask = seg_mask;
    p.out = static_cast<__half *>(out);
    p.lse_out = lse_out;
    return launch_relay(dims, MODE_FUSED, p, ws, ws_bytes, stream, &sg);
}

relay_status_t relay_baseline_decode(const relay_dims_t *dims, const void *q, const void *k_pool, const void *v_pool,
                                     const int32_t *sys_block_ids, const int32_t *block_tables,
                                     const int32_t *ctx_lens, const int32_t *q_lens, void *out, float *lse_out,
                                     void *ws, size_t ws_bytes, relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    if (!q || !out || !ctx_lens || (dims->Ls > 0 && !sys_block_ids) ||
        (dims->max_blocks_per_seq > 0 && !block_tables) || (dims->num_blocks > 0 && (!k_pool || !v_pool)))
        return RELAY_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_pool, 16) || !aligned(v_pool, 16) || !aligned(out, 16) ||
        !aligned(lse_out, 4) || !aligned(block_tables, 4) || !aligned(ctx_lens, 4) || !aligned(q_lens, 4) ||
        !aligned(sys_block_ids, 4))
        return RELAY_ERR_INVALID_ARG;
    if (dims->B == 0) return RELAY_OK;
    Params p = blank_params();
    p.q = static_cast<const __half *>(q);
    p.k_cache = static_cast<const __half *>(k_pool);
    p.v_cache = static_cast<const __half *>(v_pool);
    p.block_tables = block_tables;
    p.ctx_lens = ctx_lens;
    p.q_lens = q_lens;
    p.prefix_ids = sys_block_ids;
    p.out = static_cast<__half *>(out);
    p.lse_out = lse_out;
    return launch_relay(dims, MODE_BASELINE, p, ws, ws_bytes, stream);
}

relay_status_t relay_kv_append(const relay_dims_t *dims, const void *k_new, const void *v_new,
                               const int32_t *block_tables, const int32_t *ctx_lens, const int32_t *q_lens,
                               void *k_cache, void *v_cache, void *ws, size_t ws_bytes, relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    if (!ws || ws_bytes < 256) return RELAY_ERR_WORKSPACE;
    if (dims->B == 0) return RELAY_OK;
    if (!k_new || !v_new || !block_tables || !ctx_lens || !k_cache || !v_cache || dims->max_blocks_per_seq < 1)
        return RELAY_ERR_INVALID_ARG;
    if (!aligned(k_new, 16) || !aligned(v_new, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
        !aligned(block_tables, 4) || !aligned(ctx_lens, 4) || !aligned(q_lens, 4) || !aligned(ws, 256))
        return RELAY_ERR_INVALID_ARG;
    KvAppend a{};
    a.B = dims->B;
    a.Lq = dims->Lq;
    a.Hkv = kv_heads(dims);
    a.D = dims->D;
    a.num_blocks = dims->num_blocks;
    a.max_blocks = dims->max_blocks_per_seq;
    a.k_new = static_cast<const __half *>(k_new);
    a.v_new = static_cast<const __half *>(v_new);
    a.block_tables = block_tables;
    a.ctx_lens = ctx_lens;
    a.q_lens = q_lens;
    a.k_cache = static_cast<__half *>(k_cache);
    a.v_cache = static_cast<__half *>(v_cache);
    a.flags = static_cast<unsigned *>(ws) + CTRL_FLAGS;
    const long long warps = (long long)a.B * a.Lq * a.Hkv;
    kv_append_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? RELAY_OK : RELAY_ERR_CUDA;
}

relay_status_t relay_sys_prefill(const relay_dims_t *dims, const void *q_sys, const void *sys_k, const void *sys_v,
                                 void *out, float *lse_out, void *ws, size_t ws_bytes, relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    if (!ws || ws_bytes < 256) return RELAY_ERR_WORKSPACE;
    if (dims->Ls == 0) return RELAY_OK;
    if (dims->D != 128) return RELAY_ERR_UNSUPPORTED;
    if ((int64_t)dims->Ls * dims->H > INT_MAX / 2) return RELAY_ERR_UNSUPPORTED;
    if (!q_sys || !sys_k || !sys_v || !out) return RELAY_ERR_INVALID_ARG;
    if (!aligned(q_sys, 16) || !aligned(sys_k, 16) || !aligned(sys_v, 16) || !aligned(out, 16) ||
        !aligned(lse_out, 4) || !aligned(ws, 256))
        return RELAY_ERR_INVALID_ARG;
    const DevInfo *dev = nullptr;
    st = device_info(&dev);
    if (st != RELAY_OK) return st;
    tc::TcParams t{};
    t.B = 1;
    t.Lq = dims->Ls;
    t.H = dims->H;
    t.Ls = dims->Ls;
    t.max_q_total = dims->Ls;
    t.scale_log2 = scale_log2_of(dims);
    t.q = static_cast<const __half *>(q_sys);
    t.flags = static_cast<unsigned *>(ws);
    t.R = 1;
    t.range = dims->Ls;
    t.Hkv = kv_heads(dims);
    t.G = dims->H / t.Hkv;
    t.pairs = tc_pairs(dims->Ls * t.G);
    t.out = static_cast<__half *>(out);
    t.lse_out = lse_out;
    CUtensorMap tmK, tmV;
    if (!encode_sys_map(&tmK, sys_k, t.Hkv, dims->Ls) || !encode_sys_map(&tmV, sys_v, t.Hkv, dims->Ls))
        return RELAY_ERR_CUDA;
    // the output tile goes out through a TMA store where a group's heads fit
    // a tile evenly (else each thread stores its own row)
    CUtensorMap tmO = tmK;
    t.out_tma = (tc::kRowsTC % t.G == 0 && encode_out_map(&tmO, out, dims->H, dims->Ls, t.G)) ? 1 : 0;
    const long long grid = std::min<long long>((long long)t.pairs * t.Hkv, dev->sms);
    tc::sys_tc_kernel<true><<<(unsigned)grid, tc::kThreadsTC, tc::kSmemTC, reinterpret_cast<cudaStream_t>(stream)>>>(
        tmK, tmV, tmO, tmV, t);
    return cudaGetLastError() == cudaSuccess ? RELAY_OK : RELAY_ERR_CUDA;
}

relay_status_t relay_rope(const relay_dims_t *dims, void *q, void *k_new, const int32_t *ctx_lens,
                          const int32_t *q_lens, float base, void *ws, size_t ws_bytes, relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    if (!ws || ws_bytes < 256) return RELAY_ERR_WORKSPACE;
    if (!(base > 1.f) || !(base < 1e30f)) return RELAY_ERR_INVALID_ARG;
    if (dims->B == 0) return RELAY_OK;
    if (!q || !ctx_lens) return RELAY_ERR_INVALID_ARG;
    if (!aligned(q, 16) || !aligned(k_new, 16) || !aligned(ctx_lens, 4) || !aligned(q_lens, 4) || !aligned(ws, 256))
        return RELAY_ERR_INVALID_ARG;
    Rope a{};
    a.B = dims->B;
    a.Lq = dims->Lq;
    a.H = dims->H;
    a.Hkv = kv_heads(dims);
    a.D = dims->D;
    a.Ls = dims->Ls;
    if (dims->D / 2 > kMaxRopePairs) return RELAY_ERR_UNSUPPORTED;
    for (int j = 0; j < dims->D / 2; j++) a.inv_freq[j] = std::pow((double)base, -2.0 * j / dims->D);
    a.q = static_cast<__half *>(q);
    a.k = static_cast<__half *>(k_new);
    a.ctx_lens = ctx_lens;
    a.q_lens = q_lens;
    a.flags = static_cast<unsigned *>(ws) + CTRL_FLAGS;
    const long long warps = (long long)a.B * a.Lq * (a.H + (k_new ? a.Hkv : 0));
    rope_kernel<<<(unsigned)((warps + 7) / 8), 256, 0, reinterpret_cast<cudaStream_t>(stream)>>>(a);
    return cudaGetLastError() == cudaSuccess ? RELAY_OK : RELAY_ERR_CUDA;
}

// ----------------------------------------------------------------------------- allocation-free variant
// Scratch for relay_attention_decode_noalloc: one fixed buffer per device,
// part of the module image, never allocated or freed at run time.
static __device__ __align__(256) unsigned char g_noalloc_scratch[RELAY_NOALLOC_SCRATCH_BYTES];

}  // extern "C"

namespace {

// Device address of the scratch buffer on the current device.  The symbol's
// name is only a host-side stand-in: its device address is looked up once
// per device, with that device current, and cached.
relay_status_t noalloc_scratch(void **ws)
{
    static void *scratch[kMaxDevices] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) {
        cudaGetLastError();
        return RELAY_ERR_CUDA;
    }
    std::lock_guard<std::mutex> lk(g_mu);
    if (!scratch[dev]) {
        void *ptr = nullptr;
        if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || !ptr) {
            cudaGetLastError();
            return RELAY_ERR_CUDA;
        }
        scratch[dev] = ptr;
    }
    *ws = scratch[dev];
    return RELAY_OK;
}

}  // namespace

extern "C" {

relay_status_t relay_attention_decode_noalloc(const relay_dims_t *dims, const void *q, const void *sys_k,
                                              const void *sys_v, const void *k_cache, const void *v_cache,
                                              const int32_t *block_tables, const int32_t *ctx_lens,
                                              const int32_t *q_lens, void *out, float *lse_out,
                                              relay_stream_t stream)
{
    relay_status_t st = check_dims(dims);
    if (st != RELAY_OK) return st;
    const size_t need = relay_workspace_size(dims);
    if (need == 0 || need > RELAY_NOALLOC_SCRATCH_BYTES) return RELAY_ERR_WORKSPACE;
    if (dims->B == 0) return RELAY_OK;
    void *ws = nullptr;
    st = noalloc_scratch(&ws);
    if (st != RELAY_OK) return st;
    // the queue counters must start at zero; the rest is overwritten
    if (cudaMemsetAsync(ws, 0, 256, reinterpret_cast<cudaStream_t>(stream)) != cudaSuccess) {
        cudaGetLastError();
        return RELAY_ERR_CUDA;
    }
    return relay_attention_decode(dims, q, sys_k, sys_v, k_cache, v_cache, block_tables, ctx_lens, q_lens, out,
                                  lse_out, ws, RELAY_NOALLOC_SCRATCH_BYTES, stream);
}

relay_status_t relay_device_status(void *ws, uint32_t *flags_out, relay_stream_t stream)
{
    if (!ws) return RELAY_ERR_WORKSPACE;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    uint32_t flags = 0;
    if (cudaMemcpyAsync(&flags, ws, sizeof(flags), cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemsetAsync(ws, 0, sizeof(flags), s) != cudaSuccess || cudaStreamSynchronize(s) != cudaSuccess) {
        cudaGetLastError();
        return RELAY_ERR_CUDA;
    }
    if (flags_out) *flags_out = flags;
    return flags ? RELAY_ERR_DEVICE_CHECK : RELAY_OK;
}

relay_status_t relay_noalloc_device_status(uint32_t *flags_out, relay_stream_t stream)
{
    void *ws = nullptr;
    relay_status_t st = noalloc_scratch(&ws);
    if (st != RELAY_OK) return st;
    return relay_device_status(ws, flags_out, stream);
}

const char *relay_status_string(relay_status_t status)
{
    switch (status) {
    case RELAY_OK: return "ok";
    case RELAY_ERR_INVALID_ARG: return "invalid argument";
    case RELAY_ERR_UNSUPPORTED: return "unsupported shape or parameter";
    case RELAY_ERR_WORKSPACE: return "workspace missing or too small";
    case RELAY_ERR_CUDA: return "CUDA runtime error";
    case RELAY_ERR_DEVICE_CHECK: return "device-side check failed";
    case RELAY_ERR_TIMEOUT: return "bounded device wait timed out";
    }
    return "unknown status";
}

}  // extern "C"
