// System-attention step on the 5th-generation tensor cores (tcgen05 + TMEM),
// for batches with many query rows per head, where the step is a dense,
// compute-bound contraction (atyun.com RelayAttention article, section
// "RelayAttention": the per-request matrix-vector products over the shared
// system prompt grouped into one matrix-matrix product).
//
// One CTA of 128 threads per item (head h, 128-row tile of the batch's query
// rows, range of system keys).  Query row t of the tile lives in TMEM lane t
// and is owned by thread t, so the online softmax needs no cross-thread
// reduction.  Per 64-key tile:
//   S[128 x 64]  = Q K^T    tcgen05.mma kind::f16, M=128 N=64  (TMEM, fp32)
//   P            = exp2(S - m) in fp16, written to shared memory by its row's
//                  thread in the K-major layout the next MMA reads
//   O[128 x 128] += P V     tcgen05.mma kind::f16, M=128 N=128 (TMEM, fp32)
// O is rescaled only when a row's running maximum grows by more than 2^8
// (P <= 256 otherwise, well inside fp16).  Operands sit in shared memory in
// the 128-byte-swizzled K-major layout (rows of 128 B, 16-byte chunks XOR-ed
// with row % 8, 8-row groups 1024 B apart); V tiles are transposed to K-major
// by the threads on the way.  One thread issues the MMAs; completion reaches
// the others through mbarriers, whose waits are bounded.  The item writes one
// fp32 partial per row (normalised output and log2-sum-exp), merged later
// with the context partials.
#pragma once

#include <cuda_fp16.h>
#include <stdint.h>

namespace relay {

namespace tc {

constexpr int kThreadsTC = 128;
constexpr int kRowsTC = 128;          // query rows per item (TMEM lanes)
constexpr int kKeysTC = 64;           // keys per tile
constexpr int kStagesTC = 3;          // K / V load ring
constexpr unsigned kWaitLimit = 1u << 26;

// shared-memory map (byte offsets from a 1024-aligned base), D = 128
constexpr int kQBytes = kRowsTC * 128 * 2 / 2 * 2;          // two d-halves of [128][64] fp16 = 32 KB
constexpr int kKHalf = kKeysTC * 128;                       // one d-half of a K tile: [64][64] fp16 = 8 KB
constexpr int kKBytes = 2 * kKHalf;                         // 16 KB
constexpr int kVRawBytes = kKeysTC * 128 * 2;               // [64 keys][128 d] plain = 16 KB
constexpr int kVtBytes = 128 * kKeysTC * 2;                 // [128 d][64 keys] swizzled = 16 KB
constexpr int kPBytes = kRowsTC * kKeysTC * 2;              // [128 rows][64 keys] swizzled = 16 KB
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + kQBytes;
constexpr int kOffVRaw = kOffK + kStagesTC * kKBytes;
constexpr int kOffVt = kOffVRaw + kStagesTC * kVRawBytes;
constexpr int kOffP = kOffVt + 2 * kVtBytes;
constexpr int kOffBar = kOffP + 2 * kPBytes;               // mbarriers: S, O[0], O[1]; then TMEM base
constexpr int kSmemTC = kOffBar + 64 + 1024;                // + alignment slack
constexpr int kTmemCols = 256;                              // S: 64 columns, O: 128 columns

// --------------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

// Wait for completion `parity` of an mbarrier; false if the wait gave up.
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity)
{
    for (unsigned it = 0; it < kWaitLimit; it++) {
        unsigned ok;
        asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                     " selp.u32 %0, 1, 0, p;\n}\n"
                     : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
        if (ok) return true;
    }
    return false;
}

__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// Shared-memory matrix descriptor: K-major, 128-byte swizzle, 8-row groups
// 1024 B apart (stride byte offset), descriptor version 1.
__device__ __forceinline__ uint64_t sw128_desc(unsigned saddr)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);            // start address
    d |= (uint64_t)(16u >> 4) << 16;                      // leading byte offset (unused for this layout)
    d |= (uint64_t)(1024u >> 4) << 32;                    // stride byte offset
    d |= (uint64_t)1 << 46;                               // version
    d |= (uint64_t)2 << 61;                               // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 accumulator, both
// operands K-major, shape M x N.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N)
{
    return (1u << 4)                          // D: fp32
         | (0u << 7) | (0u << 10)             // A, B: fp16
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

__device__ __forceinline__ void umma_f16(unsigned tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, int acc)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void umma_commit(unsigned bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}

// 32 consecutive fp32 columns of this thread's TMEM lane.
__device__ __forceinline__ void tmem_ld32(unsigned taddr, float (&v)[32])
{
    unsigned r[32];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 32; i++) v[i] = __uint_as_float(r[i]);
}

__device__ __forceinline__ void tmem_st32(unsigned taddr, const float (&v)[32])
{
    unsigned r[32];
#pragma unroll
    for (int i = 0; i < 32; i++) r[i] = __float_as_uint(v[i]);
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                   "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
                   "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
                   "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

// byte offset of element chunk `c` (8 fp16) of row `r` in a swizzled [rows][64] region
__device__ __forceinline__ unsigned sw_off(int r, int c) { return (unsigned)(r * 128 + ((c ^ (r & 7)) << 4)); }

struct TcParams {
    int B, Lq, H, Ls, max_q_total;
    float scale_log2;
    const __half *q, *sys_k, *sys_v;
    const int *q_lens;
    unsigned *flags;
    float *part_o, *part_lse;        // partial slots: [part][max_q_total][H][128]
    int R, range;                    // key ranges of the system prompt
};

// Stage keys [key0, key0 + 64) of head h: K into the swizzled K-major layout
// (two d-halves), V plainly; keys at or beyond key_hi are zero-filled.
__device__ __forceinline__ void tc_load_kv(const TcParams &p, unsigned sK, unsigned sV, int h, int key0, int key_hi)
{
    const int tid = threadIdx.x;
#pragma unroll
    for (int i = 0; i < (kKeysTC * 16) / kThreadsTC; i++) {
        const int cid = tid + i * kThreadsTC;
        const int key = cid >> 4, c = cid & 15;
        const int t = key0 + key;
        const bool valid = t < key_hi;
        const size_t off = ((size_t)(valid ? t : 0) * p.H + h) * 128 + c * 8;
        const unsigned dk = sK + (c >> 3) * kKHalf + sw_off(key, c & 7);
        const unsigned dv = sV + key * 256 + c * 16;
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dk), "l"(p.sys_k + off), "r"(valid ? 16 : 0));
        asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dv), "l"(p.sys_v + off), "r"(valid ? 16 : 0));
    }
}

__device__ __forceinline__ int owner_of(const int *qo, int n, int x)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (qo[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}

// One item per CTA: blockIdx.x = (range * tiles + tile) * H + h.
__global__ void __launch_bounds__(kThreadsTC, 1) sys_tc_kernel(const TcParams p)
{
    extern __shared__ unsigned char smem_raw[];
    __shared__ int qo[513];
    __shared__ unsigned tmem_base_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned sbase = (static_cast<unsigned>(__cvta_generic_to_shared(smem_raw)) + 1023u) & ~1023u;
    const unsigned sQ = sbase + kOffQ, sK0 = sbase + kOffK, sV0 = sbase + kOffVRaw;
    const unsigned sVt0 = sbase + kOffVt, sP0 = sbase + kOffP;
    const unsigned barS = sbase + kOffBar, barO0 = barS + 8;
    unsigned char *gbase = smem_raw + (sbase - static_cast<unsigned>(__cvta_generic_to_shared(smem_raw)));

    // rows of the batch: prefix of q_lens (B <= 512)
    if (p.q_lens) {
        if (tid == 0) {
            int acc = 0;
            for (int b = 0; b < p.B; b++) { qo[b] = acc; acc += p.q_lens[b]; }
            qo[p.B] = acc;
        }
    } else {
        for (int b = tid; b <= p.B; b += kThreadsTC) qo[b] = b * p.Lq;
    }
    if (tid == 0) abort_sh = 0;
    __syncthreads();
    const int Mtot = min(qo[p.B], p.max_q_total);
    const int T = (Mtot + kRowsTC - 1) / kRowsTC;
    const int h = blockIdx.x % p.H;
    const int tau = (blockIdx.x / p.H) % max(T, 1);
    const int rho = blockIdx.x / (p.H * max(T, 1));
    if (T == 0 || rho >= p.R) return;               // the whole CTA leaves together
    const int key0 = rho * p.range;
    const int key_hi = min(key0 + p.range, p.Ls);
    const int n_tiles = key_hi > key0 ? (key_hi - key0 + kKeysTC - 1) / kKeysTC : 0;

    // TMEM: warp 0 allocates 256 columns (S at +0, O at +64)
    if (warp == 0) {
        const unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(&tmem_base_sh));
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst), "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    if (tid == 0) {
        mbar_init(barS, 1);
        mbar_init(barO0, 1);
        mbar_init(barO0 + 8, 1);
        asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const unsigned tmem = tmem_base_sh;
    const unsigned tS = tmem, tO = tmem + 64;
    const unsigned lane_off = (unsigned)(warp * 32) << 16;

    // Q tile: row t of this item is query row tau*128 + t of the batch
    const int r = tau * kRowsTC + tid;
    const bool row_ok = r < Mtot;
    {
        const __half *qrow = p.q;
        if (row_ok) {
            const int b = owner_of(qo, p.B, r);
            qrow = p.q + (((size_t)b * p.Lq + (r - qo[b])) * p.H + h) * 128;
        }
#pragma unroll
        for (int c = 0; c < 16; c++) {
            const unsigned dq = sQ + (c >> 3) * (kRowsTC * 128) + sw_off(tid, c & 7);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dq), "l"(qrow + c * 8),
                         "r"(row_ok ? 16 : 0));
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    }
    // K/V prologue
#pragma unroll
    for (int j = 0; j < kStagesTC - 1; j++) {
        if (j < n_tiles) tc_load_kv(p, sK0 + j * kKBytes, sV0 + j * kVRawBytes, h, key0 + j * kKeysTC, key_hi);
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    }

    const uint32_t idS = idesc_f16(kRowsTC, kKeysTC), idO = idesc_f16(kRowsTC, 128);
    float m_run = kNegInf, l_run = 0.f;
    // a wait that gives up sets abort_sh; every thread reads it after the next
    // barrier, so the CTA leaves the loop together
    auto wait_or_abort = [&](unsigned bar, unsigned parity) {
        if (!mbar_wait(bar, parity)) abort_sh = 1;
    };
    int done_tiles = 0;
    for (int j = 0; j < n_tiles; j++) {
        const int st = j % kStagesTC;
        const int pb = j & 1;
        // P[pb] and Vt[pb] are free once PV(j-2) is done
        if (j >= 2) wait_or_abort(barO0 + 8 * pb, ((j - 2) >> 1) & 1);
        asm volatile("cp.async.wait_group %0;\n" ::"n"(kStagesTC - 2) : "memory");
        __syncthreads();
        if (abort_sh) break;
        // next tile's loads go into the stage read by tile j-1 (its MMAs are done)
        {
            const int jn = j + kStagesTC - 1;
            if (jn < n_tiles)
                tc_load_kv(p, sK0 + (jn % kStagesTC) * kKBytes, sV0 + (jn % kStagesTC) * kVRawBytes, h,
                           key0 + jn * kKeysTC, key_hi);
            asm volatile("cp.async.commit_group;\n" ::: "memory");
        }
        // transpose V: thread tid builds row d = tid of Vt (64 keys, K-major)
        {
            const unsigned char *vr = gbase + kOffVRaw + st * kVRawBytes;
            unsigned char *vt = gbase + kOffVt + pb * kVtBytes;
#pragma unroll
            for (int kc = 0; kc < 8; kc++) {
                unsigned short e[8];
#pragma unroll
                for (int k = 0; k < 8; k++)
                    e[k] = *reinterpret_cast<const unsigned short *>(vr + (kc * 8 + k) * 256 + tid * 2);
                uint4 w;
                w.x = e[0] | ((unsigned)e[1] << 16);
                w.y = e[2] | ((unsigned)e[3] << 16);
                w.z = e[4] | ((unsigned)e[5] << 16);
                w.w = e[6] | ((unsigned)e[7] << 16);
                *reinterpret_cast<uint4 *>(vt + sw_off(tid, kc)) = w;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (tid == 0) {
            const unsigned kb = sK0 + st * kKBytes;
#pragma unroll
            for (int kk = 0; kk < 8; kk++) {
                const uint64_t ad = sw128_desc(sQ + (kk >> 2) * (kRowsTC * 128) + (kk & 3) * 32);
                const uint64_t bd = sw128_desc(kb + (kk >> 2) * kKHalf + (kk & 3) * 32);
                umma_f16(tS, ad, bd, idS, kk > 0);
            }
            umma_commit(barS);
        }
        wait_or_abort(barS, j & 1);
        tc_fence_after();
        // softmax over this row's 64 scores
        float s[64];
        {
            float a[32], c[32];
            tmem_ld32(tS + lane_off, a);
            tmem_ld32(tS + lane_off + 32, c);
#pragma unroll
            for (int i = 0; i < 32; i++) { s[i] = a[i]; s[32 + i] = c[i]; }
        }
        float mt = kNegInf;
        const int kbase = key0 + j * kKeysTC;
#pragma unroll
        for (int i = 0; i < 64; i++) {
            s[i] = (kbase + i < key_hi) ? s[i] * p.scale_log2 : kNegInf;
            mt = fmaxf(mt, s[i]);
        }
        // lazy rescale: only when this row's max grows by more than 8 (log2)
        const bool grow = mt > m_run + 8.f || (m_run == kNegInf && mt != kNegInf);
        if (__any_sync(0xffffffffu, grow)) {
            // O may still be accumulating PV(j-1): wait for it before touching O
            if (j >= 1) wait_or_abort(barO0 + 8 * ((j - 1) & 1), ((j - 1) >> 1) & 1);
            tc_fence_after();
            const float mn = grow ? mt : m_run;
            const float alpha = (m_run == kNegInf) ? 0.f : ex2(m_run - mn);
            if (j >= 1) {
#pragma unroll
                for (int q4 = 0; q4 < 4; q4++) {
                    float o[32];
                    tmem_ld32(tO + lane_off + q4 * 32, o);
#pragma unroll
                    for (int i = 0; i < 32; i++) o[i] *= alpha;
                    tmem_st32(tO + lane_off + q4 * 32, o);
                }
            }
            l_run *= alpha;
            m_run = mn;
        }
        const float mu = (m_run == kNegInf) ? 0.f : m_run;
        {
            unsigned char *pr = gbase + kOffP + pb * kPBytes;
#pragma unroll
            for (int kc = 0; kc < 8; kc++) {
                float pv[8];
#pragma unroll
                for (int k = 0; k < 8; k++) {
                    pv[k] = ex2(s[kc * 8 + k] - mu);
                    l_run += pv[k];
                }
                uint4 w;
                w.x = pack_half2(pv[0], pv[1]);
                w.y = pack_half2(pv[2], pv[3]);
                w.z = pack_half2(pv[4], pv[5]);
                w.w = pack_half2(pv[6], pv[7]);
                *reinterpret_cast<uint4 *>(pr + sw_off(tid, kc)) = w;
            }
        }
        fence_async_smem();
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (abort_sh) break;
        if (tid == 0) {
            const unsigned pa = sP0 + pb * kPBytes, vb = sVt0 + pb * kVtBytes;
#pragma unroll
            for (int kk = 0; kk < 4; kk++)
                umma_f16(tO, sw128_desc(pa + kk * 32), sw128_desc(vb + kk * 32), idO, (j > 0 || kk > 0));
            umma_commit(barO0 + 8 * pb);
        }
        done_tiles = j + 1;
    }

    // wait for the last PV, then write the row's partial
    if (done_tiles > 0 && !abort_sh) {
        const int jl = done_tiles - 1;
        wait_or_abort(barO0 + 8 * (jl & 1), (jl >> 1) & 1);
    }
    tc_fence_after();
    __syncthreads();
    const bool ok = !abort_sh && done_tiles == n_tiles;
    if (!ok && tid == 0) atomicOr(p.flags, 16u);
    const size_t prow = ((size_t)rho * p.max_q_total + r) * p.H + h;
    float *po = p.part_o + prow * 128;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
    for (int q4 = 0; q4 < 4; q4++) {
        float o[32];
        if (n_tiles > 0 && ok) {
            tmem_ld32(tO + lane_off + q4 * 32, o);   // warp-collective: every lane takes part
        } else {
#pragma unroll
            for (int i = 0; i < 32; i++) o[i] = 0.f;
        }
        if (row_ok) {
#pragma unroll
            for (int i = 0; i < 32; i += 4)
                __stcg(reinterpret_cast<float4 *>(po + q4 * 32 + i),
                       make_float4(o[i] * inv, o[i + 1] * inv, o[i + 2] * inv, o[i + 3] * inv));
        }
    }
    if (row_ok) __stcg(p.part_lse + prow, (l_run > 0.f && ok) ? m_run + lg2(l_run) : kNegInf);
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (warp == 0)
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "n"(kTmemCols) : "memory");
}

}  // namespace tc
}  // namespace relay
