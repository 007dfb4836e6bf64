// System-attention step on the 5th-generation tensor cores (tcgen05 + TMEM,
// TMA), for batches with many query rows per head, where the step is a dense,
// compute-bound contraction (atyun.com RelayAttention article, section
// "RelayAttention": the per-request matrix-vector products over the shared
// system prompt grouped into one matrix-matrix product).
//
// An item: KV head hk, a pair of 128-row tiles of its virtual rows (v = r *
// G + c: query row r of the batch with query head hk * G + c, so under
// grouped-query attention the heads of a group share every K/V stage too;
// multi-head: G = 1, v = r), a range of keys.  Both tiles share every K/V
// stage.  Warps have fixed roles:
//   warps 0-3, 4-7  softmax warpgroups, one per query tile; row t of a tile
//                   lives in TMEM lane t and is owned by thread t, so the
//                   online softmax needs no cross-thread reduction
//   warp 8          streams 128-key K and V stages in with TMA (128-byte
//                   swizzle, zero fill past the end of the keys), K and V on
//                   2-stage rings of their own (32 KB stages)
//   warp 9          owns TMEM and issues the S MMAs from one thread
//   warp 10         issues the PV MMAs from one thread
//   warp 11         completes the third warpgroup (the register split below
//                   is per warpgroup)
// In the decode step the softmax warpgroups raise their registers to 224 for
// an item and the others lower theirs to 56 (setmaxnreg): a thread holds a
// whole 128-key stage of its row.
// Per 128-key stage j and query tile t:
//   S = Q K^T        tcgen05.mma kind::f16, M=128 N=128, Q and K K-major in
//                    shared memory, fp32 into the one TMEM S buffer, which the
//                    two tiles take in turn: S_0(j), S_1(j), S_0(j+1), ...
//   P = exp2(S - m)  by the tile's warpgroup, as fp16 pairs into the tile's
//                    TMEM P buffer (tcgen05.st)
//   O += P V         tcgen05.mma, M=128 N=128: P from TMEM, V from shared
//                    memory in its natural [key][d] order (MN-major), never
//                    transposed
// The S thread issues S_t(j) once K(j) has landed and on S-read of the S the
// buffer held before (raised by that tile's warpgroup as soon as its S is in
// registers), so the other tile's S runs while a warpgroup computes its P;
// the PV thread issues PV(j) of both tiles on READY(j), raised once P(j) is in
// TMEM and V(j) has landed; P(j+1) and a rescale of O wait for PV(j)
// (O-done(j)).  A thread that has MMAs in flight waits for them to drain
// before its next shared-memory read completes, so every barrier check on
// an issuing thread empties the tensor pipe: the PV thread checks one barrier
// per stage; the S thread's checks wait for an S that has to complete before
// its warpgroup reads it anyway; the two threads' checks overlap each other's
// MMAs.  No barrier can complete twice before its waiter has seen the first
// completion, so parity waits are never a phase behind.  O is rescaled only when a
// row's running maximum grows by more than 2^8 (P <= 256 otherwise, well
// inside fp16).  Every wait is bounded in time; a wait that gives up raises
// RELAY_FLAG_WAIT_TIMEOUT and the CTA drains its copies and MMAs before it
// frees TMEM and leaves.  Each row's result is one fp32 partial (normalised
// output and log2-sum-exp), merged later with the context partials, or
// (prefill) the final fp16 row and its log-sum-exp; prefill's fp16 tiles go
// out through TMA stores from a swizzled shared-memory tile.
#pragma once

#include <cuda.h>
#include <cuda_fp16.h>
#include <stdint.h>

namespace relay {

namespace tc {

constexpr int kRowsTC = 128;          // query rows per tile (TMEM lanes)
constexpr int kKeysTC = 128;          // keys per K/V stage
constexpr int kPageTC = 16;           // tokens per page of the paged pool
constexpr int kMaxPagesTC = 1024;     // pages of a request's context on the paged path (16384 tokens)
constexpr int kMaxBatchTC = 512;      // requests of a batch
constexpr int kStagesK = 2, kStagesV = 2;   // K stage j is freed when S(j) completes, V stage j when PV(j) does
constexpr int kWarpLoad = 8, kWarpMmaS = 9, kWarpMmaPV = 10;   // warp 11 only completes the third warpgroup
constexpr int kThreadsTC = 384;
// Registers per thread after the split (setmaxnreg, per warpgroup): the
// softmax warpgroups hold a 128-key stage of S, the others need few.  The
// split draws on the block's launch allotment, threads x registers at launch
// (168 for 384 threads); the host checks that before the first launch.
constexpr int kRegSoftmax = 224, kRegRoles = 56, kRegLaunch = 168;
constexpr int kRegSplit = 256 * kRegSoftmax + 128 * kRegRoles;
static_assert(kRegSplit <= kThreadsTC * kRegLaunch, "register split above the launch allotment");
// A protocol wait gives up after RELAY_WAIT_LIMIT_NS (1 s).  A test build
// sets it to 0, so that the first wait not met at once gives up and the
// abort path below runs; draining copies and MMAs in flight before TMEM is
// freed is always bounded by 1 s, whatever the protocol limit.
#ifndef RELAY_WAIT_LIMIT_NS
#define RELAY_WAIT_LIMIT_NS 1000000000ull
#endif
constexpr unsigned long long kWaitNs = RELAY_WAIT_LIMIT_NS;
constexpr unsigned long long kDrainNs = 1000000000ull;

// shared-memory map (byte offsets from a 1024-aligned base), D = 128
constexpr int kHalfQ = kRowsTC * 128;             // one d-half of a Q tile: [128 rows][64 d] fp16 = 16 KB
constexpr int kQTile = 2 * kHalfQ;                // 32 KB
constexpr int kHalfKV = kKeysTC * 128;            // one d-half of a K or V stage: [128 keys][64 d] = 16 KB
constexpr int kStageBytes = 2 * kHalfKV;          // a K stage or a V stage: two d-halves
constexpr int kOffQ = 0;
constexpr int kOffK = kOffQ + 2 * kQTile;
constexpr int kOffV = kOffK + kStagesK * kStageBytes;
constexpr int kOffBar = kOffV + kStagesV * kStageBytes;
constexpr int kSmemTC = kOffBar + 32 * 8 + 1024;   // barriers (at most 32) + alignment slack
// TMEM columns: O tile t: 128 t .. (128); S, one buffer that the two tiles
// take in turn (fp32): 256 .. (128); P tile t (fp16 pairs): 384 + 64 t .. (64)
constexpr int kTmemCols = 512;
constexpr unsigned kColO = 0, kColS = 256, kColP = 384;
constexpr int kPagesPerStage = kKeysTC / kPageTC;   // page boxes per d-half of a context stage
// a stage of a tile pair takes about this long (GB300), for the share of SMs
// that stream decode contexts beside this grid
constexpr float kStageUs = 1.56f;

// mbarrier slots
constexpr int kBarKFull = 0, kBarKEmpty = kStagesK;                           // per K stage
constexpr int kBarVFull = 2 * kStagesK, kBarVEmpty = 2 * kStagesK + kStagesV;   // per V stage
constexpr int kBarSFull = 2 * (kStagesK + kStagesV);   // per tile: S of the tile in the S buffer
constexpr int kBarSRead = kBarSFull + 2;                // per tile: that S in its warpgroup's registers
constexpr int kBarReady = kBarSFull + 4, kBarODone = kBarSFull + 5;   // per stage, both tiles
constexpr int kBarQFull = kBarSFull + 6, kBarFin = kBarSFull + 7;
static_assert(kBarFin < 32, "mbarrier slots");

// --------------------------------------------------------------------------- PTX wrappers
__device__ __forceinline__ void mbar_init(unsigned bar, unsigned count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ bool mbar_try(unsigned bar, unsigned parity)
{
    unsigned ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 " selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

// Non-blocking test of completion `parity`.
__device__ __forceinline__ bool mbar_test(unsigned bar, unsigned parity)
{
    unsigned ok;
    asm volatile("{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
                 " selp.u32 %0, 1, 0, p;\n}\n"
                 : "=r"(ok) : "r"(bar), "r"(parity) : "memory");
    return ok != 0;
}

__device__ __forceinline__ unsigned long long global_ns()
{
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Wait for completion `parity` of an mbarrier.  Gives up (false) when another
// role has raised *abort, or after kWaitNs, raising *abort itself.
__device__ __forceinline__ bool mbar_wait(unsigned bar, unsigned parity, volatile int *abort)
{
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = global_ns();
    for (;;) {
#pragma unroll 1
        for (int i = 0; i < 64; i++)
            if (mbar_try(bar, parity)) return true;
        if (*abort) return false;
        if (global_ns() - t0 > kWaitNs) {
            *abort = 1;
            return false;
        }
    }
}

// Wait used while draining: bounded in time only.
__device__ __forceinline__ void mbar_drain(unsigned bar, unsigned parity)
{
    const unsigned long long t0 = global_ns();
    while (!mbar_try(bar, parity) && global_ns() - t0 < kDrainNs) {
    }
}

__device__ __forceinline__ void mbar_inval(unsigned bar)
{
    asm volatile("mbarrier.inval.shared::cta.b64 [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_arrive(unsigned bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(unsigned bar, unsigned bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes) : "memory");
}

// TMA: one box of a 3-D tensor map at coordinates (x, y, z) into shared memory.
__device__ __forceinline__ void tma_load_3d(unsigned dst, const CUtensorMap *tm, int x, int y, int z, unsigned bar)
{
    asm volatile("cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4}], [%5];\n"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(bar)
                 : "memory");
}

// TMA: one box of a 4-D tensor map at coordinates (x, y, z, w) into shared memory.
__device__ __forceinline__ void tma_load_4d(unsigned dst, const CUtensorMap *tm, int x, int y, int z, int w,
                                            unsigned bar)
{
    asm volatile("cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
                 " [%0], [%1, {%2, %3, %4, %5}], [%6];\n"
                 ::"r"(dst), "l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(w), "r"(bar)
                 : "memory");
}

// TMA: one box of shared memory into a 3-D tensor map at (x, y, z); elements
// outside the tensor are not written (bulk async-group of the issuing thread).
__device__ __forceinline__ void tma_store_3d(const CUtensorMap *tm, unsigned src, int x, int y, int z)
{
    asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.tile.bulk_group [%0, {%1, %2, %3}], [%4];\n"
                 ::"l"(reinterpret_cast<uint64_t>(tm)), "r"(x), "r"(y), "r"(z), "r"(src)
                 : "memory");
}

__device__ __forceinline__ void fence_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}
__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory"); }

// Shared-memory matrix descriptor, 128-byte swizzle, descriptor version 1.
// K-major operand: rows of 128 B, 8-row groups 1024 B apart (stride byte
// offset); the leading byte offset is unused.  MN-major operand: 8 K-rows of
// 128 B (64 MN elements) per 1024 B group, groups 1024 B apart along K
// (stride byte offset), 64-element MN blocks `lbo` bytes apart (leading
// byte offset).
__device__ __forceinline__ uint64_t sw128_desc(unsigned saddr, unsigned lbo = 16u)
{
    uint64_t d = 0;
    d |= (uint64_t)((saddr & 0x3FFFFu) >> 4);            // start address
    d |= (uint64_t)(lbo >> 4) << 16;                      // leading byte offset
    d |= (uint64_t)(1024u >> 4) << 32;                    // stride byte offset
    d |= (uint64_t)1 << 46;                               // version
    d |= (uint64_t)2 << 61;                               // 128-byte swizzle
    return d;
}

// Instruction descriptor, kind::f16: fp16 A and B, fp32 accumulator, shape
// M x N, A K-major, B K-major or (b_mn) MN-major.
__device__ __forceinline__ uint32_t idesc_f16(int M, int N, bool b_mn = false)
{
    return (1u << 4)                          // D: fp32
         | (0u << 7) | (0u << 10)             // A, B: fp16
         | ((b_mn ? 1u : 0u) << 16)           // B major-ness
         | ((uint32_t)(N >> 3) << 17)
         | ((uint32_t)(M >> 4) << 24);
}

// D (TMEM) (+)= A (shared memory) * B (shared memory)
__device__ __forceinline__ void umma_ss(unsigned tmem_d, uint64_t adesc, uint64_t bdesc, uint32_t idesc, int acc)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
                 ::"r"(tmem_d), "l"(adesc), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}

// D (TMEM) (+)= A (TMEM) * B (shared memory)
__device__ __forceinline__ void umma_ts(unsigned tmem_d, unsigned tmem_a, uint64_t bdesc, uint32_t idesc, int acc)
{
    asm volatile("{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
                 " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
                 ::"r"(tmem_d), "r"(tmem_a), "l"(bdesc), "r"(idesc), "r"(acc) : "memory");
}

__device__ __forceinline__ void umma_commit(unsigned bar)
{
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n" ::"r"(bar)
                 : "memory");
}

// 32 consecutive 32-bit columns of this thread's TMEM lane (completion with tmem_wait_ld).
__device__ __forceinline__ void tmem_ld32(unsigned taddr, unsigned (&r)[32])
{
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 "
                 "{%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
                 "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                   "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
                   "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
                   "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
                   "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
                 : "r"(taddr));
}

__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory"); }
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory"); }

// 32 consecutive 32-bit columns of this thread's TMEM lane (completion with tmem_wait_st).
__device__ __forceinline__ void tmem_st32(unsigned taddr, const unsigned (&r)[32])
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], "
                 "{%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
                 "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
                 ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]),
                   "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]),
                   "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]),
                   "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]),
                   "r"(r[29]), "r"(r[30]), "r"(r[31])
                 : "memory");
}

// packed fp32 pairs (two lanes of one 64-bit register)
__device__ __forceinline__ unsigned long long f2_pack(float lo, float hi)
{
    unsigned long long r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ void f2_unpack(unsigned long long v, float &lo, float &hi)
{
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo), "=f"(hi) : "l"(v));
}
__device__ __forceinline__ unsigned long long f2_fma(unsigned long long a, unsigned long long b, unsigned long long c)
{
    unsigned long long r;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(r) : "l"(a), "l"(b), "l"(c));
    return r;
}
__device__ __forceinline__ unsigned long long f2_add(unsigned long long a, unsigned long long b)
{
    unsigned long long r;
    asm("add.rn.f32x2 %0, %1, %2;" : "=l"(r) : "l"(a), "l"(b));
    return r;
}
__device__ __forceinline__ float max3f(float a, float b, float c)
{
    float r;
    asm("max.f32 %0, %1, %2, %3;" : "=f"(r) : "f"(a), "f"(b), "f"(c));
    return r;
}

// byte offset of 16-byte chunk `c` of row `r` in a 128-byte-swizzled region of 128-byte rows
__device__ __forceinline__ unsigned sw_off(int r, int c) { return (unsigned)(r * 128 + ((c ^ (r & 7)) << 4)); }

struct TcParams {
    int B, Lq, H, Ls, max_q_total;
    float scale_log2;
    const __half *q;
    const int *q_lens;
    unsigned *flags;
    float *part_o, *part_lse;        // partial slots: [part][max_q_total][H][128]
    int R, range;                    // key ranges of the system prompt
    int pairs;                       // tile pairs in the grid: ceil(ceil(max_q_total * G / 128) / 2)
    int G;                           // query heads per KV head: head h reads KV head h / G
    int Hkv;                         // KV heads
    __half *out;                     // prefill: [Ls][H][128] fp16 output
    float *lse_out;                  // prefill: [Ls][H] natural-log LSE (nullable)
    // context CTAs, the grid's CTAs from n_sys on: the query rows of the
    // requests with several rows against their own paged context
    int n_sys;                       // system CTAs at the front of the grid
    int ctx_pairs;                   // tile pairs of a request of Lq rows, ceil(ceil(Lq * G / 128) / 2)
    const int *ctx_lens;             // [B] context lengths (null: no context, system step only)
    const int *block_tables;         // [B][max_blocks] page ids
    int max_blocks, num_blocks;
    long long mq_base;               // partial row of compact row r, head h: mq_base + r * H + h
    unsigned *queue;                 // decode step: [0] items taken, [1] CTAs done; zero before the launch and after
    int n_yield;                     // at most this many SMs stream decode contexts beside the tensor cores
    int sms;                         // SMs of the GPU
    float sys_stages;                // K/V stages of all system items
    int out_tma;                     // prefill: the output tiles go out through tmKc (a map of out), else per row
};

// tile pairs for Mv virtual rows
__device__ __forceinline__ int tile_pairs(int Mv) { return ((Mv + kRowsTC - 1) / kRowsTC + 1) / 2; }

__device__ __forceinline__ int owner_of(const int *qo, int n, int x)
{
    int lo = 0, hi = n - 1;
    while (lo < hi) {
        int mid = (lo + hi + 1) >> 1;
        if (qo[mid] <= x) lo = mid; else hi = mid - 1;
    }
    return lo;
}



// Items, in queue order (longest first, so that CTAs finish together):
//   system items, item = (range * Hkv + hk) * pairs + pair: one KV head, a
//     pair of 128-row tiles of its virtual rows, a range of system keys.
//     Items that stream the same keys (one KV head, one key range) are
//     adjacent, so CTAs that run at the same time share them through L2.
//     tmK / tmV view sys_k / sys_v as [Ls][Hkv][128] fp16 with a {64 d, 1
//     head, 128 keys} box and 128-byte swizzle.
//   context items (decode step, after every system item), item - n_sys =
//     c * Hkv + hk: the rows of one request b with several query rows
//     (q_lens[b] > 1) against the request's own context, one pair of its
//     row tiles (c-th in request order, latest tile pair of a request first),
//     one KV head.  Row i of the request (0 <= i < q_lens[b]) sees context
//     keys below max(0, ctx_lens[b] - q_lens[b] + 1 + i): the chunk's own
//     keys are in the context already, causally.  tmKc / tmVc view k_cache /
//     v_cache as [num_blocks][Hkv][16][128] fp16 with a {64 d, 16 tokens, 1,
//     1} box: a 128-key stage is eight page boxes per d-half, page ids from
//     block_tables staged in shared memory; a page past the context reads
//     page id num_blocks, out of range, so the copy fills it with zeros.
//   PREFILL: causal self-attention of the system prompt itself (its Ls query
//     rows, in q = [Ls][H][128]; row t sees system keys 0..t), one key
//     range, item = pair' * Hkv + hk with tile pairs latest (longest) first:
//     an item streams keys up to its last row's position, masks per row on
//     the diagonal stages, and writes the final fp16 output and natural-log
//     LSE instead of partials.
//
// Persistent: at most one CTA per SM, each taking items from the queue
// (queue[0]) until it runs dry (prefill: a static snake order); TMEM is
// allocated once per CTA, the mbarriers are set up afresh for every item.
// The last CTA to leave (queue[1] counts them) sets both words back to zero
// for the next launch.
// In a decode step whose batch also has decode requests, the last CTAs leave
// at once: the streaming kernel, a programmatic dependent of this grid,
// starts on those SMs and streams the decode requests' contexts while the
// tensor cores of the others run; it takes the remaining SMs as this grid's
// CTAs leave.  As many SMs stream (counting those this grid leaves free
// anyway) as the decode bytes need to finish within the tensor-core phase,
// at most n_yield, from two rates measured on GB300: a stage of a tile pair
// takes about kStageUs, and a streaming CTA beside the tensor
// cores moves about 76 GB/s.  Every CTA computes the same count.
template <bool PREFILL>
__global__ void __launch_bounds__(kThreadsTC, 1)
    sys_tc_kernel(const __grid_constant__ CUtensorMap tmK, const __grid_constant__ CUtensorMap tmV,
                  const __grid_constant__ CUtensorMap tmKc, const __grid_constant__ CUtensorMap tmVc, const TcParams p)
{
    extern __shared__ unsigned char smem_raw[];
    __shared__ int qo[kMaxBatchTC + 1];          // query rows before request b
    __shared__ int ip[kMaxBatchTC + 1];          // context items (tile pairs) before request b
    __shared__ int cn_sh[kMaxBatchTC];           // context length of request b
    __shared__ int blk_sh[kMaxPagesTC];          // page ids of a context item
    __shared__ int next_sh, yield_sh;
    __shared__ unsigned tmem_base_sh;
    __shared__ int abort_sh;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const unsigned sraw = static_cast<unsigned>(__cvta_generic_to_shared(smem_raw));
    const unsigned sbase = (sraw + 1023u) & ~1023u;
    unsigned char *gbase = smem_raw + (sbase - sraw);
    auto bar = [&](int i) { return sbase + kOffBar + 8u * (unsigned)i; };
    volatile int *abort_p = &abort_sh;
    // the streaming grid that follows may take the SMs this grid frees once
    // every CTA of this grid has started (it waits for this grid before it
    // leaves)
    if (!PREFILL) asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");

    // The batch, once per CTA: row prefix qo, with the streaming kernel's
    // reading of bad lengths (a q_lens[b] outside [0, Lq] or a ctx_lens[b]
    // outside [0, 16 max_blocks] makes the request empty; that kernel raises
    // the flag), so that both number the rows alike; the context item prefix
    // ip and context lengths; whether any request decodes (one row, a
    // context).
    if (!PREFILL && warp == 0) {
        int run_q = 0, run_i = 0;
        int dec_pages = 0, ctx_stages = 0;    // decode pages of one KV head; context stages of one KV head
        for (int b0 = 0; b0 < p.B; b0 += 32) {
            const int b = b0 + lane;
            int ql = 0, n = 0;
            if (b < p.B) {
                ql = p.q_lens ? p.q_lens[b] : p.Lq;
                n = p.ctx_lens ? p.ctx_lens[b] : 0;
                if (ql < 0 || ql > p.Lq) ql = 0;
                if (n < 0 || n > p.max_blocks * kPageTC) { ql = 0; n = 0; }
                cn_sh[b] = n;
            }
            const int it = (p.ctx_pairs > 0 && ql > 1) ? tile_pairs(ql * p.G) : 0;
            dec_pages += ql == 1 ? (n + kPageTC - 1) / kPageTC : 0;
            ctx_stages += it * ((n + kKeysTC - 1) / kKeysTC);
            const int iq = warp_incl_scan(ql), ii = warp_incl_scan(it);
            if (b < p.B) {
                qo[b] = run_q + iq - ql;
                ip[b] = run_i + ii - it;
            }
            run_q += __shfl_sync(0xffffffffu, iq, 31);
            run_i += __shfl_sync(0xffffffffu, ii, 31);
        }
        dec_pages = __reduce_add_sync(0xffffffffu, dec_pages);
        ctx_stages = __reduce_add_sync(0xffffffffu, ctx_stages);
        if (lane == 0) {
            qo[p.B] = run_q;
            ip[p.B] = run_i;
            int y = 0;
            if (dec_pages > 0) {
                const float tc_us = (p.sys_stages + (float)ctx_stages * p.Hkv) * kStageUs / (float)p.sms;
                const float bytes = (float)dec_pages * p.Hkv * (kPageTC * 128 * 2 * 2);
                const float need = tc_us > 1.f ? ceilf(bytes / (76.0e3f * tc_us)) : (float)p.n_yield;
                y = min((int)fminf(need, (float)p.n_yield), p.n_yield) - (p.sms - (int)gridDim.x);
                y = max(0, min(y, (int)gridDim.x - 1));
            }
            yield_sh = y;
        }
    }
    if (tid == 0) abort_sh = 0;
    __syncthreads();
    const int n_items = PREFILL ? p.pairs * p.Hkv : p.n_sys + ip[p.B] * p.Hkv;
    const bool yield = !PREFILL && (int)blockIdx.x >= (int)gridDim.x - yield_sh;
    if (!yield && warp == kWarpMmaS) {
        const unsigned dst = static_cast<unsigned>(__cvta_generic_to_shared(&tmem_base_sh));
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n" ::"r"(dst), "n"(kTmemCols)
                     : "memory");
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
    }
    // prefill: static items in snake order over the longest-first list
    // (CTA c takes c, 2G - 1 - c, 2G + c, ...; G CTAs), which gives every CTA
    // a similar load without a queue; decode step: the queue
    int round = 0;
    auto snake = [&](int r) {
        const int G = (int)gridDim.x, c = (int)blockIdx.x;
        return (r & 1) ? (r + 1) * G - 1 - c : r * G + c;
    };
    if (tid == 0) next_sh = PREFILL ? snake(0) : yield ? n_items : (int)atomicAdd(p.queue, 1u);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const unsigned tmem = tmem_base_sh;
    auto tO = [&](int t) { return tmem + kColO + (unsigned)(t * 128); };
    const unsigned tS = tmem + kColS;
    auto tP = [&](int t) { return tmem + kColP + (unsigned)(t * 64); };
    auto kstage = [&](int s) { return sbase + kOffK + (unsigned)(s * kStageBytes); };
    auto vstage = [&](int s) { return sbase + kOffV + (unsigned)(s * kStageBytes); };
    // An item's coordinates.  run: it has rows (uniform over the CTA).
    struct Item {
        bool ctx, run;
        int hk, pair, rho, Mv, cb, cql, cn, n_act;
    };
    auto describe = [&](int item) {
        Item d{};
        d.ctx = !PREFILL && item >= p.n_sys;
        if (PREFILL) {
            d.Mv = p.Ls * p.G;
            d.hk = item % p.Hkv;
            d.pair = p.pairs - 1 - item / p.Hkv;
        } else if (!d.ctx) {
            d.Mv = min(qo[p.B], p.max_q_total) * p.G;      // virtual rows of a KV head
            d.hk = (item / p.pairs) % p.Hkv;
            d.pair = item % p.pairs;
            d.rho = item / (p.Hkv * p.pairs);
        } else {
            const int c = (item - p.n_sys) / p.Hkv;
            d.hk = (item - p.n_sys) % p.Hkv;
            d.cb = owner_of(ip, p.B, c);
            d.cql = qo[d.cb + 1] - qo[d.cb];
            d.cn = cn_sh[d.cb];
            d.Mv = d.cql * p.G;
            d.pair = tile_pairs(d.Mv) - 1 - (c - ip[d.cb]);   // latest tile pair first
        }
        const int T = (d.Mv + kRowsTC - 1) / kRowsTC;
        d.run = item < n_items && 2 * d.pair < T && (d.ctx || d.rho < p.R);
        d.n_act = (2 * d.pair + 1 < T) ? 2 : 1;            // query tiles with rows
        return d;
    };
    // Virtual row v = (2 pair + wg) 128 + row of an item: query row r (a
    // context item: row i of request cb, compact row r), query head h.
    auto row_of = [&](const Item &d, int wg, int row, int &r, int &h, int &i_ctx) {
        const int v = (2 * d.pair + wg) * kRowsTC + row;
        i_ctx = v / p.G;
        r = d.ctx ? qo[d.cb] + i_ctx : v / p.G;
        h = d.hk * p.G + v % p.G;
        return wg < d.n_act && v < d.Mv && (!d.ctx || r < p.max_q_total);
    };
    // this thread's query row of an item into the K-major, 128-byte-swizzled
    // Q tile of its warpgroup (zeros for a row the item does not have)
    auto load_q = [&](const Item &d, int wg, int row) {
        int r, h, i_ctx;
        const bool ok = row_of(d, wg, row, r, h, i_ctx);
        const __half *qrow = p.q;
        if (ok && PREFILL) {
            qrow = p.q + ((size_t)r * p.H + h) * 128;
        } else if (ok && d.ctx) {
            qrow = p.q + (((size_t)d.cb * p.Lq + i_ctx) * p.H + h) * 128;
        } else if (ok) {
            const int b = owner_of(qo, p.B, r);
            qrow = p.q + (((size_t)b * p.Lq + (r - qo[b])) * p.H + h) * 128;
        }
        const unsigned sQ = sbase + kOffQ + (unsigned)(wg * kQTile);
#pragma unroll
        for (int c = 0; c < 16; c++) {
            const unsigned dq = sQ + (c >> 3) * kHalfQ + sw_off(row, c & 7);
            asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;\n" ::"r"(dq), "l"(qrow + c * 8),
                         "r"(ok ? 16 : 0));
        }
        asm volatile("cp.async.commit_group;\n" ::: "memory");
    };
    auto fetch = [&]() { return *abort_p ? n_items : PREFILL ? snake(++round) : (int)atomicAdd(p.queue, 1u); };

    bool q_pref = false;          // this thread's Q row of `item` is in flight already
    for (int item = next_sh; item < n_items;) {
        const Item d = describe(item);
        if (!d.run) {                                    // nothing to do (uniform over the CTA)
            __syncthreads();
            if (tid == 0) next_sh = fetch();
            __syncthreads();
            item = next_sh;
            q_pref = false;
            continue;
        }
        const bool ctx = d.ctx;
        const int hk = d.hk, pair = d.pair, rho = d.rho, Mv = d.Mv, cb = d.cb, cql = d.cql, cn = d.cn;
        const int n_act = d.n_act;
        const int v_last = min(Mv, (2 * pair + n_act) * kRowsTC) - 1;   // the item's last virtual row
        const int key0 = (PREFILL || ctx) ? 0 : rho * p.range;
        // prefill: every key up to the position of the item's last row; context:
        // every key its last row sees
        const int key_hi = PREFILL ? v_last / p.G + 1
                         : ctx     ? min(max(cn - cql + 1 + v_last / p.G, 0), cn)
                                   : min(key0 + p.range, p.Ls);
        const int n_tiles = key_hi > key0 ? (key_hi - key0 + kKeysTC - 1) / kKeysTC : 0;
        const int n_pages = ctx ? (key_hi + kPageTC - 1) / kPageTC : 0;   // context pages read

        if (tid == 0) {
            for (int s = 0; s < kStagesK; s++) {
                mbar_init(bar(kBarKFull + s), 1);
                mbar_init(bar(kBarKEmpty + s), 1);
            }
            for (int s = 0; s < kStagesV; s++) {
                mbar_init(bar(kBarVFull + s), 1);
                mbar_init(bar(kBarVEmpty + s), 1);
            }
            for (int t = 0; t < 2; t++) {                // per tile
                mbar_init(bar(kBarSFull + t), 1);
                mbar_init(bar(kBarSRead + t), 4);          // one arrival per warp of the tile's warpgroup
            }
            mbar_init(bar(kBarReady), 4 * n_act);          // one arrival per warp of each active warpgroup
            mbar_init(bar(kBarODone), 1);
            mbar_init(bar(kBarQFull), 256);
            mbar_init(bar(kBarFin), 2);                  // one commit from each MMA thread
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        }
        __syncthreads();
        bool pref_next = false;   // this thread has loaded its Q row of the next item
        // each role's registers for the item (back to the launch count at its
        // end); prefill's items are short, and it measured faster without
        if (!PREFILL) {
            if (warp < 8)
                asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegSoftmax));
            else
                asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegRoles));
        }
        if (warp < 8) {
            // ------------------------------------------------------------ softmax warpgroups
            const int wg = warp >> 2;
            const int row = tid & 127;
            const unsigned lane_off = (unsigned)((warp & 3) * 32) << 16;
            int r, h, i_ctx;
            const bool row_ok = row_of(d, wg, row, r, h, i_ctx);
            // context keys this row sees: below lim_ctx
            const int lim_ctx = min(max(cn - cql + 1 + i_ctx, 0), cn);
            if (!q_pref) load_q(d, wg, row);
            asm volatile("cp.async.wait_all;\n" ::: "memory");
            fence_async_smem();
            mbar_arrive(bar(kBarQFull));
            float m_run = kNegInf, l_run = 0.f;
            int done = 0;
            if (wg < n_act) {
                for (int j = 0; j < n_tiles; j++) {
                    bool ok = mbar_wait(bar(kBarSFull + wg), j & 1, abort_p);
                    if (!__all_sync(0xffffffffu, ok)) break;
                    tc_fence_after();
                    float s[128];
                    {
                        unsigned a[4][32];
#pragma unroll
                        for (int c4 = 0; c4 < 4; c4++) tmem_ld32(tS + lane_off + c4 * 32, a[c4]);
                        tmem_wait_ld();
#pragma unroll
                        for (int i = 0; i < 128; i++) s[i] = __uint_as_float(a[i >> 5][i & 31]);
                    }
                    // S(j) of this tile is in registers: the S buffer may take the next S
                    tc_fence_before();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kBarSRead + wg));
                    const int kbase = key0 + j * kKeysTC;
                    // keys visible to this row: below lim
                    const int lim = PREFILL ? r + 1 : ctx ? lim_ctx : key_hi;
                    if (kbase + kKeysTC > lim) {
#pragma unroll
                        for (int i = 0; i < 128; i++)
                            if (kbase + i >= lim) s[i] = kNegInf;
                    }
                    float mx[8];
#pragma unroll
                    for (int k = 0; k < 8; k++) {
                        mx[k] = max3f(s[k], s[8 + k], s[16 + k]);
#pragma unroll
                        for (int c = 24; c < 120; c += 16) mx[k] = max3f(mx[k], s[c + k], s[c + 8 + k]);
                        mx[k] = fmaxf(mx[k], s[120 + k]);
                    }
                    const float mraw =
                        max3f(max3f(mx[0], mx[1], mx[2]), max3f(mx[3], mx[4], mx[5]), fmaxf(mx[6], mx[7]));
                    const float mt = mraw * p.scale_log2;       // scale > 0: the max commutes with it
                    // lazy rescale: only when this row's max grows by more than 8 (log2)
                    const bool grow = mt > m_run + 8.f || (m_run == kNegInf && mt != kNegInf);
                    const bool any_grow = __any_sync(0xffffffffu, grow);
                    float mn = m_run, alpha = 1.f;
                    if (any_grow) {
                        mn = grow ? mt : m_run;
                        alpha = (m_run == kNegInf) ? 0.f : ex2(m_run - mn);
                    }
                    const float mu = (mn == kNegInf) ? 0.f : mn;
                    unsigned pk[64];
                    const unsigned long long sc2 = f2_pack(p.scale_log2, p.scale_log2), nmu2 = f2_pack(-mu, -mu);
                    unsigned long long ls[4] = {0ull, 0ull, 0ull, 0ull};     // pairs of +0.0f
#pragma unroll
                    for (int i = 0; i < 64; i++) {
                        float x0, x1;
                        f2_unpack(f2_fma(f2_pack(s[2 * i], s[2 * i + 1]), sc2, nmu2), x0, x1);
                        const float p0 = ex2(x0), p1 = ex2(x1);
                        ls[i & 3] = f2_add(ls[i & 3], f2_pack(p0, p1));
                        pk[i] = pack_half2(p0, p1);
                    }
                    float lsum;
                    {
                        float a0, a1;
                        f2_unpack(f2_add(f2_add(ls[0], ls[1]), f2_add(ls[2], ls[3])), a0, a1);
                        lsum = a0 + a1;
                    }
                    // PV(j-1), the last reader of this tile's P buffer and the
                    // last writer of its O, has completed
                    if (j >= 1) {
                        ok = mbar_wait(bar(kBarODone), (j - 1) & 1, abort_p);
                        if (!__all_sync(0xffffffffu, ok)) break;
                        tc_fence_after();
                    }
                    // P row, fp16 pairs, into this tile's P buffer: the A operand
                    // of the PV MMA, read from TMEM
                    tmem_st32(tP(wg) + lane_off, *reinterpret_cast<const unsigned(*)[32]>(pk));
                    tmem_st32(tP(wg) + lane_off + 32, *reinterpret_cast<const unsigned(*)[32]>(pk + 32));
                    if (any_grow && j >= 1) {
                        // O holds PV(0..j-1): rescale it to the new running max
#pragma unroll
                        for (int q4 = 0; q4 < 4; q4++) {
                            unsigned o[32];
                            tmem_ld32(tO(wg) + lane_off + q4 * 32, o);
                            tmem_wait_ld();
#pragma unroll
                            for (int i = 0; i < 32; i++) o[i] = __float_as_uint(__uint_as_float(o[i]) * alpha);
                            tmem_st32(tO(wg) + lane_off + q4 * 32, o);
                        }
                    }
                    l_run = l_run * alpha + lsum;
                    m_run = mn;
                    // the PV thread checks only READY: V(j) must have landed
                    // (checked while the TMEM stores complete)
                    ok = mbar_wait(bar(kBarVFull + j % kStagesV), (j / kStagesV) & 1, abort_p);
                    tmem_wait_st();
                    if (!__all_sync(0xffffffffu, ok)) break;
                    if (ctx && wg == 0 && j == n_tiles - 1 && cn < n_pages * kPageTC) {
                        // the last page's slots past the context hold whatever the
                        // pool holds there: zero their V rows (P is 0 on them, and
                        // 0 times a NaN would not be)
                        const int lo = cn - kbase, cnt = (n_pages * kPageTC - cn) * 16;   // 16-byte chunks
                        unsigned char *vs = gbase + kOffV + (j % kStagesV) * kStageBytes;
                        for (int c = row; c < cnt; c += kRowsTC)
                            *reinterpret_cast<uint4 *>(vs + ((c >> 3) & 1) * kHalfKV + (lo + (c >> 4)) * 128 +
                                                       (c & 7) * 16) = make_uint4(0u, 0u, 0u, 0u);
                        fence_async_smem();
                    }
                    tc_fence_before();   // S(j) loads and the TMEM stores before the MMAs that follow
                    __syncwarp();
                    if (lane == 0) mbar_arrive(bar(kBarReady));
                    done = j + 1;
                }
            }
            // Prefill: the next item of the static order and its query rows,
            // loaded ahead of the last PV MMAs and the epilogue: the Q tile is
            // free once S(n_tiles - 1), its last reader, has completed (an idle
            // tile's at any time).  The softmax warps meet on named barrier 1.
            // (The decode step takes its next item from the queue only once
            // the item is done: taken earlier, the last items of the queue
            // would wait behind long ones, which costs more than the query
            // load of a long item.)
            if (PREFILL) {
                if (tid == 0) next_sh = fetch();
                asm volatile("bar.sync 1, 256;\n" ::: "memory");
                const Item dn = describe(next_sh);
                if (dn.run && !*abort_p && (wg >= n_act || done == n_tiles)) {
                    load_q(dn, wg, row);
                    pref_next = true;
                }
            }
            if (wg < n_act) {
                // the row's partial: normalised O and log2-sum-exp, once every MMA
                // has completed (the single-shot barrier the MMA thread commits last)
                bool fin = done == n_tiles;
                if (fin && n_tiles > 0) fin = mbar_wait(bar(kBarFin), 0, abort_p);
                fin = __all_sync(0xffffffffu, fin);
                tc_fence_after();
                if (!fin && lane == 0) atomicOr(p.flags, RELAY_FLAG_WAIT_TIMEOUT);
                const size_t prow = PREFILL ? (size_t)r * p.H + h
                                  : ctx     ? (size_t)p.mq_base + (size_t)r * p.H + h
                                            : ((size_t)rho * p.max_q_total + r) * p.H + h;
                const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
                if (PREFILL && p.out_tma) {
                    // The tile's fp16 rows into its warpgroup's K stage (free:
                    // every MMA of the item has completed), in the 128-byte-
                    // swizzled layout of the output map's box, then two TMA
                    // stores (one per d-half) by one thread; rows past Ls are
                    // not written.  The stage must be read out before the next
                    // item's K copies: the storing thread waits for that before
                    // the item ends.
                    unsigned char *so = gbase + kOffK + wg * kStageBytes;
#pragma unroll
                    for (int q4 = 0; q4 < 4; q4++) {
                        unsigned o[32];
                        if (fin && n_tiles > 0) {
                            tmem_ld32(tO(wg) + lane_off + q4 * 32, o);   // warp-collective
                            tmem_wait_ld();
                        } else {
#pragma unroll
                            for (int i = 0; i < 32; i++) o[i] = 0u;
                        }
#pragma unroll
                        for (int k = 0; k < 4; k++) {
                            const int c = (q4 & 1) * 4 + k;               // 16-byte chunk within the d-half
                            const float *f = reinterpret_cast<const float *>(o) + 8 * k;
                            *reinterpret_cast<uint4 *>(so + (q4 >> 1) * kHalfKV + sw_off(row, c)) =
                                make_uint4(pack_half2(f[0] * inv, f[1] * inv), pack_half2(f[2] * inv, f[3] * inv),
                                           pack_half2(f[4] * inv, f[5] * inv), pack_half2(f[6] * inv, f[7] * inv));
                        }
                    }
                    fence_async_smem();
                    if (wg == 0)
                        asm volatile("bar.sync 2, 128;\n" ::: "memory");
                    else
                        asm volatile("bar.sync 3, 128;\n" ::: "memory");
                    if (row == 0) {
                        const int v0 = (2 * pair + wg) * kRowsTC;
                        const unsigned src = sbase + kOffK + (unsigned)(wg * kStageBytes);
                        tma_store_3d(&tmKc, src, 0, hk * p.G, v0 / p.G);
                        tma_store_3d(&tmKc, src + kHalfKV, 64, hk * p.G, v0 / p.G);
                        asm volatile("cp.async.bulk.commit_group;\n" ::: "memory");
                        asm volatile("cp.async.bulk.wait_group.read 0;\n" ::: "memory");
                    }
                }
#pragma unroll
                for (int q4 = 0; q4 < 4 && !(PREFILL && p.out_tma); q4++) {
                    unsigned o[32];
                    if (fin && n_tiles > 0) {
                        tmem_ld32(tO(wg) + lane_off + q4 * 32, o);   // warp-collective
                        tmem_wait_ld();
                    } else {
#pragma unroll
                        for (int i = 0; i < 32; i++) o[i] = 0u;
                    }
                    if (row_ok && PREFILL) {
                        __half *po = p.out + prow * 128 + q4 * 32;
#pragma unroll
                        for (int i = 0; i < 32; i += 8)
                            *reinterpret_cast<uint4 *>(po + i) = make_uint4(
                                pack_half2(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv),
                                pack_half2(__uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv),
                                pack_half2(__uint_as_float(o[i + 4]) * inv, __uint_as_float(o[i + 5]) * inv),
                                pack_half2(__uint_as_float(o[i + 6]) * inv, __uint_as_float(o[i + 7]) * inv));
                    } else if (row_ok) {
                        float *po = p.part_o + prow * 128;
#pragma unroll
                        for (int i = 0; i < 32; i += 4)
                            __stcg(reinterpret_cast<float4 *>(po + q4 * 32 + i),
                                   make_float4(__uint_as_float(o[i]) * inv, __uint_as_float(o[i + 1]) * inv,
                                               __uint_as_float(o[i + 2]) * inv, __uint_as_float(o[i + 3]) * inv));
                    }
                }
                if (row_ok && PREFILL) {
                    if (p.lse_out)
                        p.lse_out[prow] = (l_run > 0.f && fin) ? (m_run + lg2(l_run)) * 0.69314718055994531f : kNegInf;
                } else if (row_ok) {
                    __stcg(p.part_lse + prow, (l_run > 0.f && fin) ? m_run + lg2(l_run) : kNegInf);
                }
            }
        } else if (warp == kWarpLoad) {
            // ------------------------------------------------------------ TMA producer
            // K runs up to kStagesK stages ahead and V up to kStagesV, each as
            // soon as its ring has room (polled, so neither ring holds up the other)
            bool bad_blk = false;
            if (ctx) {
                // the request's page ids, checked: an id outside [0, num_blocks)
                // raises the flag and reads as zeros
                const int *bt = p.block_tables + (size_t)cb * p.max_blocks;
                for (int i = lane; i < n_pages; i += 32) {
                    int blk = bt[i];
                    if ((unsigned)blk >= (unsigned)p.num_blocks) {
                        bad_blk = true;
                        blk = p.num_blocks;
                    }
                    blk_sh[i] = blk;
                }
                __syncwarp();
                if (__any_sync(0xffffffffu, bad_blk) && lane == 0) atomicOr(p.flags, RELAY_FLAG_BAD_BLOCK);
            }
            // kPagesPerStage page boxes per d-half of a context stage (pages
            // past the context: page id num_blocks, zero fill)
            auto load_ctx = [&](unsigned dst, const CUtensorMap *tm, int j, unsigned mb) {
#pragma unroll
                for (int q = 0; q < kPagesPerStage; q++) {
                    const int pg = kPagesPerStage * j + q;
                    const int blk = pg < n_pages ? blk_sh[pg] : p.num_blocks;
                    tma_load_4d(dst + q * (kPageTC * 128), tm, 0, 0, hk, blk, mb);
                    tma_load_4d(dst + kHalfKV + q * (kPageTC * 128), tm, 64, 0, hk, blk, mb);
                }
            };
            if (lane == 0) {
                int jk = 0, jv = 0;
                unsigned long long t_last = global_ns();
                while ((jk < n_tiles || jv < n_tiles) && !*abort_p) {
                    bool progress = false;
                    if (jk < n_tiles &&
                        (jk < kStagesK || mbar_test(bar(kBarKEmpty + jk % kStagesK), ((jk / kStagesK) - 1) & 1))) {
                        const int s = jk % kStagesK, z = key0 + jk * kKeysTC;
                        mbar_expect_tx(bar(kBarKFull + s), kStageBytes);
                        if (ctx) {
                            load_ctx(kstage(s), &tmKc, jk, bar(kBarKFull + s));
                        } else {
                            tma_load_3d(kstage(s), &tmK, 0, hk, z, bar(kBarKFull + s));
                            tma_load_3d(kstage(s) + kHalfKV, &tmK, 64, hk, z, bar(kBarKFull + s));
                        }
                        jk++;
                        progress = true;
                    }
                    // V stage jv % kStagesV held V(jv - kStagesV): free once that PV has completed
                    if (jv < n_tiles &&
                        (jv < kStagesV || mbar_test(bar(kBarVEmpty + jv % kStagesV), ((jv / kStagesV) - 1) & 1))) {
                        const int s = jv % kStagesV, z = key0 + jv * kKeysTC;
                        mbar_expect_tx(bar(kBarVFull + s), kStageBytes);
                        if (ctx) {
                            load_ctx(vstage(s), &tmVc, jv, bar(kBarVFull + s));
                        } else {
                            tma_load_3d(vstage(s), &tmV, 0, hk, z, bar(kBarVFull + s));
                            tma_load_3d(vstage(s) + kHalfKV, &tmV, 64, hk, z, bar(kBarVFull + s));
                        }
                        jv++;
                        progress = true;
                    }
                    if (progress) {
                        t_last = global_ns();
                    } else if (global_ns() - t_last > kWaitNs) {
                        *abort_p = 1;
                        break;
                    }
                }
                // no copy may still be in flight when the CTA leaves
                for (int s = 0; s < kStagesK && s < jk; s++)
                    mbar_drain(bar(kBarKFull + s), ((s + ((jk - 1 - s) / kStagesK) * kStagesK) / kStagesK) & 1);
                for (int s = 0; s < kStagesV && s < jv; s++)
                    mbar_drain(bar(kBarVFull + s), ((s + ((jv - 1 - s) / kStagesV) * kStagesV) / kStagesV) & 1);
            }
        } else if (warp == kWarpMmaS) {
            // ------------------------------------------------------------ S = Q K^T
            if (lane == 0) {
                const uint32_t idS = idesc_f16(kRowsTC, kKeysTC);
                int n_s = 0;                             // stages whose S MMAs have all been issued
                int pt = -1, pj = 0;                     // the S last issued into the buffer: tile, stage
                bool ok = mbar_wait(bar(kBarQFull), 0, abort_p);
                for (int j = 0; ok && j < n_tiles; j++) {
                    // K(j) landed (checking drains the S in flight, which has to
                    // complete before its warpgroup reads it anyway)
                    ok = mbar_wait(bar(kBarKFull + j % kStagesK), (j / kStagesK) & 1, abort_p);
                    const unsigned kb = kstage(j % kStagesK);
                    for (int t = 0; ok && t < n_act; t++) {
                        // the buffer's previous S is in its warpgroup's registers
                        if (pt >= 0) ok = mbar_wait(bar(kBarSRead + pt), pj & 1, abort_p);
                        if (!ok) break;
                        tc_fence_after();
                        const unsigned qb = sbase + kOffQ + (unsigned)(t * kQTile);
#pragma unroll
                        for (int kk = 0; kk < 8; kk++)
                            umma_ss(tS, sw128_desc(qb + (kk >> 2) * kHalfQ + (kk & 3) * 32),
                                    sw128_desc(kb + (kk >> 2) * kHalfKV + (kk & 3) * 32), idS, kk > 0);
                        umma_commit(bar(kBarSFull + t));
                        pt = t;
                        pj = j;
                    }
                    if (!ok) break;
                    umma_commit(bar(kBarKEmpty + j % kStagesK));
                    n_s++;
                }
                // every S MMA has completed once the final barrier fires;
                // the K-empty signals of the last stages, which nobody waits
                // for, have landed too before the barriers are set up again
                umma_commit(bar(kBarFin));
                mbar_drain(bar(kBarFin), 0);
                for (int s = 0; s < kStagesK && s < n_s; s++)
                    mbar_drain(bar(kBarKEmpty + s), ((n_s - 1 - s) / kStagesK) & 1);
            }
        } else if (warp == kWarpMmaPV) {
            // ------------------------------------------------------------ O += P V
            if (lane == 0) {
                const uint32_t idO = idesc_f16(kRowsTC, 128, true);
                bool ok = true;
                int n_pv = 0;                            // PV stages issued
                for (int j = 0; ok && j < n_tiles; j++) {
                    const int sv = j % kStagesV;
                    // READY(j): P(j) of every tile stored and V(j) landed
                    ok = mbar_wait(bar(kBarReady), j & 1, abort_p);
                    if (!ok) break;
                    tc_fence_after();
                    const unsigned vb = vstage(sv);
                    for (int t = 0; t < n_act; t++) {
                        // A = P(j) from TMEM: 16 keys = 8 columns of fp16 pairs per MMA
#pragma unroll
                        for (int kk = 0; kk < kKeysTC / 16; kk++)
                            umma_ts(tO(t), tP(t) + kk * 8, sw128_desc(vb + kk * 2048, kHalfKV), idO,
                                    (j > 0 || kk > 0));
                    }
                    umma_commit(bar(kBarODone));
                    umma_commit(bar(kBarVEmpty + sv));    // V stage sv free for the producer
                    n_pv++;
                }
                umma_commit(bar(kBarFin));
                mbar_drain(bar(kBarFin), 0);
                if (n_pv > 0) mbar_drain(bar(kBarODone), (n_pv - 1) & 1);
                for (int v = 0; v < kStagesV && v < n_pv; v++)
                    mbar_drain(bar(kBarVEmpty + v), ((n_pv - 1 - v) / kStagesV) & 1);
            }
        }

        if (!PREFILL) {
            if (warp < 8)
                asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegLaunch));
            else
                asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegLaunch));
        }
        // every role is done with the item, and every barrier phase it started
        // has completed: the barriers may be set up again for the next item
        tc_fence_before();
        __syncthreads();
        if (tid == 0 && !PREFILL) next_sh = fetch();
        if (tid == 0 && !*abort_p) {
            for (int s = 0; s < kStagesK; s++) {
                mbar_inval(bar(kBarKFull + s));
                mbar_inval(bar(kBarKEmpty + s));
            }
            for (int s = 0; s < kStagesV; s++) {
                mbar_inval(bar(kBarVFull + s));
                mbar_inval(bar(kBarVEmpty + s));
            }
            for (int t = 0; t < 2; t++) {
                mbar_inval(bar(kBarSFull + t));
                mbar_inval(bar(kBarSRead + t));
            }
            mbar_inval(bar(kBarReady));
            mbar_inval(bar(kBarODone));
            mbar_inval(bar(kBarQFull));
            mbar_inval(bar(kBarFin));
        }
        if (!PREFILL) __syncthreads();
        tc_fence_after();
        item = *abort_p ? n_items : next_sh;
        q_pref = pref_next;
    }

    // query rows prefetched for an item that did not run (after a wait gave up)
    asm volatile("cp.async.wait_all;\n" ::: "memory");
    // prefill output tiles stored through TMA by this thread have been written
    if (PREFILL && p.out_tma && (tid == 0 || tid == kRowsTC)) asm volatile("cp.async.bulk.wait_group 0;\n" ::: "memory");
    tc_fence_before();
    __syncthreads();
    if (abort_sh && tid == 0) atomicOr(p.flags, RELAY_FLAG_WAIT_TIMEOUT);
    if (!yield && warp == kWarpMmaS) {
        __syncwarp();
        tc_fence_after();
        asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(tmem), "n"(kTmemCols) : "memory");
    }
    // the last CTA out resets the queue
    if (!PREFILL && tid == 0) {
        __threadfence();
        if (atomicAdd(p.queue + 1, 1u) == gridDim.x - 1) {
            p.queue[0] = 0u;
            p.queue[1] = 0u;
        }
    }
}

}  // namespace tc
}  // namespace relay
