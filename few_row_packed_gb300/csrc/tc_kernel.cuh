// tc_kernel.cuh -- the few-row verify kernel on the 5th-generation tensor
// cores: Y[M,N] = X[M,K] . W[K,N], M <= 8, for the packed formats of tc_layout.h.
//
// Design (GB300, sm_103a):
//   * Persistent grid of thread-block clusters.  Cluster y owns a contiguous,
//     balanced range of 128-column tiles; its S CTAs split K into slices.
//     Inside a CTA, three decode warpgroups (one 128-column tile at a time, one
//     thread per weight column) take tiles round-robin and, when a CTA has
//     fewer tiles than warpgroups, also split the slice's chunks (SW ways).
//     The S * SW partial sums of a tile meet in the owner CTA's shared memory
//     (distributed shared memory across the cluster) and are added in a fixed
//     order: deterministic, no global workspace.
//   * Each warpgroup owns a ring of shared-memory stages filled with 1-D bulk
//     async copies of packed records (its decode warps take turns issuing
//     the refills) and one MMA warp.  The decode warps announce each stored A
//     slot with a non-blocking arrival on a hardware named barrier (one per A
//     slot of the ring); the MMA warp syncs on it and issues the slot's
//     tcgen05.mma from converged code (elect.sync).  One commit per chunk
//     tells the decoders that the chunk's A slots are free and its
//     accumulators ready; the decoders release accumulators through an
//     mbarrier.  Every wait is bounded, and a wait that gives up sets the
//     plan's status word and lets the kernel run to its end.
//   * Decode: each thread turns its column's codes into fp16/bf16 pairs with
//     one LOP3 per pair, (word_variant & mask) ^ base, placing a code in a
//     mantissa/exponent field so the value is code_value + c for a small
//     integer c fixed by the bit position (the "codes turned into exact halves
//     with 0x6400 less 1024" idea of the Ishizuki README credits, extended to
//     every position of the word).  The pairs go to tensor memory with
//     tcgen05.st: they are the A operand (128 weight columns x 16 K).
//   * MMA: tcgen05.mma kind::f16, M = 128 columns, N = 16 (the <= 8 rows of X,
//     rows 8-15 alias rows 0-7 and are ignored), K = 16, A from tensor memory,
//     B = X from shared memory, fp32 accumulator in tensor memory, one
//     accumulator per scale group (Ishizuki README, "Kernels written for the
//     verify": each weight is decoded once and used against every row).
//   * Epilogue per group: the warpgroup reads its accumulator back and adds
//     scale * (acc - sum_k c_k x_k) (+ bias * row sum) in fp32, so every
//     tensor-core operand is an exact small integer (the "row-sum prep" of the
//     dflash-mlx-bonsai2 README).
//   * Packed weights stream before griddepcontrol.wait (no kernel writes
//     them); X is read and Y written only after it.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <utility>

#include "tc_internal.h"

namespace lbv {

namespace cg = cooperative_groups;

// ---------------------------------------------------------------------------
// Decode specification of slot s of a word: shift the word (positive = left),
// keep the W-bit field at `target` (and target + 16), XOR the base.  The
// fp16/bf16 value is  code_value + c  (sign1: w + c with w = +-1).
struct DecSpec {
    int shift;
    int target;
    uint32_t base;   // 16-bit pattern, replicated into both halves
    int c;
    int bid;         // index of `base` among the format's distinct bases
};

// 1-bit sign: targets fp16 15 (base -1.0, c 0), 14 (0, 1), 10 (2.0, 3),
// 9..5 (2^(11-j), 2^(11-j)+1); bf16 15, 14, 7 (2.0, 3), 6..2 (2^(8-j), +1).
__host__ __device__ constexpr DecSpec sign1_spec(int xt, int s)
{
    if (xt == LBV_F16) {
        // left shifts only: slots 0-4 -> 5-9, 11-12 -> 14-15, 13 -> 14
        const int sh = (s <= 4) ? 5 : (s == 11 || s == 12) ? 3 : (s == 13) ? 1 : 0;
        const int j = s + sh;
        return j == 15   ? DecSpec{sh, j, 0xBC00u, 0, 0}
               : j == 14 ? DecSpec{sh, j, 0x0000u, 1, 1}
               : j == 10 ? DecSpec{sh, j, 0x4000u, 3, 2}
               : j == 9  ? DecSpec{sh, j, 0x4400u, 5, 3}
               : j == 8  ? DecSpec{sh, j, 0x4800u, 9, 4}
               : j == 7  ? DecSpec{sh, j, 0x4C00u, 17, 5}
               : j == 6  ? DecSpec{sh, j, 0x5000u, 33, 6}
                         : DecSpec{sh, j, 0x5400u, 65, 7};   // j == 5
    } else {
        const int sh = (s <= 1) ? 5 : (s >= 8 && s <= 13) ? -6 : 0;
        const int j = s + sh;
        return j == 15   ? DecSpec{sh, j, 0xBF80u, 0, 0}
               : j == 14 ? DecSpec{sh, j, 0x0000u, 1, 1}
               : j == 7  ? DecSpec{sh, j, 0x4000u, 3, 2}
               : j == 6  ? DecSpec{sh, j, 0x4080u, 5, 3}
               : j == 5  ? DecSpec{sh, j, 0x4100u, 9, 4}
               : j == 4  ? DecSpec{sh, j, 0x4180u, 17, 5}
               : j == 3  ? DecSpec{sh, j, 0x4200u, 33, 6}
                         : DecSpec{sh, j, 0x4280u, 65, 7};   // j == 2
    }
}

// 2-bit code q at bits 2s: value q + c.  fp16 targets 4 (64.0, c 64),
// 6 (16.0, 16), 8 (4.0, 4); bf16 targets 1 (64.0), 3 (16.0), 5 (4.0).
__host__ __device__ constexpr DecSpec affine2_spec(int xt, int s)
{
    if (xt == LBV_F16) {
        const int sh = (s <= 1) ? 4 : (s <= 4) ? 0 : -6;
        const int j = 2 * s + sh;
        return j == 4 ? DecSpec{sh, j, 0x5400u, 64, 0}
               : j == 6 ? DecSpec{sh, j, 0x4C00u, 16, 1}
                        : DecSpec{sh, j, 0x4400u, 4, 2};
    } else {
        const int sh = (s <= 2) ? 1 : (s <= 5) ? -5 : -11;
        const int j = 2 * s + sh;
        return j == 1 ? DecSpec{sh, j, 0x4280u, 64, 0}
               : j == 3 ? DecSpec{sh, j, 0x4180u, 16, 1}
                        : DecSpec{sh, j, 0x4080u, 4, 2};
    }
}

// Q4_0 nibble q at bits 4s: value q + c.  fp16: target 4, base 64.0, c 64;
// bf16: target 3, base 16.0, c 16.
__host__ __device__ constexpr DecSpec q4_0_spec(int xt, int s)
{
    return xt == LBV_F16 ? DecSpec{4 - 4 * s, 4, 0x5400u, 64, 0}
                         : DecSpec{3 - 4 * s, 3, 0x4180u, 16, 0};
}

template <int FMT>
__host__ __device__ constexpr DecSpec dec_spec(int xt, int s)
{
    return FMT == LBV_FMT_SIGN1_G128 ? sign1_spec(xt, s)
           : FMT == LBV_FMT_AFFINE2  ? affine2_spec(xt, s)
                                     : q4_0_spec(xt, s);
}

template <int FMT>
__host__ __device__ constexpr int num_bases()
{
    return FMT == LBV_FMT_SIGN1_G128 ? 8 : FMT == LBV_FMT_AFFINE2 ? 3 : 1;
}

template <int FMT>
__host__ __device__ constexpr uint32_t base_of(int xt, int bid)
{
    uint32_t b = 0;
    for (int s = 0; s < 16; ++s)
        if (dec_spec<FMT>(xt, s).bid == bid)
            b = dec_spec<FMT>(xt, s).base;
    return b | (b << 16);
}

template <int FMT>
__host__ __device__ constexpr int code_bits()
{
    return FMT == LBV_FMT_SIGN1_G128 ? 1 : FMT == LBV_FMT_AFFINE2 ? 2 : 4;
}

template <int FMT, int XT, int S>
__device__ __forceinline__ uint32_t decode(uint32_t w, const uint32_t (&bases)[num_bases<FMT>()])
{
    constexpr DecSpec d = dec_spec<FMT>(XT, S);
    constexpr uint32_t field = (1u << code_bits<FMT>()) - 1u;
    constexpr uint32_t mask = (field << d.target) | (field << (d.target + 16));
    constexpr int shl = d.shift > 0 ? d.shift : 0;
    constexpr int shr = d.shift < 0 ? -d.shift : 0;
    const uint32_t v = shl ? (w << shl) : shr ? (w >> shr) : w;
    // (v & mask) ^ base as one LOP3 with an immediate mask (written in C the
    // compiler splits it into two logic operations)
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(r) : "r"(v), "n"(mask), "r"(bases[d.bid]));
    return r;
}

// ---------------------------------------------------------------------------
// Per-format constants (see tc_layout.h)

template <int FMT, int GROUP>
struct TcTraits;
template <>
struct TcTraits<LBV_FMT_SIGN1_G128, 128> {
    static constexpr int CK = 128, CB = 16, SB = 2, GK = 128;
    static constexpr bool AFFINE = false;
};
template <int G>
struct TcTraits<LBV_FMT_AFFINE2, G> {
    static constexpr int CK = G == 128 ? 128 : 64, CB = G == 128 ? 32 : 16,
                         SB = G == 32 ? 8 : 4, GK = G;
    static constexpr bool AFFINE = true;
};
template <>
struct TcTraits<LBV_FMT_Q4_0, 32> {
    static constexpr int CK = 64, CB = 32, SB = 4, GK = 32;
    static constexpr bool AFFINE = false;
};

template <int FMT, int GROUP>
struct TcGeo {
    using T = TcTraits<FMT, GROUP>;
    static constexpr int W = code_bits<FMT>();
    static constexpr int PPW = 16 / W;               // pairs per 32-bit word
    static constexpr int NWORD = T::CB / 4;
    static constexpr int SLOTS = T::CK / 64;         // A slots (64 K) per chunk
    static constexpr int KSTEPS = T::CK / 16;        // MMA k-steps per chunk
    static constexpr int KSG = T::GK / 16;           // k-steps per scale group
    static constexpr int GPC = T::CK / T::GK;        // scale groups per chunk (1 or 2)
    static constexpr int IU = KSG > 4 ? KSG / 4 : 1; // slots per MMA issue unit (whole groups)
    static constexpr int REC = 128 * (T::CB + T::SB);
    static constexpr int NSIDE = T::SB / 2;          // fp16 side values per column and chunk
    static constexpr int NWG = kTcWarpgroups;        // decode warpgroups per CTA
    static constexpr int DEC_THREADS = NWG * 128;    // decode warps 0 .. 4*NWG-1
    static constexpr int THREADS = DEC_THREADS + NWG * 32;   // + one MMA warp per warpgroup
    // ring stages per warpgroup: about 18 KB in flight each
    static constexpr int NST = REC * 8 <= 18432 ? 8 : 18432 / REC;
    static constexpr int LAG = 2;                    // the epilogue trails decode by LAG chunks
    // accumulators (16 TMEM columns each): the epilogue's LAG chunks, the
    // chunk being decoded, and (when they fit) one more so the MMA warp can
    // run ahead
    static constexpr int ND = GPC == 1 ? LAG + 2 : 2 * (LAG + 1);
    static constexpr int TMEM_WG = 512 / NWG / 32 * 32;   // tensor-memory columns per warpgroup
    static constexpr int NA = (TMEM_WG - ND * 16) / 32;   // A slots (32 TMEM columns each)
    static constexpr int TMEM_COLS = 512;            // allocation (>= NWG * TMEM_WG)
    static_assert(NWG * TMEM_WG <= TMEM_COLS && NA >= 2, "tensor memory budget");
    static_assert((T::CK / 64) % IU == 0, "issue units tile a chunk");
    // chunk-done barriers (a ring over chunks).  A waiter looks back at most
    // max(LAG, NA / SLOTS) chunks; two more keep any barrier from completing
    // two phases past a pending waiter.
    static constexpr int NCD = (LAG > NA / SLOTS ? LAG : NA / SLOTS) + 2;
    static_assert(IU * 64 == T::CK, "an issue unit is one chunk");
    static constexpr int NBAR_WG = 2 * NST + NCD + ND;
    static_assert(1 + NWG * NA <= 16, "named barriers: one per A slot of each warpgroup");
};

// Shared memory carve-up (bytes), 128-byte aligned pieces:
//   stages [NWG][NST][REC] | xs (B operand) [kst][2][8][16] | corr, rsum
//   [groups][8] | part [owned][nparts][8][128] | bars | ctab | tmem slot
// nparts = S * SW partial sums per tile (no part buffer when it is 1).
template <int FMT, int GROUP>
struct TcSmem {
    using G = TcGeo<FMT, GROUP>;
    size_t stages = 0, xs = 0, corr = 0, rsum = 0, part = 0, bars = 0, ctab = 0, tmem = 0, total = 0;
    __host__ __device__ TcSmem() {}
    __host__ __device__ TcSmem(int cps, int owned_max, int nparts)
    {
        auto up = [](size_t v) { return (v + 127) & ~(size_t)127; };
        const int ngroups = cps * G::GPC;
        stages = 0;
        xs = up(stages + (size_t)G::NWG * G::NST * G::REC);
        corr = up(xs + (size_t)cps * G::KSTEPS * 256);
        rsum = up(corr + (size_t)ngroups * 8 * 4);
        part = up(rsum + (size_t)ngroups * 8 * 4);
        bars = up(part + (nparts > 1 ? (size_t)owned_max * nparts * 8 * 128 * 4 : 0));
        ctab = up(bars + (size_t)G::NWG * G::NBAR_WG * 8);
        tmem = ctab + 16 * 4;
        total = up(tmem + 16);
    }
};

// ---------------------------------------------------------------------------
// PTX helpers

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_arrive(uint32_t bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n" ::"r"(bar) : "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// Non-blocking test of an mbarrier phase.
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// One potentially blocking try (the hardware suspends the thread for a
// while if the phase is not complete).
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

__device__ __forceinline__ uint64_t globaltimer_ns()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;\n" : "=l"(t));
    return t;
}

// Bounded wait: false if the phase did not complete within about a second
// (2^31 SM cycles; the cycle counter is cheap to read, unlike the global
// timer).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity)
{
    if (mbar_try(bar, parity))
        return true;
    const long long t0 = clock64();
    while (!mbar_try(bar, parity))
        if (clock64() - t0 > (1ll << 31))
            return false;
    return true;
}

__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

__device__ __forceinline__ void named_bar_sync(int id, int threads)
{
    asm volatile("bar.sync %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void named_bar_arrive(int id, int threads)
{
    asm volatile("bar.arrive %0, %1;\n" ::"r"(id), "r"(threads) : "memory");
}

__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32])
{
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,"
        "%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};\n"
        ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]),
        "r"(r[6]), "r"(r[7]), "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]),
        "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]), "r"(r[17]), "r"(r[18]), "r"(r[19]),
        "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]), "r"(r[25]), "r"(r[26]),
        "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
        : "memory");
}

__device__ __forceinline__ void tmem_wait_st()
{
    asm volatile("tcgen05.wait::st.sync.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&d)[8])
{
    uint32_t r[8];
    asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];\n"
                 : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]),
                   "=r"(r[6]), "=r"(r[7])
                 : "r"(taddr)
                 : "memory");
    asm volatile("tcgen05.wait::ld.sync.aligned;\n" ::: "memory");
#pragma unroll
    for (int i = 0; i < 8; ++i)
        d[i] = __uint_as_float(r[i]);
}

// Arrives on `bar` once every MMA issued so far by the elected lane has
// completed.
__device__ __forceinline__ void umma_commit(uint32_t bar)
{
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n}\n"
        ::"r"(bar)
        : "memory");
}

// The four k-steps of one A slot (A tensor-memory addresses a0..a3, B
// descriptors b0..b3, all computed by the caller so they stay warp-uniform):
// k-step j accumulates into d0 (j < 2) or d1 (j >= 2) and adds to it when bit
// j of ACC is set; then NC commits (to c0, c1, c2) -- all issued by one
// elected lane in a single block.
#define LBV_UMMA_SLOT_BODY                                                     \
    "{\n .reg .pred e, p0, p1, p2, p3;\n"                                      \
    " setp.ne.b32 p0, %15, 0;\n setp.ne.b32 p1, %16, 0;\n"                     \
    " setp.ne.b32 p2, %17, 0;\n setp.ne.b32 p3, %18, 0;\n"                     \
    " elect.sync _|e, 0xffffffff;\n"                                         \
    " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%2], %6, %10, p0;\n"       \
    " @e tcgen05.mma.cta_group::1.kind::f16 [%0], [%3], %7, %10, p1;\n"       \
    " @e tcgen05.mma.cta_group::1.kind::f16 [%1], [%4], %8, %10, p2;\n"       \
    " @e tcgen05.mma.cta_group::1.kind::f16 [%1], [%5], %9, %10, p3;\n"
#define LBV_UMMA_COMMIT(N) \
    " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%" #N "];\n"
#define LBV_UMMA_SLOT_ARGS                                                              \
    "r"(d0), "r"(d1), "r"(a), "r"(a + 8u), "r"(a + 16u), "r"(a + 24u), "l"(b), "l"(b + 16u), \
        "l"(b + 32u), "l"(b + 48u), "r"(idesc), "r"(c0), "r"(c1), "r"(c2), "r"(0u), "r"(f0),  \
        "r"(f1), "r"(f2), "r"(f3)

template <int ACC, int NC>
__device__ __forceinline__ void umma_slot(uint32_t d0, uint32_t d1, uint32_t a, uint64_t b,
                                          uint32_t idesc, uint32_t c0, uint32_t c1, uint32_t c2)
{
    const uint32_t f0 = ACC & 1, f1 = (ACC >> 1) & 1, f2 = (ACC >> 2) & 1, f3 = (ACC >> 3) & 1;
    if constexpr (NC == 0)
        asm volatile(LBV_UMMA_SLOT_BODY "}\n" ::LBV_UMMA_SLOT_ARGS : "memory");
    else if constexpr (NC == 1)
        asm volatile(LBV_UMMA_SLOT_BODY LBV_UMMA_COMMIT(11) "}\n" ::LBV_UMMA_SLOT_ARGS : "memory");
    else if constexpr (NC == 2)
        asm volatile(LBV_UMMA_SLOT_BODY LBV_UMMA_COMMIT(11) LBV_UMMA_COMMIT(12) "}\n"
                     ::LBV_UMMA_SLOT_ARGS : "memory");
    else
        asm volatile(LBV_UMMA_SLOT_BODY LBV_UMMA_COMMIT(11) LBV_UMMA_COMMIT(12) LBV_UMMA_COMMIT(13)
                     "}\n" ::LBV_UMMA_SLOT_ARGS : "memory");
}

// Shared-memory matrix descriptor, K-major without swizzle: core matrices of
// 8 rows x 16 bytes, K-adjacent cores `lbo` bytes apart, N-adjacent `sbo`.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)((lbo >> 4) & 0x3FFFu) << 16) |
           ((uint64_t)((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f16: fp32 accumulator, A/B fp16 or bf16,
// both K-major, N = 16, M = 128.
template <int XT>
__host__ __device__ constexpr uint32_t idesc_f16()
{
    return (1u << 4) | ((uint32_t)(XT == LBV_BF16) << 7) | ((uint32_t)(XT == LBV_BF16) << 10) |
           ((16u >> 3) << 17) | ((128u >> 4) << 24);
}

// ---------------------------------------------------------------------------

template <int FMT, int XT, int GROUP>
struct TcKernel {
    using T = TcTraits<FMT, GROUP>;
    using G = TcGeo<FMT, GROUP>;
    static constexpr int NB = num_bases<FMT>();

    struct Ctx {
        const TcParams* p;
        unsigned char* smem;
        TcSmem<FMT, GROUP> lay;
        uint32_t tmem;
        int S, SW, rank, c0, nch, t0, t1;
    };

    // The work of one warpgroup: tiles t0 + tl + TL * u (u < nu) of the
    // cluster's range, slice chunks [cw0, cw0 + nchw) of each.
    struct Work {
        int TL, tl, ws, nu, cw0, nchw;
    };

    static __device__ __forceinline__ Work work_of(const Ctx& c, int wg)
    {
        Work w;
        w.TL = G::NWG / c.SW;
        w.tl = wg % w.TL;
        w.ws = wg / w.TL;
        const int ntile = c.t1 - c.t0;
        w.nu = w.tl < ntile ? (ntile - 1 - w.tl) / w.TL + 1 : 0;
        w.cw0 = (c.nch * w.ws) / c.SW;
        w.nchw = (c.nch * (w.ws + 1)) / c.SW - w.cw0;   // may be 0: the partial is then 0
        return w;
    }

    static __device__ __forceinline__ uint32_t bar_addr(const Ctx& c, int wg, int i)
    {
        return smem_u32(c.smem + c.lay.bars) + (uint32_t)((wg * G::NBAR_WG + i) * 8);
    }
    // barrier indices within a warpgroup's block
    static constexpr int B_FULL = 0, B_EMPTY = G::NST, B_CDONE = 2 * G::NST,
                         B_DEMPTY = 2 * G::NST + G::NCD;
    // Waits until the MMAs of the warpgroup's chunk number qc have completed.
    static __device__ __forceinline__ bool wait_chunk(const Ctx& c, int wg, int qc)
    {
        return mbar_wait(bar_addr(c, wg, B_CDONE + qc % G::NCD), (uint32_t)((qc / G::NCD) & 1));
    }
    // hardware named barrier of A slot a of warpgroup wg (0 is __syncthreads)
    static __device__ __forceinline__ int abar_id(int wg, int a) { return 1 + wg * G::NA + a; }

    // ---- prologue: X slice as the B operand, per-group corrections ----
    static __device__ void stage_x(const Ctx& c, int tid)
    {
        const TcParams& p = *c.p;
        const int kb = c.c0 * T::CK;
        const int nks = c.nch * G::KSTEPS;
        const int pieces = nks * 2 * 8;                 // (k-step, core, row) 16-byte pieces
        const uint16_t* X = reinterpret_cast<const uint16_t*>(p.X);
        unsigned char* xs = c.smem + c.lay.xs;
        constexpr int NT = G::DEC_THREADS;
        constexpr int B = 4;
        for (int i0 = tid; i0 < pieces; i0 += B * NT) {
            uint4 v[B];
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int i = i0 + b * NT;
                v[b] = make_uint4(0u, 0u, 0u, 0u);
                if (i < pieces) {
                    const int m = i & 7, ki = (i >> 3) & 1, ks = i >> 4;
                    const int k = kb + ks * 16 + ki * 8;
                    if (m < p.M && k < p.K) {
                        const uint16_t* src = X + (size_t)m * p.ldx + k;
                        if (p.x_vec) {
                            v[b] = *reinterpret_cast<const uint4*>(src);
                        } else {
                            v[b].x = (uint32_t)src[0] | ((uint32_t)src[1] << 16);
                            v[b].y = (uint32_t)src[2] | ((uint32_t)src[3] << 16);
                            v[b].z = (uint32_t)src[4] | ((uint32_t)src[5] << 16);
                            v[b].w = (uint32_t)src[6] | ((uint32_t)src[7] << 16);
                        }
                    }
                }
            }
#pragma unroll
            for (int b = 0; b < B; ++b) {
                const int i = i0 + b * NT;
                if (i < pieces)   // piece i lives at ks*256 + ki*128 + m*16 == 16*i
                    *reinterpret_cast<uint4*>(xs + (size_t)i * 16) = v[b];
            }
        }
    }

    template <int XT_>
    static __device__ __forceinline__ float2 pair_f2(uint32_t v)
    {
        if constexpr (XT_ == LBV_F16) {
            __half2 h = *reinterpret_cast<__half2*>(&v);
            return __half22float2(h);
        } else {
            __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
            return __bfloat1622float2(h);
        }
    }

    // corr[g][m] = sum_k c_k x[m][k] (Q4_0: + 8 * rowsum), rsum[g][m] = rowsum
    static __device__ void corrections(const Ctx& c, int warp, int lane)
    {
        const unsigned char* xs = c.smem + c.lay.xs;
        const float* ctab = reinterpret_cast<const float*>(c.smem + c.lay.ctab);
        float* corr = reinterpret_cast<float*>(c.smem + c.lay.corr);
        float* rsum = reinterpret_cast<float*>(c.smem + c.lay.rsum);
        const int ngroups = c.nch * G::GPC;
        const int m = lane >> 2, q = lane & 3;          // row, quarter of the group
        for (int gr = warp; gr < ngroups; gr += G::NWG * 4) {
            const int kbeg = gr * T::GK;                 // slice-relative K of the group
            float cs = 0.f, rs = 0.f;
            for (int kk = q * (T::GK / 4); kk < (q + 1) * (T::GK / 4); kk += 8) {
                const int k = kbeg + kk;                 // multiple of 8
                const uint4 v = *reinterpret_cast<const uint4*>(
                    xs + (size_t)(k >> 4) * 256 + ((k >> 3) & 1) * 128 + m * 16);
                const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const float2 f = pair_f2<XT>(w4[e]);
                    const int pr = ((k % T::CK) >> 1) + e;   // pair index within the chunk
                    const float cc = ctab[pr % G::PPW];
                    cs += cc * (f.x + f.y);
                    rs += f.x + f.y;
                }
            }
            cs += __shfl_xor_sync(0xffffffffu, cs, 1);
            cs += __shfl_xor_sync(0xffffffffu, cs, 2);
            rs += __shfl_xor_sync(0xffffffffu, rs, 1);
            rs += __shfl_xor_sync(0xffffffffu, rs, 2);
            if (q == 0) {
                corr[gr * 8 + m] = FMT == LBV_FMT_Q4_0 ? cs + 8.f * rs : cs;
                rsum[gr * 8 + m] = rs;
            }
        }
    }

    // ---- producer (warp 0 of a warpgroup): record of batch q into its stage ----
    static __device__ __forceinline__ void produce(const Ctx& c, const Work& w, int wg, int q,
                                                   int lane)
    {
        const TcParams& p = *c.p;
        const int u = q / w.nchw, cl = q - u * w.nchw;
        const int tile = c.t0 + w.tl + w.TL * u;
        const uint8_t* src = p.W + ((size_t)tile * p.nchunks + c.c0 + w.cw0 + cl) * G::REC;
        const int st = q % G::NST;
#ifdef LBV_CHECKED
        // checked build: the record lies inside the packed matrix (else no copy:
        // its waiters give up and the status records both)
        if (tile < 0 || tile >= p.ntiles || c.c0 + w.cw0 + cl < 0 ||
            c.c0 + w.cw0 + cl >= p.nchunks) {
            if (lane == 0)
                atomicOr(p.err, 2u);
            return;
        }
#endif
        if (lane == 0) {
            const uint32_t fb = bar_addr(c, wg, B_FULL + st);
            mbar_expect_tx(fb, (uint32_t)G::REC);
            bulk_g2s(smem_u32(c.smem + c.lay.stages + (size_t)(wg * G::NST + st) * G::REC), src,
                     (uint32_t)G::REC, fb);
        }
    }

    // ---- the MMA warp of warpgroup wg: every A slot, in order ----
    // It loops over issue units (IU slots holding whole scale groups), so
    // which k-steps start a group and which commits follow a slot are
    // compile-time facts.
    static __device__ void mma_warp(const Ctx& c, const Work& w, int wg, bool& ok)
    {
        const uint32_t idesc = idesc_f16<XT>();
        const uint32_t tm = c.tmem + (uint32_t)(wg * G::TMEM_WG);
        const uint32_t dcol = tm + (uint32_t)(G::NA * 32);
        const uint64_t xdesc0 = smem_desc(smem_u32(c.smem + c.lay.xs) +
                                              (uint32_t)(w.cw0 * G::KSTEPS * 256), 128, 0);
        const int units_per_tile = w.nchw * G::SLOTS / G::IU;
        constexpr int GPU_ = G::IU * 4 / G::KSG;            // groups per unit (1 or 2)
        int s = 0, a = 0, gi = 0, qc = 0;
        for (int u = 0; u < w.nu; ++u) {
            uint64_t b = xdesc0;                             // k-step 0 of the tile's first chunk
            for (int j = 0; j < units_per_tile; ++j) {
                // the accumulators of the unit's groups have been read
#pragma unroll
                for (int g = 0; g < GPU_; ++g) {
                    const int gg = gi + g;
                    if (gg >= G::ND && ok &&
                        !mbar_wait(bar_addr(c, wg, B_DEMPTY + gg % G::ND), (uint32_t)(((gg / G::ND) - 1) & 1)))
                        ok = false;
                }
#pragma unroll
                for (int i = 0; i < G::IU; ++i) {
                    named_bar_sync(abar_id(wg, a), 160);     // the four decode warps stored slot s + i
                    tc_fence_after();
                    const uint32_t a_t = tm + (uint32_t)(a * 32);
                    const uint32_t cdone = bar_addr(c, wg, B_CDONE + qc % G::NCD);
                    const uint32_t d0 = dcol + (uint32_t)((gi % G::ND) * 16);
                    // one commit per chunk (= unit), after its last slot
                    if constexpr (GPU_ == 2) {
                        const uint32_t d1 = dcol + (uint32_t)(((gi + 1) % G::ND) * 16);
                        umma_slot<0xA, 1>(d0, d1, a_t, b, idesc, cdone, 0u, 0u);
                    } else if (i == 0 && i == G::IU - 1) {
                        umma_slot<0xE, 1>(d0, d0, a_t, b, idesc, cdone, 0u, 0u);
                    } else if (i == 0) {
                        umma_slot<0xE, 0>(d0, d0, a_t, b, idesc, 0u, 0u, 0u);
                    } else if (i == G::IU - 1) {
                        umma_slot<0xF, 1>(d0, d0, a_t, b, idesc, cdone, 0u, 0u);
                    } else {
                        umma_slot<0xF, 0>(d0, d0, a_t, b, idesc, 0u, 0u, 0u);
                    }
                    b += (uint64_t)(4 * 256 >> 4);
                    a = a + 1 == G::NA ? 0 : a + 1;
                }
                s += G::IU;
                gi += GPU_;
                ++qc;
            }
        }
        // the last commits are the last arrivals any barrier gets: wait for
        // them before tensor and shared memory go away
        for (int i = 0; i < G::NCD && i < qc; ++i)
            if (ok && !wait_chunk(c, wg, qc - 1 - i))
                ok = false;
    }

    // Slot s is stored by this warp: once its store is complete, announce it
    // to the MMA warp (non-blocking).
    static __device__ __forceinline__ void complete_slot(int wg, int s)
    {
        tmem_wait_st();
        tc_fence_before();
        named_bar_arrive(abar_id(wg, s % G::NA), 160);
    }

    // ---- one warp of a decode warpgroup ----
    static __device__ void warp_loop(const Ctx& c, const Work& w, int wg, int wq, int lane, bool& ok)
    {
        const int col = wq * 32 + lane;                      // column within the tile
        const float* corr = reinterpret_cast<const float*>(c.smem + c.lay.corr);
        const float* rsum = reinterpret_cast<const float*>(c.smem + c.lay.rsum);
        float* part = reinterpret_cast<float*>(c.smem + c.lay.part);
        const uint32_t lane_off = (uint32_t)(wq * 32) << 16;
        const uint32_t tm_wg = c.tmem + (uint32_t)(wg * G::TMEM_WG) + lane_off;

        uint32_t bases[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i)
            asm volatile("mov.b32 %0, %1;\n" : "=r"(bases[i]) : "r"(base_of<FMT>(XT, i)));

        const int Q = w.nu * w.nchw;
        int q = 0, s = 0, gc = 0;
        bool pending = false;        // a stored slot not yet completed (named barrier + issue)
        for (int u = 0; u < w.nu; ++u) {
            const int tile = c.t0 + w.tl + w.TL * u;
            float y[8];
#pragma unroll
            for (int m = 0; m < 8; ++m)
                y[m] = 0.f;
            // side values (scale, bias) of the last LAG chunks' groups:
            // hs[j], hb[j] belong to chunk cl - 1 - j
            float hs[G::LAG][G::GPC], hb[G::LAG][G::GPC];
#pragma unroll
            for (int j = 0; j < G::LAG; ++j)
#pragma unroll
                for (int gi = 0; gi < G::GPC; ++gi)
                    hs[j][gi] = hb[j][gi] = 0.f;
            for (int cl = 0; cl < w.nchw + G::LAG; ++cl) {
                float cs[G::GPC] = {}, cb[G::GPC] = {};
                if (cl < w.nchw) {
                    const int st = q % G::NST;
                    if (ok && !mbar_wait(bar_addr(c, wg, B_FULL + st), (uint32_t)((q / G::NST) & 1)))
                        ok = false;
                    const unsigned char* sp = c.smem + c.lay.stages + (size_t)(wg * G::NST + st) * G::REC;
                    uint32_t wv[G::NWORD];
#pragma unroll
                    for (int h = 0; h < T::CB / 16; ++h) {
                        const uint4 v = *reinterpret_cast<const uint4*>(sp + h * 2048 + col * 16);
                        wv[4 * h + 0] = v.x;
                        wv[4 * h + 1] = v.y;
                        wv[4 * h + 2] = v.z;
                        wv[4 * h + 3] = v.w;
                    }
                    uint16_t sv[G::NSIDE];
#pragma unroll
                    for (int i = 0; i < G::NSIDE; ++i)
                        sv[i] = reinterpret_cast<const uint16_t*>(sp + 128 * T::CB + col * T::SB)[i];
                    __syncwarp();
                    if (lane == 0)
                        mbar_arrive(bar_addr(c, wg, B_EMPTY + st));
                    // warp q mod 4 refills the stage read one batch ago (all four
                    // warps are done with it)
                    if (wq == (q & 3) && q >= 1 && q - 1 + G::NST < Q) {
                        const int qr = q - 1;
                        if (ok && !mbar_wait(bar_addr(c, wg, B_EMPTY + qr % G::NST), (uint32_t)((qr / G::NST) & 1)))
                            ok = false;
                        produce(c, w, wg, qr + G::NST, lane);
                    }
                    ++q;
#pragma unroll
                    for (int gi = 0; gi < G::GPC; ++gi) {
                        if constexpr (T::AFFINE) {
                            cs[gi] = __half2float(__ushort_as_half(sv[2 * gi]));
                            cb[gi] = __half2float(__ushort_as_half(sv[2 * gi + 1]));
                        } else {
                            cs[gi] = __half2float(__ushort_as_half(sv[gi]));
                            cb[gi] = 0.f;
                        }
                    }
                    // decode and store each A slot of the chunk.  A slot's
                    // store completes while the next slot is decoded: its
                    // announcement (wait::st, the named-barrier arrival) is
                    // deferred to just before the next store.
#pragma unroll
                    for (int si = 0; si < G::SLOTS; ++si) {
                        uint32_t r[32];
                        decode_slot(wv, si, bases, r);
                        if (pending)
                            complete_slot(wg, s - 1);
                        const int a = s % G::NA;
                        // the A slot's previous contents were consumed by the
                        // MMAs of chunk (s - NA) / SLOTS
                        if (s >= G::NA && ok && !wait_chunk(c, wg, (s - G::NA) / G::SLOTS))
                            ok = false;
                        tc_fence_after();
                        tmem_st32(tm_wg + (uint32_t)(a * 32), r);
                        pending = true;
                        ++s;
                    }
                }
                // the last chunk's MMAs need its last slot before its epilogue
                if (cl >= w.nchw && pending) {
                    complete_slot(wg, s - 1);
                    pending = false;
                }
                // epilogue of chunk cl - LAG's groups (their MMAs ran while the
                // later chunks were decoded)
                if (cl >= G::LAG) {
#pragma unroll
                    for (int gi = 0; gi < G::GPC; ++gi) {
                        const int d = gc % G::ND;
                        if (ok && !wait_chunk(c, wg, gc / G::GPC))
                            ok = false;
                        tc_fence_after();
                        float acc[8];
                        tmem_ld8(tm_wg + (uint32_t)(G::NA * 32 + d * 16), acc);
                        tc_fence_before();
                        __syncwarp();
                        if (lane == 0)
                            mbar_arrive(bar_addr(c, wg, B_DEMPTY + d));
                        ++gc;
                        const int gr = (w.cw0 + cl - G::LAG) * G::GPC + gi;   // group within the slice
                        const float4 c0v = *reinterpret_cast<const float4*>(corr + gr * 8);
                        const float4 c1v = *reinterpret_cast<const float4*>(corr + gr * 8 + 4);
                        const float cv[8] = {c0v.x, c0v.y, c0v.z, c0v.w, c1v.x, c1v.y, c1v.z, c1v.w};
#pragma unroll
                        for (int m = 0; m < 8; ++m)
                            y[m] = fmaf(hs[G::LAG - 1][gi], acc[m] - cv[m], y[m]);
                        if constexpr (T::AFFINE) {
                            const float4 r0 = *reinterpret_cast<const float4*>(rsum + gr * 8);
                            const float4 r1 = *reinterpret_cast<const float4*>(rsum + gr * 8 + 4);
                            const float rv[8] = {r0.x, r0.y, r0.z, r0.w, r1.x, r1.y, r1.z, r1.w};
#pragma unroll
                            for (int m = 0; m < 8; ++m)
                                y[m] = fmaf(hb[G::LAG - 1][gi], rv[m], y[m]);
                        }
                    }
                }
#pragma unroll
                for (int j = G::LAG - 1; j > 0; --j)
#pragma unroll
                    for (int gi = 0; gi < G::GPC; ++gi) {
                        hs[j][gi] = hs[j - 1][gi];
                        hb[j][gi] = hb[j - 1][gi];
                    }
#pragma unroll
                for (int gi = 0; gi < G::GPC; ++gi) {
                    hs[0][gi] = cs[gi];
                    hb[0][gi] = cb[gi];
                }
            }
            store_tile(c, w, tile, col, y, part);
        }
        // after a give-up, let the copies still in flight land
        if (!ok) {
            const int issued = min(Q, q + G::NST);
            for (int qq = q; qq < issued; ++qq)
                mbar_wait(bar_addr(c, wg, B_FULL + qq % G::NST), (uint32_t)((qq / G::NST) & 1));
        }
    }

    // decode the 32 pairs of A slot si (pairs 32*si .. 32*si + 31 of the chunk)
    template <int... R>
    static __device__ __forceinline__ void decode_pairs(std::integer_sequence<int, R...>,
                                                        const uint32_t (&wv)[G::NWORD], int base,
                                                        const uint32_t (&bases)[NB],
                                                        uint32_t (&r)[32])
    {
        ((r[R] = decode<FMT, XT, R % G::PPW>(wv[(base + R) / G::PPW], bases)), ...);
    }

    static __device__ __forceinline__ void decode_slot(const uint32_t (&wv)[G::NWORD], int si,
                                                       const uint32_t (&bases)[NB],
                                                       uint32_t (&r)[32])
    {
        if (G::SLOTS == 1 || si == 0)
            decode_pairs(std::make_integer_sequence<int, 32>{}, wv, 0, bases, r);
        else
            decode_pairs_hi(std::make_integer_sequence<int, 32>{}, wv, bases, r);
    }

    template <int... R>
    static __device__ __forceinline__ void decode_pairs_hi(std::integer_sequence<int, R...>,
                                                           const uint32_t (&wv)[G::NWORD],
                                                           const uint32_t (&bases)[NB],
                                                           uint32_t (&r)[32])
    {
        ((r[R] = decode<FMT, XT, (32 + R) % G::PPW>(wv[((32 + R) / G::PPW) % G::NWORD], bases)), ...);
    }

    // Partial sums: with nparts = S * SW > 1 the tile's partial goes to the
    // owner CTA (tile index i within the cluster range: owner rank i % S,
    // owner slot i / S), entry rank * SW + ws of that slot.
    static __device__ __forceinline__ void store_tile(const Ctx& c, const Work& w, int tile, int col,
                                                      const float (&y)[8], float* part)
    {
        const TcParams& p = *c.p;
        const int np = c.S * c.SW;
        if (np > 1) {
            const int i = tile - c.t0;
            float* base = part;
            if (c.S > 1)
                base = cg::this_cluster().map_shared_rank(part, (unsigned)(i % c.S));
            float* dst = base + ((size_t)((i / c.S) * np + c.rank * c.SW + w.ws) * 8) * 128 + col;
#pragma unroll
            for (int m = 0; m < 8; ++m)
                dst[m * 128] = y[m];
            return;
        }
        const int n = tile * 128 + col;
        if (n < p.N)
#pragma unroll
            for (int m = 0; m < 8; ++m)
                if (m < p.M)
                    p.Y[(size_t)m * p.ldy + n] = y[m];
    }

    static __device__ void reduce_parts(const Ctx& c, int tid, int nthreads)
    {
        const TcParams& p = *c.p;
        const float* part = reinterpret_cast<const float*>(c.smem + c.lay.part);
        const int S = c.S, np = S * c.SW;
        const int nown = (c.t1 - c.t0 - c.rank + S - 1) / S;     // tiles t0 + rank + S*k
        for (int e = tid; e < nown * 8 * 128; e += nthreads) {
            const int k = e / (8 * 128), r = e % (8 * 128);
            const int m = r >> 7, col = r & 127;
            const float* src = part + (size_t)(k * np) * 8 * 128 + r;
            float acc = 0.f;
            for (int qq = 0; qq < np; ++qq)
                acc += src[(size_t)qq * 8 * 128];
            const int n = (c.t0 + c.rank + S * k) * 128 + col;
            if (n < p.N && m < p.M)
                p.Y[(size_t)m * p.ldy + n] = acc;
        }
    }

    static __device__ void run(const TcParams& p, unsigned char* smem)
    {
        const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
        Ctx c;
        c.p = &p;
        c.smem = smem;
        c.S = p.splits;
        c.SW = p.wsplit;
        c.rank = (int)blockIdx.x;
        c.c0 = blockIdx.x * p.cps;
        c.nch = min(p.cps, p.nchunks - c.c0);
        c.t0 = (int)(((unsigned)p.ntiles * blockIdx.y) / gridDim.y);
        c.t1 = (int)(((unsigned)p.ntiles * (blockIdx.y + 1)) / gridDim.y);
        const int owned_max = ((p.ntiles + gridDim.y - 1) / gridDim.y + c.S - 1) / c.S;
        c.lay = TcSmem<FMT, GROUP>(p.cps, owned_max, c.S * c.SW);
        uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + c.lay.tmem);

        if (c.S > 1)
            cluster_arrive_relaxed();
        if (warp == 0) {
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;\n"
                         ::"r"(smem_u32(tmem_slot)), "n"(G::TMEM_COLS)
                         : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
        } else if (tid == 32) {
            for (int w = 0; w < G::NWG; ++w) {
                for (int i = 0; i < G::NST; ++i) {
                    mbar_init(bar_addr(c, w, B_FULL + i), 1);
                    mbar_init(bar_addr(c, w, B_EMPTY + i), 4);
                }
                for (int i = 0; i < G::NCD; ++i)
                    mbar_init(bar_addr(c, w, B_CDONE + i), 1);
                for (int i = 0; i < G::ND; ++i)
                    mbar_init(bar_addr(c, w, B_DEMPTY + i), 4);
            }
            asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
        } else if (tid >= 64 && tid < 80) {
            float* ctab = reinterpret_cast<float*>(smem + c.lay.ctab);
            ctab[tid - 64] = (float)dec_spec<FMT>(XT, tid - 64).c;
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        c.tmem = *tmem_slot;

        const bool is_mma = warp >= G::NWG * 4;
        const int wg = is_mma ? warp - G::NWG * 4 : warp / 4, wq = warp % 4;
        const Work w = work_of(c, wg);
        if (is_mma) {
            // the packed weights start streaming before the previous kernel
            // ends; lane l fills stage l
            const int first = min(G::NST, w.nu * w.nchw);
            for (int q = lane; q < first; q += 32)
                produce(c, w, wg, q, 0);
        } else {
            griddep_wait();
            stage_x(c, tid);
            fence_proxy_async_smem();       // X is read by the tensor core (async proxy)
        }
        __syncthreads();
        if (!is_mma)
            corrections(c, warp, lane);
        __syncthreads();
        griddep_launch_dependents();
        if (c.S > 1)
            cluster_wait();                 // peers run: their partial buffers are live

        bool ok = true;
        if (is_mma)
            mma_warp(c, w, wg, ok);
        else
            warp_loop(c, w, wg, wq, lane, ok);
        if (!ok)
            atomicOr(p.err, 1u);
        if (c.S * c.SW > 1) {
            if (c.S > 1)
                cg::this_cluster().sync();
            else
                __syncthreads();
            reduce_parts(c, tid, G::THREADS);
        }
        tc_fence_before();
        __syncthreads();
        tc_fence_after();
        if (warp == 0)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;\n" ::"r"(c.tmem),
                         "n"(G::TMEM_COLS)
                         : "memory");
    }
};

template <int FMT, int XT, int GROUP>
__global__ void __launch_bounds__(TcGeo<FMT, GROUP>::THREADS, 1) lbv_tc_kernel(const TcParams p)
{
    extern __shared__ __align__(1024) unsigned char smem[];
    TcKernel<FMT, XT, GROUP>::run(p, smem);
}

// ---------------------------------------------------------------------------
// Host side

template <int FMT, int GROUP>
inline size_t tc_smem_bytes(int cps, int owned_max, int nparts)
{
    return TcSmem<FMT, GROUP>(cps, owned_max, nparts).total;
}

inline void tc_fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], const TcShape& sh,
                           int threads, bool pdl, cudaStream_t st)
{
    cfg = {};
    cfg.gridDim = dim3((unsigned)sh.splits, (unsigned)sh.ctas_n, 1u);
    cfg.blockDim = dim3((unsigned)threads, 1u, 1u);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = st;
    unsigned na = 0;
    if (sh.splits > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)sh.splits;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
}

template <int FMT, int XT, int GROUP>
inline cudaError_t tc_launch_t(const TcShape& sh, const TcParams& p, const LaunchOpts& o,
                               cudaStream_t st)
{
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    tc_fill_config(cfg, attr, sh, TcGeo<FMT, GROUP>::THREADS, o.pdl, st);
    void* args[] = {const_cast<TcParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, (void*)lbv_tc_kernel<FMT, XT, GROUP>, args);
}

template <int FMT, int XT, int GROUP>
inline cudaError_t tc_prepare_t(const TcShape& sh)
{
    return cudaFuncSetAttribute((void*)lbv_tc_kernel<FMT, XT, GROUP>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sh.smem > kMaxDynSmem ? (int)sh.smem : kMaxDynSmem);
}

template <int FMT, int XT, int GROUP>
inline int tc_max_clusters_t(const TcShape& sh)
{
    if (tc_prepare_t<FMT, XT, GROUP>(sh) != cudaSuccess)
        return 0;
    void* k = (void*)lbv_tc_kernel<FMT, XT, GROUP>;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    TcShape s1 = sh;
    s1.ctas_n = 1;
    tc_fill_config(cfg, attr, s1, TcGeo<FMT, GROUP>::THREADS, false, nullptr);
    int n = 0;
    if (sh.splits > 1) {
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess)
            return 0;
        return n;
    }
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, TcGeo<FMT, GROUP>::THREADS, sh.smem) !=
        cudaSuccess)
        return 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return n * sms;
}

}  // namespace lbv
