// t8_kernel.cuh -- the few-row verify on the 5th-generation tensor cores with
// e4m3 operands: Y[M,N] = X[M,K] . W[K,N], M <= 8, for the g128 formats of
// t8_layout.h (1-bit sign, 2-bit affine).
//
// Why e4m3.  A decoded weight is a small integer code; written to tensor
// memory as an fp16 A operand it costs 2 bytes of tensor-memory store per
// weight, and that store stream bounds a decode-in-registers tcgen05 kernel
// near the legacy mma.sync rate.  As an e4m3 byte the same code costs 1 byte:
// the field (word >> 4s) & (mask << f) of a packed word reads, byte by byte,
// as the e4m3 value code * 2^(f - 9) (subnormals, continued by the lowest
// normals), so four weights take one LOP3 and no base offset or correction
// term exists.  The activations are the B operand of kind::f8f6f4 as well:
// per 128-K group and row, x * 2^(sig - f) with the power of two that brings
// the group's largest |x * 2^-f| into [2^7, 2^8) is split exactly into three
// e4m3 terms t0 + t1/16 + t2/256, each the leading 4 significant bits of
// what is left (an fp16 or bf16 value has at most 11 significant bits), one
// B row per (term, activation row): N = 32 (24 used).  Products of e4m3
// values are exact and the tensor core sums them in fp32.
//
// Measured on GB300 this kernel is slower than the mma.sync one.  Every group
// stores 4 KB of A and reads back 3 KB of accumulator per warp (the fp16
// group scale has to be applied outside the tensor core), and each decode
// warp runs that store, its wait, the read-back, its wait and the shared
// loads as one serial chain per group, four such warps per scheduler.  It
// is kept as an opt-in, parity-tested path.
//
// Structure (one CTA per SM, 640 threads):
//   * Four warpgroups, each of four decode warps (warp q owns tensor-memory
//     lanes 32q..32q+31 = columns 32q..32q+31 of the warpgroup's tile) and
//     one MMA warp.  A warpgroup takes the tiles t0 + wg, t0 + wg + 4, ... of
//     its cluster and walks each over the CTA's K slice one 128-K group at a
//     time.
//   * Per group: each decode thread loads its column's codes from its
//     warpgroup's ring of bulk-copied stages (one copy per stage of the tile's
//     four quarters; the MMA warp refills a slot once the decode warps have
//     stored the slot's last group), writes 32 e4m3 words to the group's A
//     slot (tcgen05.st), and arrives on the slot's mbarrier; the MMA warp
//     issues four M128 N32 K32 MMAs into the slot's accumulator and commits;
//     one group later the decode threads read the accumulator back
//     (tcgen05.ld) and fold  scale * 2^(9 - sig) * (acc0 + acc1/16 + acc2/256)
//     (+ bias * row sum) into eight fp32 row sums, two rows per fp32x2 op.
//     Two A slots and two accumulators per warpgroup (4 x 128 tensor-memory
//     columns).
//   * K is split across the S CTAs of a cluster.  Tile i of the cluster
//     belongs to rank i % S; the other ranks send their partial rows into the
//     owner's shared memory with asynchronous stores counted on its mbarrier
//     for that tile; the owner parks its own partial until it finishes its
//     next tile, then adds the S partials in rank order (deterministic) and
//     writes Y or updates the argmax keys.
//   * Prologue: the X slice is staged (bulk copies, after
//     griddepcontrol.wait), optionally sign-flipped and rotated (FWHT-128,
//     the fused head), then split into the B tiles and the per-(group, row)
//     constants (2^(9 - sig), row sum), one warp per group; packed weights
//     start streaming before the wait.  Every wait is bounded; a wait
//     that gives up sets the plan's status word and lets the kernel end.
#pragma once

#include "t8_internal.h"
#include "verify_kernel.cuh"

namespace lbv {

namespace t8 {

// ---------------------------------------------------------------------------
// tcgen05 / cluster helpers

__device__ __forceinline__ void tc_fence_before()
{
    asm volatile("tcgen05.fence::before_thread_sync;\n" ::: "memory");
}

__device__ __forceinline__ void tc_fence_after()
{
    asm volatile("tcgen05.fence::after_thread_sync;\n" ::: "memory");
}

// 32 consecutive tensor-memory columns of this warp's 32 lanes.
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

// Columns 0..23 of an accumulator (term j, row m at column 8j + m).  The
// loads and their wait are one asm statement, so no use of the registers can
// be scheduled before the wait.
__device__ __forceinline__ void tmem_ld24(uint32_t taddr, float (&d)[24])
{
    uint32_t r[24];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,"
        "%14,%15}, [%24];\n"
        "tcgen05.ld.sync.aligned.32x32b.x8.b32 {%16,%17,%18,%19,%20,%21,%22,%23}, [%25];\n"
        "tcgen05.wait::ld.sync.aligned;\n"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]),
          "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]),
          "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23])
        : "r"(taddr), "r"(taddr + 16u)
        : "memory");
#pragma unroll
    for (int i = 0; i < 24; ++i)
        d[i] = __uint_as_float(r[i]);
}

// Shared-memory matrix descriptor, K-major, no swizzle: core matrices of 8
// rows x 16 bytes, LBO = 128 bytes between the two core matrices along K,
// SBO = 256 bytes between the four along N.
__device__ __forceinline__ uint64_t b_desc(uint32_t addr)
{
    return (uint64_t)((addr >> 4) & 0x3FFFu) | ((uint64_t)(128u >> 4) << 16) |
           ((uint64_t)(256u >> 4) << 32) | (1ull << 46);
}

// Instruction descriptor, kind::f8f6f4: fp32 accumulator, A and B e4m3, both
// K-major, N = 32, M = 128.
constexpr uint32_t kIdesc = (1u << 4) | ((32u >> 3) << 17) | ((128u >> 4) << 24);

// Four M128 N32 K32 MMAs of one group into accumulator `d` (the first one
// overwrites it), then a commit that arrives on `bar` once they complete.
// Run by one elected lane of a converged warp.
__device__ __forceinline__ void mma_group(uint32_t d, uint32_t a, uint64_t b0, uint32_t bar)
{
    asm volatile(
        "{\n .reg .pred e;\n elect.sync _|e, 0xffffffff;\n"
        " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %6, 0;\n"
        " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%7], %3, %6, 1;\n"
        " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%8], %4, %6, 1;\n"
        " @e tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%9], %5, %6, 1;\n"
        " @e tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%10];\n}\n"
        ::"r"(d), "r"(a), "l"(b0), "l"(b0 + 64u), "l"(b0 + 128u), "l"(b0 + 192u), "r"(kIdesc),
        "r"(a + 8u), "r"(a + 16u), "r"(a + 24u), "r"(bar)
        : "memory");
}

// Two fp32 values as one 64-bit register pair (lo first), and the packed
// fp32x2 arithmetic of sm_100+: each half is rounded like its scalar op.
__device__ __forceinline__ uint64_t f2pack(float lo, float hi)
{
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};\n" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}

__device__ __forceinline__ float2 f2unpack(uint64_t v)
{
    float2 r;
    asm("mov.b64 {%0, %1}, %2;\n" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}

__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c)
{
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;\n" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

__device__ __forceinline__ uint64_t fmul2(uint64_t a, uint64_t b)
{
    uint64_t d;
    asm("mul.rn.f32x2 %0, %1, %2;\n" : "=l"(d) : "l"(a), "l"(b));
    return d;
}

// Bounded wait with cluster-scope acquire (arrivals from peer CTAs).
__device__ __forceinline__ bool mbar_wait_cluster(uint32_t bar, uint32_t parity,
                                                  uint32_t limit = 1u << 20)
{
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok)
            return true;
        if (i >= 4096u)
            __nanosleep(1000);
    }
    return false;
}

__device__ __forceinline__ uint32_t mapa(uint32_t addr, uint32_t rank)
{
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;\n" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}

__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr)
{
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];\n"
                 ::"r"(cluster_addr)
                 : "memory");
}

// Four fp32 values into a peer CTA's shared memory (16-byte aligned), counted
// on the peer's mbarrier as 16 bytes of its transaction once they land.
__device__ __forceinline__ void st_async_v4(uint32_t cluster_addr, float a, float b, float c,
                                            float d, uint32_t cluster_bar)
{
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.f32 [%0], {%1, %2, %3, %4}, [%5];\n"
        ::"r"(cluster_addr), "f"(a), "f"(b), "f"(c), "f"(d), "r"(cluster_bar)
        : "memory");
}

__device__ __forceinline__ uint32_t cluster_rank()
{
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;\n" : "=r"(r));
    return r;
}

__device__ __forceinline__ void cluster_arrive()
{
    asm volatile("barrier.cluster.arrive.release.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void cluster_wait_acq()
{
    asm volatile("barrier.cluster.wait.acquire.aligned;\n" ::: "memory");
}

// Two fp32 values -> e4m3, round to nearest even, saturating: byte 0 from lo.
__device__ __forceinline__ uint32_t e4m3x2(float lo, float hi)
{
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;\n" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// The two e4m3 values of the low 16 bits (byte 0 -> .x), exactly.
__device__ __forceinline__ float2 e4m3x2_to_f2(uint32_t v)
{
    uint32_t h;
    asm("{\n .reg .b16 t;\n cvt.u16.u32 t, %1;\n cvt.rn.f16x2.e4m3x2 %0, t;\n}\n"
        : "=r"(h)
        : "r"(v));
    const __half2 hh = *reinterpret_cast<const __half2*>(&h);
    return __half22float2(hh);
}

// 2^e as a float for e in [-126, 127].
__device__ __forceinline__ float pow2f(int e)
{
    return __int_as_float((127 + e) << 23);
}

}  // namespace t8

// ---------------------------------------------------------------------------
// Shared-memory carve-up (byte offsets), used by the kernel and by the host's
// size query alike:
//   ring [NS][4 warpgroups][stage] | B tiles [gps * 4][1024] | X rows [8][RS]
//   (unless staged in the ring) | epilogue constants [gps][8] float2 |
//   partial slots [owned][S - 1][128][8] float | mbarriers ring [4][NS],
//   full [4][2], done [4][2], pready [owned], X | misc words [18] | keys [8]
struct T8Carve {
    size_t b, x, ep, part, bars, misc, keys, end;
};

template <int FMT>
__host__ __device__ inline T8Carve t8_carve(int gps, int splits, int owned, int x_in_ring)
{
    constexpr int W = FMT == LBV_FMT_SIGN1_G128 ? 1 : 2;
    constexpr int REC = 32 * ((W == 1 ? 16 : 32) + (W == 1 ? 2 : 4));
    constexpr size_t STAGE_B = (size_t)kT8GroupsPerStage<FMT> * 4 * REC;
    T8Carve c;
    c.b = (size_t)kT8Stages * 4 * STAGE_B;
    const size_t after_b = c.b + (size_t)gps * 4096;
    c.x = x_in_ring ? (size_t)kT8EarlyStages * 4 * STAGE_B : after_b;
    c.ep = after_b + (x_in_ring ? 0 : (size_t)8 * (gps * kT8GroupK * 2 + 16));
    c.part = c.ep + (size_t)gps * 8 * sizeof(float2);
    c.bars = c.part + (splits > 1 ? (size_t)owned * (splits - 1) * 1024 * sizeof(float) : 0);
    c.misc = c.bars + (size_t)(4 * kT8Stages + 16 + owned + 1) * 8;
    c.keys = c.misc + 18 * 4;
    c.end = c.keys + 8 * 8;
    return c;
}

template <int FMT, int XT>
struct T8Kernel {
    static constexpr int W = FMT == LBV_FMT_SIGN1_G128 ? 1 : 2;   // bits per code
    static constexpr int CB = W == 1 ? 16 : 32;                    // code bytes per column-group
    static constexpr int SB = W == 1 ? 2 : 4;                      // side bytes per column-group
    static constexpr int REC = 32 * (CB + SB);                     // record (quarter, group)

    // e4m3 value of the code of group-local k: code * 2^(f - 9), f = fshift(k).
    static __host__ __device__ constexpr int fshift(int k)
    {
        return W == 2 ? 2 * ((k >> 2) & 1) : ((k >> 2) & 3);
    }

    static __device__ __forceinline__ void decode(const uint4 (&c)[CB / 16], uint32_t (&r)[32])
    {
        if constexpr (W == 2) {
            const uint32_t w[8] = {c[0].x, c[0].y, c[0].z, c[0].w, c[1].x, c[1].y, c[1].z, c[1].w};
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                const uint32_t x = w[i], y = x >> 4;
                r[4 * i + 0] = x & 0x03030303u;
                r[4 * i + 1] = x & 0x0C0C0C0Cu;
                r[4 * i + 2] = y & 0x03030303u;
                r[4 * i + 3] = y & 0x0C0C0C0Cu;
            }
        } else {
            const uint32_t w[4] = {c[0].x, c[0].y, c[0].z, c[0].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const uint32_t x = w[i], y = x >> 4;
#pragma unroll
                for (int j = 0; j < 4; ++j) {
                    r[8 * i + j] = x & (0x01010101u << j);
                    r[8 * i + 4 + j] = y & (0x01010101u << j);
                }
            }
        }
    }

    // Ring stage of a warpgroup: the bulk copy of groups g .. g + ngr - 1 of a
    // tile, all four quarters (contiguous in the layout).
    static __device__ __forceinline__ void issue_stage(const T8Params& p, int tile, int g, int ngr,
                                                       uint32_t dst, uint32_t bar)
    {
        const size_t rec = ((size_t)tile * (size_t)p.ngroups + (size_t)g) * 4;
        const uint32_t bytes = (uint32_t)ngr * 4 * REC;
#ifdef LBV_CHECKED
        // checked build: the stage lies inside the packed matrix (else no copy:
        // its waiters give up and the status records both)
        if (tile < 0 || tile >= p.ntiles || g < 0 || ngr < 1 || g + ngr > p.ngroups) {
            atomicOr(p.err, 2u);
            return;
        }
#endif
        mbar_expect_tx(bar, bytes);
        bulk_g2s(dst, p.W + rec * REC, bytes, bar);
    }

    // Stage X[0..M) x [k0, k0 + ks) at xs (row m at xs + m * RS).  Aligned X:
    // thread 0 issues one bulk copy per row (completing on xbar).  Otherwise
    // all threads copy it with plain loads.
    static __device__ __forceinline__ bool stage_x(const T8Params& p, unsigned char* xs, int RS,
                                                   uint32_t xbar, int k0, int ks)
    {
        const uint16_t* X = reinterpret_cast<const uint16_t*>(p.X);
#ifdef LBV_CHECKED
        // checked build: the slice lies inside K and fits the row buffer
        if (k0 < 0 || ks < 0 || k0 + ks > p.K || ks * 2 > RS || p.M < 1 || p.M > 8) {
            if (threadIdx.x == 0)
                atomicOr(p.err, 2u);
            return false;
        }
#endif
        if (p.x_vec) {
            if (threadIdx.x == 0) {
                mbar_expect_tx(xbar, (uint32_t)(p.M * ks * 2));
                for (int m = 0; m < p.M; ++m)
                    bulk_g2s(smem_u32(xs + (size_t)m * RS), X + (size_t)m * p.ldx + k0,
                             (uint32_t)(ks * 2), xbar);
            }
            return true;
        }
        for (int i = threadIdx.x; i < p.M * ks; i += kT8Threads) {
            const int m = i / ks, k = i - m * ks;
            reinterpret_cast<uint16_t*>(xs + (size_t)m * RS)[k] = X[(size_t)m * p.ldx + k0 + k];
        }
        return false;
    }

    static __device__ __forceinline__ float x_at(const unsigned char* xs, int RS, int m, int k)
    {
        const uint16_t u = reinterpret_cast<const uint16_t*>(xs + (size_t)m * RS)[k];
        if constexpr (XT == LBV_F16)
            return __half2float(__ushort_as_half(u));
        else
            return __uint_as_float((uint32_t)u << 16);
    }

    // Eight X values of row m at slice-local k0 (16-byte aligned), as floats.
    static __device__ __forceinline__ void x8_at(const unsigned char* xs, int RS, int m, int k0,
                                                 float (&x)[8])
    {
        const uint4 v = *reinterpret_cast<const uint4*>(xs + (size_t)m * RS + (size_t)k0 * 2);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            if constexpr (XT == LBV_F16) {
                const float2 f = f16pair(w[i]);
                x[2 * i] = f.x;
                x[2 * i + 1] = f.y;
            } else {
                x[2 * i] = __uint_as_float(w[i] << 16);
                x[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
            }
        }
    }

    // B tiles and the per-(group, row) epilogue constants from the staged
    // (rotated) X, one warp per group g of the slice: lane L takes row
    // m = L % 8 and K tile L / 8 of the group (32 values).  For each (g, m)
    // with m < M the warp finds the group's max |x * 2^-f| and the power of
    // two 2^sig that brings it into [2^7, 2^8) (sig = 0 for a zero group,
    // clamped to [-116, 120]); v = x * 2^(sig - f) is split as
    // t0 + t1/16 + t2/256 with each term v, 16 (v - t0), ... truncated to its
    // leading 4 significant bits (the fp32 pattern masked): exact for the 11
    // significant bits of an fp16 (8 of a bf16) value, every term below 256.
    // ep[g] = (U_0..U_7, R_0..R_7): U_m = 2^(9 - sig), R_m the row sum of the
    // group's x in fp32 (negated for sign1, whose fold is s (2 acc - R)); rows >= M
    // and the fourth term (B rows 24..31) are zeros.
    static __device__ void build_b(const unsigned char* xs, int RS, int M, int gcnt,
                                   unsigned char* bsm, float* ep)
    {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int m = lane & 7, jq = lane >> 3;
        for (int g = warp; g < gcnt; g += kT8Threads / 32) {
            const int k0 = g * 128 + jq * 32;                        // slice-local
            float x[32];
            float mx = 0.f, sum = 0.f;
            if (m < M) {
#pragma unroll
                for (int i = 0; i < 4; ++i)
                    x8_at(xs, RS, m, k0 + 8 * i, *reinterpret_cast<float(*)[8]>(x + 8 * i));
#pragma unroll
                for (int i = 0; i < 8; ++i) {                        // quads: one f each
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        a = fmaxf(a, fabsf(x[4 * i + e]));
                        sum += x[4 * i + e];
                    }
                    mx = fmaxf(mx, a * t8::pow2f(-fshift(jq * 32 + 4 * i)));
                }
            }
            // the four lanes of row m: K tiles 0..3 of the group, a fixed tree
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
            sum += __shfl_xor_sync(0xffffffffu, sum, 8);
            mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
            sum += __shfl_xor_sync(0xffffffffu, sum, 16);
            int sg = 0;
            if (mx > 0.f && mx == mx) {
                frexpf(mx, &sg);                      // mx = f * 2^sg, f in [0.5, 1)
                sg = max(-116, min(120, 8 - sg));
            }
            uint32_t t[3][8] = {};
            if (m < M) {
#pragma unroll
                for (int e = 0; e < 32; e += 2) {
                    const float c = t8::pow2f(sg - fshift(jq * 32 + e));   // same f for k, k + 1
                    float v0 = x[e] * c, v1 = x[e + 1] * c;
#pragma unroll
                    for (int j = 0; j < 3; ++j) {
                        const float a0 = __uint_as_float(__float_as_uint(v0) & 0xFFF00000u);
                        const float a1 = __uint_as_float(__float_as_uint(v1) & 0xFFF00000u);
                        t[j][e / 4] |= t8::e4m3x2(a0, a1) << (8 * (e % 4));
                        v0 = (v0 - a0) * 16.f;
                        v1 = (v1 - a1) * 16.f;
                    }
                }
            }
            unsigned char* dst = bsm + (size_t)(4 * g + jq) * 1024 + m * 16;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
#pragma unroll
                for (int j = 0; j < 3; ++j)
                    *reinterpret_cast<uint4*>(dst + h * 128 + j * 256) =
                        make_uint4(t[j][4 * h], t[j][4 * h + 1], t[j][4 * h + 2], t[j][4 * h + 3]);
                *reinterpret_cast<uint4*>(dst + h * 128 + 3 * 256) = make_uint4(0u, 0u, 0u, 0u);
            }
            if (jq == 0) {
                ep[g * 16 + m] = m < M ? t8::pow2f(9 - sg) : 0.f;
                ep[g * 16 + 8 + m] = m < M ? (W == 2 ? sum : -sum) : 0.f;
            }
        }
    }

    // Fused head epilogue: the CTA's keys go to the workspace; the CTA that
    // finishes last turns the keys into the rows' argmax columns and logits
    // and leaves the workspace zeroed for the next call.
    static __device__ void amax_finish(const T8Params& p, const unsigned long long* akeys,
                                       unsigned* last)
    {
        const int tid = (int)threadIdx.x;
        if (tid < p.M) {
            const unsigned long long k = akeys[tid];
            if (k)
                atomicMax(p.amax_keys + tid, k);
            __threadfence();
        }
        __syncthreads();
        if (tid == 0) {
            const unsigned total = gridDim.x * gridDim.y;
            *last = atomicAdd(p.amax_done, 1u) == total - 1u;
        }
        __syncthreads();
        if (*last) {
            __threadfence();
            if (tid < p.M) {
                const unsigned long long k = atomicExch(p.amax_keys + tid, 0ull);
                p.amax_idx[tid] = (int)(0xffffffffu - (uint32_t)k);
                if (p.amax_val)
                    p.amax_val[tid] = amax_key_value(k);
            }
            if (tid == 0)
                atomicExch(p.amax_done, 0u);
        }
    }

    static __device__ void run(const T8Params& p, unsigned char* smem)
    {
        constexpr int NS = kT8Stages, NEARLY = kT8EarlyStages, GPS = kT8GroupsPerStage<FMT>;
        constexpr int STAGE_B = GPS * 4 * REC;                   // a warpgroup's stage
        const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
        const int S = p.splits;
        const int rank = S > 1 ? (int)t8::cluster_rank() : 0;
        const int cy = blockIdx.y, ny = gridDim.y;
        const int g0 = rank * p.gps;
        const int gcnt = min(p.gps, p.ngroups - g0);            // >= 1 (host guarantees)
        const int ks = gcnt * kT8GroupK;
        const int t0 = (int)(((long long)p.ntiles * cy) / ny);
        const int t1 = (int)(((long long)p.ntiles * (cy + 1)) / ny);
        const int ntc = t1 - t0;

        // shared memory carve-up (t8_carve)
        const T8Carve cv = t8_carve<FMT>(p.gps, S, p.owned, p.x_in_ring);
        unsigned char* ring = smem;
        unsigned char* bsm = smem + cv.b;
        const int RS = ks * 2 + 16;
        unsigned char* xs = smem + cv.x;
        float* ep = reinterpret_cast<float*>(smem + cv.ep);
        float* part = reinterpret_cast<float*>(smem + cv.part);
        uint64_t* bars = reinterpret_cast<uint64_t*>(smem + cv.bars);
        // ring[4][NS], full[4][2], done[4][2], pready[owned], xbar
        const uint32_t bar_ring = smem_u32(bars);
        const uint32_t bar_full = bar_ring + 4 * NS * 8;
        const uint32_t bar_done = bar_full + 8 * 8;
        const uint32_t bar_pready = bar_done + 8 * 8;
        const uint32_t xbar = bar_pready + (uint32_t)p.owned * 8;
        unsigned* misc = reinterpret_cast<unsigned*>(smem + cv.misc);
        uint32_t* tslot = misc;                      // [0]: tensor-memory base
        unsigned* last = misc + 1;                   // [1]: last-CTA flag
        unsigned long long* akeys = reinterpret_cast<unsigned long long*>(smem + cv.keys);
        {
            // the carve-up must end inside the launch's dynamic shared memory
            uint32_t dyn;
            asm volatile("mov.u32 %0, %%dynamic_smem_size;\n" : "=r"(dyn));
            if (cv.end > (size_t)dyn) {
                if (threadIdx.x == 0)
                    atomicOr(p.err, 2u);
                return;                              // uniform: every CTA has the same carve-up
            }
        }

        const bool is_issuer = warp >= kT8DecodeWarps;
        const int wg = is_issuer ? warp - kT8DecodeWarps : warp >> 2;
        const int q = warp & 3;
        const int ntw = wg < ntc ? (ntc - wg + 3) / 4 : 0;       // tiles of this warpgroup
        const int nst_tile = (gcnt + GPS - 1) / GPS;             // ring stages per tile
        const int nstage = ntw * nst_tile;                       // this warpgroup's stages
        const int total = ntw * gcnt;                            // groups of this warpgroup

        if (tid == 0) {
            for (int i = 0; i < 4 * NS; ++i)
                mbar_init(bar_ring + i * 8, 1);
            for (int i = 0; i < 8; ++i) {
                mbar_init(bar_full + i * 8, 4);
                mbar_init(bar_done + i * 8, 1);
            }
            for (int i = 0; i < p.owned; ++i)
                mbar_init(bar_pready + i * 8, 1);
            mbar_init(xbar, 1);
            mbar_init_fence();
            // an owned tile's slot completes once the other ranks' partial
            // rows (128 columns x 8 rows each) have landed
            for (int i = 0; i < p.owned; ++i)
                mbar_expect_tx(bar_pready + i * 8, (uint32_t)(S - 1) * 128u * 8u * 4u);
        }
        if (tid < 8)
            akeys[tid] = 0ull;
        if (warp == kT8DecodeWarps) {                // the first MMA warp owns the allocation
            asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], 512;\n"
                         ::"r"(smem_u32(tslot)) : "memory");
            asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;\n" ::: "memory");
        }
        t8::tc_fence_before();
        __syncthreads();
        t8::tc_fence_after();
        const uint32_t tmem = *tslot;
        if (S > 1)
            t8::cluster_arrive();                    // barriers initialised (release)

        // ring stages of a warpgroup, issued by its MMA warp: stage s -> (tile,
        // first group, groups), slot s % NS
        auto issue_s = [&](int s) {
            const int ti = s / nst_tile, g = (s - ti * nst_tile) * GPS;
            issue_stage(p, t0 + wg + 4 * ti, g0 + g, min(GPS, gcnt - g),
                        smem_u32(ring + ((size_t)(s % NS) * 4 + wg) * STAGE_B),
                        bar_ring + (wg * NS + s % NS) * 8);
        };
        bool ok = true;
        int issued = 0;                              // stages the warpgroup's MMA warp issued
        if (is_issuer && lane == 0)
            for (; issued < min(NEARLY, nstage); ++issued)
                issue_s(issued);

        griddep_wait();
        const bool x_async = stage_x(p, xs, RS, xbar, g0 * kT8GroupK, ks);
        if (!p.x_in_ring && is_issuer && lane == 0)
            for (; issued < min(NS, nstage); ++issued)
                issue_s(issued);
        __syncthreads();
        bool x_ok = true;
        if (x_async && !mbar_try(xbar, 0) && !mbar_wait(xbar, 0))
            x_ok = false;
        const bool all_x = __syncthreads_and(x_ok);
        if (!all_x && tid == 0)
            atomicOr(p.err, 1u);
        if (p.rot && all_x) {
            if (p.signs) {
                flip_signs(p.signs, xs, RS, p.M, g0 * kT8GroupK, ks, tid, kT8Threads);
                __syncthreads();
            }
            rotate_x<XT>(smem_u32(xs), RS, gcnt, warp, kT8Threads / 32, lane);
            __syncthreads();
        }
        build_b(xs, RS, p.M, gcnt, bsm, ep);
        fence_proxy_async_smem();                    // B (generic writes) before the MMAs read it
        __syncthreads();
        griddep_launch_dependents();
        if (S > 1)
            t8::cluster_wait_acq();                  // every peer runs, its barriers initialised
        if (p.x_in_ring && is_issuer && lane == 0)
            for (; issued < min(NS, nstage); ++issued)
                issue_s(issued);
        issued = min(NS, nstage);                    // what the MMA warp issued; refills go on from here

        const uint32_t tm_wg = tmem + (uint32_t)(wg * 128);
        if (is_issuer) {
            // ---- MMA warp: one group per A slot, alternating slots.  Once
            // the four decode warps have stored the last group of a ring
            // stage they have read all of it, so the MMA warp refills its slot.
            int done_n = 0;
            int g = 0;
            for (int c = 0; c < total && ok; ++c) {
                const int slot = c & 1;
                if (!mbar_wait(bar_full + (wg * 2 + slot) * 8, (uint32_t)((c >> 1) & 1))) {
                    ok = false;
                    break;
                }
                t8::tc_fence_after();
                t8::mma_group(tm_wg + 64u + (uint32_t)slot * 32u, tm_wg + (uint32_t)slot * 32u,
                              t8::b_desc(smem_u32(bsm) + (uint32_t)g * 4096u),
                              bar_done + (wg * 2 + slot) * 8);
                // after the MMAs, so that a full copy queue stalls only the refill
                if ((g % GPS) == GPS - 1 || g == gcnt - 1) {
                    if (lane == 0 && issued < nstage)
                        issue_s(issued);
                    issued = min(issued + 1, nstage);
                }
                done_n = c + 1;
                if (++g == gcnt)
                    g = 0;
            }
            // the last commits complete before tensor memory is released
            for (int c = max(0, done_n - 2); c < done_n; ++c)
                if (!mbar_wait(bar_done + (wg * 2 + (c & 1)) * 8, (uint32_t)((c >> 1) & 1)))
                    ok = false;
            // every stage issued has landed before the CTA exits (the last NS
            // issued; an earlier stage of a slot was read before its slot was
            // refilled)
            for (int st = max(0, issued - NS); st < issued; ++st)
                if (!mbar_wait(bar_ring + (wg * NS + st % NS) * 8, (uint32_t)((st / NS) & 1)))
                    ok = false;

        } else {
            // ---- decode warp
            const uint32_t ta = tm_wg | ((uint32_t)(q * 32) << 16);
            uint64_t Y2[4];                          // rows 2i, 2i + 1 as packed pairs
#pragma unroll
            for (int i = 0; i < 4; ++i)
                Y2[i] = 0ull;
            uint32_t sb_prev = 0u;                   // side word (fp16 scale, bias) of the group behind
            float pend[8];                           // an owned tile's own partial, parked
            int pend_li = -1;
            int consumed = 0;                        // ring stages read
            int ge = 0, te = 0;                      // epilogue cursor: group, tile index
            uint4 cw[CB / 16];                       // codes of the next group to decode
            uint32_t sb_nx = 0u;                     // converted where it is used, one group later
            // loads group gl's codes and side values (waiting for its stage
            // first when gl opens one)
            auto load_group = [&](int gl) -> bool {
                const int slot_r = consumed % NS;
                const int gi = gl % GPS;
                if (gi == 0 && !mbar_wait(bar_ring + (wg * NS + slot_r) * 8,
                                          (uint32_t)((consumed / NS) & 1),
                                          p.wait_limit ? p.wait_limit : 1u << 20))
                    return false;
                const unsigned char* rec =
                    ring + ((size_t)slot_r * 4 + wg) * STAGE_B + (size_t)(gi * 4 + q) * REC;
#pragma unroll
                for (int i = 0; i < CB / 16; ++i)
                    cw[i] = *reinterpret_cast<const uint4*>(rec + i * 512 + lane * 16);
                if constexpr (W == 2)
                    sb_nx = *reinterpret_cast<const uint32_t*>(rec + CB * 32 + lane * 4);
                else
                    sb_nx = *reinterpret_cast<const uint16_t*>(rec + CB * 32 + lane * 2);
                if (gi == GPS - 1 || gl == gcnt - 1)
                    ++consumed;
                return true;
            };
            // folds accumulator e (group ge of tile te) into Y; at a tile's last
            // group, with a K split, hands the partial to the owner, or (owner)
            // parks it and reduces the tile parked before, whose partials
            // arrived a tile ago
            auto epilogue = [&](int e) -> bool {
                // the group's constants first: their shared loads then overlap the
                // wait for the MMAs and the accumulator read instead of following it
                const float4* e4 = reinterpret_cast<const float4*>(ep + ge * 16);
                const float4 Ua = e4[0], Ub = e4[1], Ra = e4[2], Rb = e4[3];
                if (!mbar_wait(bar_done + (wg * 2 + (e & 1)) * 8, (uint32_t)((e >> 1) & 1)))
                    return false;
                t8::tc_fence_after();
                float d[24];
                t8::tmem_ld24(ta + 64u + (uint32_t)((e & 1) * 32), d);
                const uint64_t U2[4] = {t8::f2pack(Ua.x, Ua.y), t8::f2pack(Ua.z, Ua.w),
                                        t8::f2pack(Ub.x, Ub.y), t8::f2pack(Ub.z, Ub.w)};
                const uint64_t R2[4] = {t8::f2pack(Ra.x, Ra.y), t8::f2pack(Ra.z, Ra.w),
                                        t8::f2pack(Rb.x, Rb.y), t8::f2pack(Rb.z, Rb.w)};
                const uint64_t k16 = t8::f2pack(1.f / 16.f, 1.f / 16.f);
                const uint64_t k256 = t8::f2pack(1.f / 256.f, 1.f / 256.f);
                const float2 sb = f16pair(sb_prev);   // (scale, bias); sign1: (scale, 0)
                const uint64_t s2 = t8::f2pack(sb.x, sb.x);
                const uint64_t b2 = W == 2 ? t8::f2pack(sb.y, sb.y) : t8::f2pack(2.f, 2.f);
                // rows 2i, 2i + 1 at once:
                //   acc = U (d0 + d1 / 16 + d2 / 256)  (the three terms of X)
                //   affine2: Y += s acc + b R;  sign1: Y += s (2 acc - R)
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    const uint64_t t0 = t8::f2pack(d[2 * i], d[2 * i + 1]);
                    const uint64_t t1 = t8::f2pack(d[8 + 2 * i], d[9 + 2 * i]);
                    const uint64_t t2 = t8::f2pack(d[16 + 2 * i], d[17 + 2 * i]);
                    const uint64_t acc =
                        t8::fmul2(U2[i], t8::ffma2(t2, k256, t8::ffma2(t1, k16, t0)));
                    if constexpr (W == 2)
                        Y2[i] = t8::ffma2(s2, acc, t8::ffma2(b2, R2[i], Y2[i]));
                    else
                        Y2[i] = t8::ffma2(s2, t8::ffma2(b2, acc, R2[i]), Y2[i]);
                }
                if (++ge == gcnt) {
                    const int li = wg + 4 * te;
                    float Y[8];
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const float2 v = t8::f2unpack(Y2[i]);
                        Y[2 * i] = v.x;
                        Y[2 * i + 1] = v.y;
                    }
                    if (S == 1) {
                        emit(p, t0 + li, q * 32 + lane, lane, Y, akeys);
                    } else if (li % S != rank) {
                        send_partial(p, li, q * 32 + lane, rank, Y, part, bar_pready);
                    } else {
                        if (pend_li >= 0)
                            reduce_emit(p, t0 + pend_li, pend_li, q * 32 + lane, lane, rank, pend,
                                        part, bar_pready, akeys, ok);
                        pend_li = li;
#pragma unroll
                        for (int m = 0; m < 8; ++m)
                            pend[m] = Y[m];
                    }
                    ge = 0;
                    ++te;
#pragma unroll
                    for (int i = 0; i < 4; ++i)
                        Y2[i] = 0ull;
                }
                return true;
            };
            // Per group c: decode (codes loaded one group ahead), tensor-memory
            // store, arrive (the MMAs of c run meanwhile), load group c + 1,
            // then the epilogue of group c - 1.
            if (total > 0 && !load_group(0))
                ok = false;
            int g = 0;                               // decode cursor (slice-local group)
            for (int c = 0; c < total && ok; ++c) {
                uint32_t r[32];
                decode(cw, r);
                t8::tmem_st32(ta + (uint32_t)((c & 1) * 32), r);
                t8::tmem_wait_st();
                t8::tc_fence_before();
                __syncwarp();
                if (lane == 0)
                    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];\n"
                                 ::"r"(bar_full + (wg * 2 + (c & 1)) * 8) : "memory");
                const uint32_t sb_c = sb_nx;
                if (++g == gcnt)
                    g = 0;
                const bool loaded = c + 1 >= total || load_group(g);
                if (!loaded) {
                    ok = false;
                    break;
                }
                if (c >= 1 && !epilogue(c - 1)) {
                    ok = false;
                    break;
                }
                sb_prev = sb_c;
            }
            if (ok && total > 0 && !epilogue(total - 1))
                ok = false;
            if (pend_li >= 0 && ok)
                reduce_emit(p, t0 + pend_li, pend_li, q * 32 + lane, lane, rank, pend, part,
                            bar_pready, akeys, ok);
        }
        if (!ok && lane == 0)
            atomicOr(p.err, 1u);
        t8::tc_fence_before();
        __syncthreads();
        t8::tc_fence_after();
        if (p.amax_keys)
            amax_finish(p, akeys, last);
        if (warp == kT8DecodeWarps)
            asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, 512;\n" ::"r"(tmem)
                         : "memory");
        if (S > 1) {
            // no peer still writes into this CTA's shared memory when it exits
            t8::cluster_arrive();
            t8::cluster_wait_acq();
        }
    }

    // Rows m of column n = 128 * tile + col: Y (when stored) and the CTA's
    // argmax keys.
    static __device__ __forceinline__ void emit(const T8Params& p, int tile, int col, int lane,
                                                const float (&y)[8], unsigned long long* akeys)
    {
        const int n = tile * kT8TileN + col;
        if (p.store_y && n < p.N) {
#pragma unroll
            for (int m = 0; m < 8; ++m)
                if (m < p.M)
                    p.Y[(size_t)m * p.ldy + n] = y[m];
        }
        if (p.amax_keys) {
#pragma unroll
            for (int m = 0; m < 8; ++m) {
                if (m >= p.M)
                    break;
                unsigned long long k = n < p.N ? amax_key(y[m], n) : 0ull;
#pragma unroll
                for (int s = 16; s >= 1; s >>= 1) {
                    const unsigned long long o = __shfl_xor_sync(0xffffffffu, k, s);
                    k = o > k ? o : k;
                }
                if (lane == 0 && k)
                    atomicMax(akeys + m, k);
            }
        }
    }

    // K split: cluster tile li belongs to rank li % S, at slot li / S.  A
    // non-owner writes its partial rows (all 8, column-major) into the
    // owner's slot for its rank (distributed shared memory) with asynchronous
    // stores that count on the owner's mbarrier of that tile.
    static __device__ __forceinline__ void send_partial(const T8Params& p, int li, int col,
                                                        int rank, const float (&y)[8],
                                                        const float* part, uint32_t bar_pready)
    {
        const int S = p.splits;
        const int owner = li % S, j = li / S;
        const int si = rank < owner ? rank : rank - 1;
        const uint32_t base = smem_u32(part + ((size_t)(j * (S - 1) + si) * 128 + col) * 8);
        const uint32_t rbase = t8::mapa(base, (uint32_t)owner);
        const uint32_t rbar = t8::mapa(bar_pready + (uint32_t)j * 8, (uint32_t)owner);
        t8::st_async_v4(rbase, y[0], y[1], y[2], y[3], rbar);
        t8::st_async_v4(rbase + 16u, y[4], y[5], y[6], y[7], rbar);
    }

    // The owner of cluster tile li: wait for the other slices' partials, add
    // the S partials in rank order (deterministic), emit.
    static __device__ __forceinline__ void reduce_emit(const T8Params& p, int tile, int li, int col,
                                                       int lane, int rank, const float (&own)[8],
                                                       const float* part, uint32_t bar_pready,
                                                       unsigned long long* akeys, bool& ok)
    {
        const int S = p.splits, j = li / S;
        if (!t8::mbar_wait_cluster(bar_pready + (uint32_t)j * 8, 0)) {
            ok = false;
            return;
        }
        float acc[8];
#pragma unroll
        for (int m = 0; m < 8; ++m)
            acc[m] = 0.f;
        for (int rk = 0; rk < S; ++rk) {
            if (rk == rank) {
#pragma unroll
                for (int m = 0; m < 8; ++m)
                    acc[m] += own[m];
            } else {
                const int si = rk < rank ? rk : rk - 1;
                const float4* src =
                    reinterpret_cast<const float4*>(part + ((size_t)(j * (S - 1) + si) * 128 + col) * 8);
                const float4 lo = src[0], hi = src[1];
                acc[0] += lo.x;
                acc[1] += lo.y;
                acc[2] += lo.z;
                acc[3] += lo.w;
                acc[4] += hi.x;
                acc[5] += hi.y;
                acc[6] += hi.z;
                acc[7] += hi.w;
            }
        }
        emit(p, tile, col, lane, acc, akeys);
    }
};

template <int FMT, int XT>
__global__ void __launch_bounds__(kT8Threads, 1) lbv_t8_kernel(const __grid_constant__ T8Params p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    T8Kernel<FMT, XT>::run(p, smem);
}

// Dense fp16 dequant of the record layout (test export): one thread per
// (tile, quarter, group, column), through the kernel's own decode (e4m3 bytes
// read back as codes): W[k][n] = s * code + b rounded once to fp16 (affine2),
// +-s (sign1).
template <int FMT>
__global__ void __launch_bounds__(256) lbv_t8_dequant_kernel(const uint8_t* Wp, int K, int N,
                                                             int ntiles, int ngroups, uint16_t* W)
{
    using Kern = T8Kernel<FMT, LBV_F16>;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (long long)ntiles * 4 * ngroups * 32)
        return;
    const int lane = (int)(idx & 31);
    const long long rec_i = idx >> 5;                // (tile * ngroups + g) * 4 + q
    const int q = (int)(rec_i % 4);
    const long long tg = rec_i / 4;
    const int g = (int)(tg % ngroups);
    const int n = (int)(tg / ngroups) * kT8TileN + q * 32 + lane;
    if (n >= N)
        return;
    const uint8_t* rec = Wp + (size_t)rec_i * Kern::REC;
    uint4 cw[Kern::CB / 16];
    for (int i = 0; i < Kern::CB / 16; ++i)
        cw[i] = reinterpret_cast<const uint4*>(rec + i * 512)[lane];
    uint32_t r[32];
    Kern::decode(cw, r);
    const uint16_t* sd = reinterpret_cast<const uint16_t*>(rec + 32 * Kern::CB + lane * Kern::SB);
    for (int c = 0; c < 32; ++c)
        for (int b = 0; b < 4; b += 2) {
            const float2 v = t8::e4m3x2_to_f2(r[c] >> (8 * b));
            for (int h = 0; h < 2; ++h) {
                const int kl = 4 * c + b + h, k = g * kT8GroupK + kl;
                if (k >= K)
                    continue;
                const float code = (h ? v.y : v.x) * t8::pow2f(9 - Kern::fshift(kl));
                uint16_t out;
                if constexpr (FMT == LBV_FMT_SIGN1_G128) {
                    out = code != 0.f ? sd[0] : (uint16_t)(sd[0] ^ 0x8000u);
                } else {
                    const double sc = (double)__half2float(__ushort_as_half(sd[0]));
                    const double bi = (double)__half2float(__ushort_as_half(sd[1]));
                    out = __half_as_ushort(__double2half(sc * (double)code + bi));
                }
                W[(size_t)k * N + n] = out;
            }
        }
}

template <int FMT>
cudaError_t t8_dequant_t(const uint8_t* Wp, int K, int N, int ntiles, int ngroups, uint16_t* W,
                         cudaStream_t st)
{
    const long long total = (long long)ntiles * 4 * ngroups * 32;
    lbv_t8_dequant_kernel<FMT><<<(unsigned)((total + 255) / 256), 256, 0, st>>>(Wp, K, N, ntiles,
                                                                               ngroups, W);
    return cudaGetLastError();
}

// Shared-memory bytes of a launch shape (the kernel's carve-up).
template <int FMT>
__host__ __device__ inline size_t t8_smem_bytes_t(int gps, int splits, int owned, int x_in_ring)
{
    return t8_carve<FMT>(gps, splits, owned, x_in_ring).end;
}

// Whether the X rows of a slice fit in the ring stages issued after the
// prologue.
template <int FMT>
__host__ __device__ inline bool t8_x_fits_ring(int gps)
{
    constexpr int W = FMT == LBV_FMT_SIGN1_G128 ? 1 : 2;
    constexpr int REC = 32 * ((W == 1 ? 16 : 32) + (W == 1 ? 2 : 4));
    constexpr int STAGE_B = kT8GroupsPerStage<FMT> * 4 * REC;
    return (size_t)8 * (gps * kT8GroupK * 2 + 16) <=
           (size_t)(kT8Stages - kT8EarlyStages) * 4 * STAGE_B;
}

template <int FMT, int XT>
cudaError_t t8_launch_t(const T8Shape& sh, const T8Params& p, const LaunchOpts& o,
                        cudaStream_t st)
{
    auto kern = lbv_t8_kernel<FMT, XT>;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sh.splits, (unsigned)sh.ctas_n, 1);
    cfg.blockDim = dim3(kT8Threads, 1, 1);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    int na = 0;
    attr[na].id = cudaLaunchAttributeClusterDimension;
    attr[na].val.clusterDim.x = (unsigned)sh.splits;
    attr[na].val.clusterDim.y = 1;
    attr[na].val.clusterDim.z = 1;
    ++na;
    if (o.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    return cudaLaunchKernelEx(&cfg, kern, p);
}

template <int FMT, int XT>
cudaError_t t8_prepare_t(const T8Shape& sh)
{
    (void)sh;
    return cudaFuncSetAttribute(lbv_t8_kernel<FMT, XT>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                kT8MaxSmem);
}

template <int FMT, int XT>
int t8_max_clusters_t(const T8Shape& sh)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sh.splits, (unsigned)sh.ctas_n, 1);
    cfg.blockDim = dim3(kT8Threads, 1, 1);
    cfg.dynamicSmemBytes = sh.smem;
    cudaLaunchAttribute attr;
    attr.id = cudaLaunchAttributeClusterDimension;
    attr.val.clusterDim.x = (unsigned)sh.splits;
    attr.val.clusterDim.y = 1;
    attr.val.clusterDim.z = 1;
    cfg.attrs = &attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, lbv_t8_kernel<FMT, XT>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        return 0;
    }
    return n;
}

}  // namespace lbv
