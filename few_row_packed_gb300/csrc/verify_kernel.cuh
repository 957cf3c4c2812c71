// verify_kernel.cuh -- the few-row verify kernel, Y[M,N] = X[M,K] . W[K,N],
// M <= 8, for the packed formats of layout.h.
//
// Design (GB300, sm_103a):
//   * One warp owns TPW 16-column tiles and streams their packed codes with
//     one 16-byte non-caching load per lane per chunk, D chunks in flight.
//   * Decode is one LOP3 per A-fragment register: (word_variant & mask) ^ base
//     places a code in the mantissa/exponent field of an fp16 or bf16 whose
//     value is  code_value + c  for a small integer c fixed by the bit position
//     (the pages' "codes turned into exact halves with 0x6400 less 1024" idea,
//     extended to every position of the word).  Only 1-3 shifts per 32-bit
//     word bring the remaining positions into place.
//   * mma.sync m16n8k16 (fp16 or bf16 in, fp32 accumulate): the 16 weight
//     columns are the M side, the M <= 8 activation rows the N side (rows >= M
//     are zero), so each decoded weight is used against every row at once
//     (Ishizuki README, "Kernels written for the verify").
//   * The offsets c enter each group's accumulator as its initial value
//     -sum_k c_k x_k (precomputed per group and row from the staged
//     activations, the "row-sum prep" of the dflash-mlx-bonsai2 README); the
//     group scale (and bias * row sum for affine) is applied in fp32 once per
//     group, so every operand of the tensor core is an exact small integer.
//   * The CTA stages its K slice of X once in shared memory in fragment order.
//     A split of K across a thread-block cluster is reduced through
//     distributed shared memory in a fixed order (deterministic, no workspace).
//   * Weight loads for the first chunks are issued before griddepcontrol.wait,
//     so under programmatic dependent launch they overlap the previous kernel.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <utility>

#include "lbv_internal.h"

namespace lbv {

namespace cg = cooperative_groups;

template <int FMT, int GROUP>
struct Traits;

template <>
struct Traits<LBV_FMT_SIGN1_G128, 128> {
    static constexpr int CHUNK_K = 256, KT = 16, W = 1, GPC = 2, KTG = 8, SIDE_W = 2;
    static constexpr bool AFFINE = false;
};
template <int G>
struct Traits<LBV_FMT_AFFINE2, G> {
    static constexpr int CHUNK_K = 128, KT = 8, W = 2, GPC = 128 / G, KTG = G / 16,
                         SIDE_W = 2 * (128 / G);
    static constexpr bool AFFINE = true;
};
template <>
struct Traits<LBV_FMT_Q4_0, 32> {
    static constexpr int CHUNK_K = 64, KT = 4, W = 4, GPC = 2, KTG = 2, SIDE_W = 2;
    static constexpr bool AFFINE = false;
};

// ---------------------------------------------------------------------------
// Decode specification of slot s of a word: shift the word (positive = left),
// then keep the W-bit field at `target` (and target + 16) and XOR `base`.
// The resulting fp16/bf16 value is  code_value + c.
struct DecSpec {
    int shift;
    int target;
    uint32_t base;   // 16-bit pattern, replicated into both halves
    int c;
};

// 1-bit sign: value = w + c with w = +-1 (bit 1 -> +1).
//   fp16 targets: 15 (base -1.0, c 0), 14 (0, 1), 10 (2.0, 3), 9..5 (2^(11-j), 2^(11-j)+1)
//   bf16 targets: 15 (-1.0, 0), 14 (0, 1), 7 (2.0, 3), 6..2 (2^(8-j), 2^(8-j)+1)
__host__ __device__ constexpr DecSpec sign1_spec(int xt, int s)
{
    if (xt == LBV_F16) {
        const int sh = (s <= 4) ? 5 : (s >= 11 && s <= 13) ? -3 : 0;
        const int j = s + sh;
        return j == 15   ? DecSpec{sh, j, 0xBC00u, 0}
               : j == 14 ? DecSpec{sh, j, 0x0000u, 1}
               : j == 10 ? DecSpec{sh, j, 0x4000u, 3}
               : j == 9  ? DecSpec{sh, j, 0x4400u, 5}
               : j == 8  ? DecSpec{sh, j, 0x4800u, 9}
               : j == 7  ? DecSpec{sh, j, 0x4C00u, 17}
               : j == 6  ? DecSpec{sh, j, 0x5000u, 33}
                         : DecSpec{sh, j, 0x5400u, 65};   // j == 5
    } else {
        const int sh = (s <= 1) ? 5 : (s >= 8 && s <= 13) ? -6 : 0;
        const int j = s + sh;
        return j == 15   ? DecSpec{sh, j, 0xBF80u, 0}
               : j == 14 ? DecSpec{sh, j, 0x0000u, 1}
               : j == 7  ? DecSpec{sh, j, 0x4000u, 3}
               : j == 6  ? DecSpec{sh, j, 0x4080u, 5}
               : j == 5  ? DecSpec{sh, j, 0x4100u, 9}
               : j == 4  ? DecSpec{sh, j, 0x4180u, 17}
               : j == 3  ? DecSpec{sh, j, 0x4200u, 33}
                         : DecSpec{sh, j, 0x4280u, 65};   // j == 2
    }
}

// 2-bit affine code q at bits 2s: value = q + c.
//   fp16 targets 4 (64.0, c 64), 6 (16.0, 16), 8 (4.0, 4)
//   bf16 targets 1 (64.0, 64), 3 (16.0, 16), 5 (4.0, 4)
__host__ __device__ constexpr DecSpec affine2_spec(int xt, int s)
{
    if (xt == LBV_F16) {
        const int sh = (s <= 1) ? 4 : (s <= 4) ? 0 : -6;
        const int j = 2 * s + sh;
        return j == 4 ? DecSpec{sh, j, 0x5400u, 64}
               : j == 6 ? DecSpec{sh, j, 0x4C00u, 16}
                        : DecSpec{sh, j, 0x4400u, 4};
    } else {
        const int sh = (s <= 2) ? 1 : (s <= 5) ? -5 : -11;
        const int j = 2 * s + sh;
        return j == 1 ? DecSpec{sh, j, 0x4280u, 64}
               : j == 3 ? DecSpec{sh, j, 0x4180u, 16}
                        : DecSpec{sh, j, 0x4080u, 4};
    }
}

// Q4_0 nibble q at bits 4s: value = q + c, one target per dtype.
//   fp16: target 4, base 64.0, c 64;  bf16: target 3, base 16.0, c 16
__host__ __device__ constexpr DecSpec q4_0_spec(int xt, int s)
{
    return xt == LBV_F16 ? DecSpec{4 - 4 * s, 4, 0x5400u, 64} : DecSpec{3 - 4 * s, 3, 0x4180u, 16};
}

template <int FMT>
__host__ __device__ constexpr DecSpec dec_spec(int xt, int s)
{
    return FMT == LBV_FMT_SIGN1_G128 ? sign1_spec(xt, s)
           : FMT == LBV_FMT_AFFINE2  ? affine2_spec(xt, s)
                                     : q4_0_spec(xt, s);
}

template <int FMT, int XT, int S>
__device__ __forceinline__ uint32_t decode(uint32_t w)
{
    constexpr DecSpec d = dec_spec<FMT>(XT, S);
    constexpr int W = Traits<FMT, FMT == LBV_FMT_SIGN1_G128 ? 128 : FMT == LBV_FMT_Q4_0 ? 32 : 64>::W;
    constexpr uint32_t field = (1u << W) - 1u;
    constexpr uint32_t mask = (field << d.target) | (field << (d.target + 16));
    constexpr uint32_t base = d.base | (d.base << 16);
    constexpr int shl = d.shift > 0 ? (d.shift > 31 ? 31 : d.shift) : 0;
    constexpr int shr = d.shift < 0 ? (-d.shift > 31 ? 31 : -d.shift) : 0;
    const uint32_t v = shl ? (w << shl) : shr ? (w >> shr) : w;
    return (v & mask) ^ base;
}

// Offset c of slot s (runtime s: prologue only).
template <int FMT, int XT>
__device__ __forceinline__ float slot_coef(int s)
{
    float c = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i)
        if (i == s)
            c = (float)dec_spec<FMT>(XT, i).c;
    return c;
}

// ---------------------------------------------------------------------------
// Small device helpers

template <int XT>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    if constexpr (XT == LBV_F16) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

__device__ __forceinline__ uint4 ldg_stream16(const uint4* p)
{
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ uint2 ldg_nc8(const void* p)
{
    uint2 r;
    asm volatile("ld.global.nc.v2.u32 {%0,%1}, [%2];\n" : "=r"(r.x), "=r"(r.y) : "l"(p));
    return r;
}

__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

template <int XT>
__device__ __forceinline__ float2 pair_to_float2(uint32_t v)
{
    if constexpr (XT == LBV_F16) {
        __half2 h = *reinterpret_cast<__half2*>(&v);
        return __half22float2(h);
    } else {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
        return __bfloat1622float2(h);
    }
}

__device__ __forceinline__ float2 f16pair(uint32_t v)
{
    __half2 h = *reinterpret_cast<__half2*>(&v);
    return __half22float2(h);
}

template <int NW_>
struct SideBuf {
    uint32_t w[NW_];
};

// ---------------------------------------------------------------------------
// Shared memory carve-up (bytes): xf | corr | rsum (affine) | part
__host__ __device__ inline size_t smem_xf_bytes(int kt, int cps)
{
    return (size_t)cps * kt * 256u;
}

// ---------------------------------------------------------------------------

template <int FMT, int XT, int GROUP, int NW, int TPW>
struct VerifyKernel {
    using T = Traits<FMT, GROUP>;
    static constexpr int D = 4;                    // chunks in flight per warp
    using Side = SideBuf<T::SIDE_W>;

    static __device__ __forceinline__ void load_chunk(const VerifyParams& p, int unit, int chunk,
                                                      int lane, uint4 (&w)[TPW], Side (&s)[TPW])
    {
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl) {
            const int tile = unit * TPW + tl;
            if (tile < p.ntiles) {
                const size_t tc = (size_t)tile * p.nchunks + chunk;
                w[tl] = ldg_stream16(p.codes + tc * 32 + lane);
                const uint8_t* sp = p.side + (tc * 8 + (lane >> 2)) * (T::SIDE_W * 4);
#pragma unroll
                for (int i = 0; i < T::SIDE_W; i += 2) {
                    const uint2 v = ldg_nc8(sp + i * 4);
                    s[tl].w[i] = v.x;
                    s[tl].w[i + 1] = v.y;
                }
            } else {
                w[tl] = make_uint4(0u, 0u, 0u, 0u);
#pragma unroll
                for (int i = 0; i < T::SIDE_W; ++i)
                    s[tl].w[i] = 0u;
            }
        }
    }

    // One k-tile (chunk-local index KTC) of TPW tiles: decode the four A
    // registers of slots 2*ktl and 2*ktl + 1 from the column-g word and the
    // column-(g+8) word of the right half, then one mma per tile.
    template <int KTC>
    static __device__ __forceinline__ void do_ktile(const uint4 (&w)[TPW], uint32_t b0,
                                                    uint32_t b1, float (&acc)[TPW][4])
    {
        constexpr int half = KTC / (T::KT / 2);
        constexpr int ktl = KTC % (T::KT / 2);
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl) {
            const uint32_t wa = half ? w[tl].z : w[tl].x;
            const uint32_t wb = half ? w[tl].w : w[tl].y;
            const uint32_t a0 = decode<FMT, XT, 2 * ktl>(wa);
            const uint32_t a1 = decode<FMT, XT, 2 * ktl>(wb);
            const uint32_t a2 = decode<FMT, XT, 2 * ktl + 1>(wa);
            const uint32_t a3 = decode<FMT, XT, 2 * ktl + 1>(wb);
            mma16816<XT>(acc[tl], a0, a1, a2, a3, b0, b1);
        }
    }

    template <int GI, int... P>
    static __device__ __forceinline__ void do_pairs(std::integer_sequence<int, P...>,
                                                    const uint4 (&w)[TPW], int cl,
                                                    const uint4* __restrict__ xf, int lane,
                                                    float (&acc)[TPW][4])
    {
        (
            [&] {
                constexpr int ktc = GI * T::KTG + 2 * P;
                const uint4 bq = xf[((cl * T::KT + ktc) >> 1) * 32 + lane];
                do_ktile<ktc>(w, bq.x, bq.y, acc);
                do_ktile<ktc + 1>(w, bq.z, bq.w, acc);
            }(),
            ...);
    }

    // One scale group GI of a chunk: accumulate from the group's correction,
    // then y += scale * acc (+ bias * rowsum for affine) in fp32.
    template <int GI>
    static __device__ __forceinline__ void do_group(const uint4 (&w)[TPW], const Side (&s)[TPW],
                                                    int cl, const uint4* __restrict__ xf,
                                                    const float* __restrict__ corr,
                                                    const float* __restrict__ rsum,
                                                    float (&y)[TPW][4], int lane)
    {
        const int t = lane & 3;
        const int gr = cl * T::GPC + GI;
        const float2 I = *reinterpret_cast<const float2*>(corr + gr * 8 + 2 * t);
        float acc[TPW][4];
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl) {
            acc[tl][0] = I.x;
            acc[tl][1] = I.y;
            acc[tl][2] = I.x;
            acc[tl][3] = I.y;
        }
        do_pairs<GI>(std::make_integer_sequence<int, T::KTG / 2>{}, w, cl, xf, lane, acc);
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl) {
            if constexpr (T::AFFINE) {
                const float2 sc = f16pair(s[tl].w[2 * GI]);
                const float2 bi = f16pair(s[tl].w[2 * GI + 1]);
                const float2 R = *reinterpret_cast<const float2*>(rsum + gr * 8 + 2 * t);
                y[tl][0] = fmaf(sc.x, acc[tl][0], fmaf(bi.x, R.x, y[tl][0]));
                y[tl][1] = fmaf(sc.x, acc[tl][1], fmaf(bi.x, R.y, y[tl][1]));
                y[tl][2] = fmaf(sc.y, acc[tl][2], fmaf(bi.y, R.x, y[tl][2]));
                y[tl][3] = fmaf(sc.y, acc[tl][3], fmaf(bi.y, R.y, y[tl][3]));
            } else {
                const float2 sc = f16pair(s[tl].w[GI]);
                y[tl][0] = fmaf(sc.x, acc[tl][0], y[tl][0]);
                y[tl][1] = fmaf(sc.x, acc[tl][1], y[tl][1]);
                y[tl][2] = fmaf(sc.y, acc[tl][2], y[tl][2]);
                y[tl][3] = fmaf(sc.y, acc[tl][3], y[tl][3]);
            }
        }
    }

    template <int... G>
    static __device__ __forceinline__ void do_groups(std::integer_sequence<int, G...>,
                                                     const uint4 (&w)[TPW], const Side (&s)[TPW],
                                                     int cl, const uint4* __restrict__ xf,
                                                     const float* __restrict__ corr,
                                                     const float* __restrict__ rsum,
                                                     float (&y)[TPW][4], int lane)
    {
        (do_group<G>(w, s, cl, xf, corr, rsum, y, lane), ...);
    }

    // One chunk (cl = chunk index within the slice) of TPW tiles.
    static __device__ __forceinline__ void process_chunk(const uint4 (&w)[TPW],
                                                         const Side (&s)[TPW], int cl,
                                                         const uint4* __restrict__ xf,
                                                         const float* __restrict__ corr,
                                                         const float* __restrict__ rsum,
                                                         float (&y)[TPW][4], int lane)
    {
        do_groups(std::make_integer_sequence<int, T::GPC>{}, w, s, cl, xf, corr, rsum, y, lane);
    }

    static __device__ void run(const VerifyParams& p, unsigned char* smem)
    {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int g = lane >> 2, t = lane & 3;
        const int c0 = blockIdx.x * p.cps;
        const int nch = min(p.cps, p.nchunks - c0);   // >= 1 (host guarantees)

        uint4* xf = reinterpret_cast<uint4*>(smem);
        float* corr = reinterpret_cast<float*>(smem + smem_xf_bytes(T::KT, p.cps));
        float* rsum = corr + p.cps * T::GPC * 8;
        float* part = rsum + (T::AFFINE ? p.cps * T::GPC * 8 : 0);

        // this warp's units of TPW tiles
        const int nunits = (p.ntiles + TPW - 1) / TPW;
        const int ustride = gridDim.y * NW;
        const int u0 = blockIdx.y * NW + warp;
        const int nu = (u0 < nunits) ? (nunits - 1 - u0) / ustride + 1 : 0;
        const int Q = nu * nch;

        // Weights are read-only: start streaming before waiting on the
        // previous kernel in the stream.
        uint4 wb[D][TPW];
        Side sb[D][TPW];
        int lq = 0, lu = u0, lc = 0;
#pragma unroll
        for (int d = 0; d < D; ++d) {
            if (lq < Q) {
                load_chunk(p, lu, c0 + lc, lane, wb[d], sb[d]);
                ++lq;
                if (++lc == nch) {
                    lc = 0;
                    lu += ustride;
                }
            }
        }

        griddep_wait();

        // ---- stage X[0..8) x [kb, kb + nch*CHUNK_K) in fragment order ----
        {
            const int kb = c0 * T::CHUNK_K;
            const int p8 = (nch * T::CHUNK_K) / 8;      // 8-element pieces per row
            uint32_t* xw = reinterpret_cast<uint32_t*>(xf);
            const uint16_t* X = reinterpret_cast<const uint16_t*>(p.X);
            for (int i = threadIdx.x; i < 8 * p8; i += NW * 32) {
                const int m = i / p8;
                const int k8 = (i - m * p8) * 8;
                const int kg = kb + k8;
                uint4 v = make_uint4(0u, 0u, 0u, 0u);
                if (m < p.M && kg < p.K) {            // K % 8 == 0: all 8 in range
                    const uint16_t* src = X + (size_t)m * p.ldx + kg;
                    if (p.x_vec) {
                        v = *reinterpret_cast<const uint4*>(src);
                    } else {
                        v.x = (uint32_t)src[0] | ((uint32_t)src[1] << 16);
                        v.y = (uint32_t)src[2] | ((uint32_t)src[3] << 16);
                        v.z = (uint32_t)src[4] | ((uint32_t)src[5] << 16);
                        v.w = (uint32_t)src[6] | ((uint32_t)src[7] << 16);
                    }
                }
                const int kt = k8 >> 4, hi = (k8 >> 3) & 1;
                const int base = (((kt >> 1) * 32 + 4 * m) * 4) + (kt & 1) * 2 + hi;
                xw[base + 0] = v.x;
                xw[base + 4] = v.y;
                xw[base + 8] = v.z;
                xw[base + 12] = v.w;
            }
        }
        __syncthreads();

        // ---- per-group corrections: init = -sum_k c_k x_k (and row sums) ----
        {
            const int ngr = nch * T::GPC;
            for (int gr = warp; gr < ngr; gr += NW) {
                const int cl = gr / T::GPC, gi = gr - cl * T::GPC;
                float cs = 0.f, rs = 0.f;
#pragma unroll
                for (int ktg = 0; ktg < T::KTG; ++ktg) {
                    const int ktc = gi * T::KTG + ktg;
                    const int kts = cl * T::KT + ktc;
                    const uint4 q = xf[(kts >> 1) * 32 + lane];
                    const float2 f0 = pair_to_float2<XT>((kts & 1) ? q.z : q.x);
                    const float2 f1 = pair_to_float2<XT>((kts & 1) ? q.w : q.y);
                    const int ktl = ktc % (T::KT / 2);
                    const float s0 = f0.x + f0.y, s1 = f1.x + f1.y;
                    cs += slot_coef<FMT, XT>(2 * ktl) * s0 + slot_coef<FMT, XT>(2 * ktl + 1) * s1;
                    rs += s0 + s1;
                }
                cs += __shfl_xor_sync(0xffffffffu, cs, 1);
                cs += __shfl_xor_sync(0xffffffffu, cs, 2);
                rs += __shfl_xor_sync(0xffffffffu, rs, 1);
                rs += __shfl_xor_sync(0xffffffffu, rs, 2);
                if (t == 0) {
                    if constexpr (FMT == LBV_FMT_Q4_0)
                        corr[gr * 8 + g] = -(float)(dec_spec<FMT>(XT, 0).c + 8) * rs;
                    else
                        corr[gr * 8 + g] = -cs;
                    if constexpr (T::AFFINE)
                        rsum[gr * 8 + g] = rs;
                }
            }
        }
        __syncthreads();
        griddep_launch_dependents();

        // ---- main loop ----
        float y[TPW][4];
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl)
            y[tl][0] = y[tl][1] = y[tl][2] = y[tl][3] = 0.f;
        int cu = u0, cc = 0;
#pragma unroll 1
        for (int q0 = 0; q0 < Q; q0 += D) {
#pragma unroll
            for (int d = 0; d < D; ++d) {
                if (q0 + d < Q) {
                    uint4 w[TPW];
                    Side s[TPW];
#pragma unroll
                    for (int tl = 0; tl < TPW; ++tl) {
                        w[tl] = wb[d][tl];
                        s[tl] = sb[d][tl];
                    }
                    if (lq < Q) {
                        load_chunk(p, lu, c0 + lc, lane, wb[d], sb[d]);
                        ++lq;
                        if (++lc == nch) {
                            lc = 0;
                            lu += ustride;
                        }
                    }
                    process_chunk(w, s, cc, xf, corr, rsum, y, lane);
                    if (++cc == nch) {
                        if (p.splits == 1)
                            store_y(p, cu, y, g, t);
                        else
                            store_part(part, warp, y, lane);
#pragma unroll
                        for (int tl = 0; tl < TPW; ++tl)
                            y[tl][0] = y[tl][1] = y[tl][2] = y[tl][3] = 0.f;
                        cc = 0;
                        cu += ustride;
                    }
                }
            }
        }

        if (p.splits > 1)
            cluster_reduce(p, part);
    }

    static __device__ __forceinline__ void store_y(const VerifyParams& p, int unit,
                                                   const float (&y)[TPW][4], int g, int t)
    {
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl) {
            const int tile = unit * TPW + tl;
            if (tile >= p.ntiles)
                continue;
            const int n0 = tile * 16 + g, n1 = n0 + 8;
            const int m0 = 2 * t, m1 = 2 * t + 1;
            if (m0 < p.M) {
                if (n0 < p.N) p.Y[(size_t)m0 * p.ldy + n0] = y[tl][0];
                if (n1 < p.N) p.Y[(size_t)m0 * p.ldy + n1] = y[tl][2];
            }
            if (m1 < p.M) {
                if (n0 < p.N) p.Y[(size_t)m1 * p.ldy + n0] = y[tl][1];
                if (n1 < p.N) p.Y[(size_t)m1 * p.ldy + n1] = y[tl][3];
            }
        }
    }

    static __device__ __forceinline__ void store_part(float* part, int warp,
                                                      const float (&y)[TPW][4], int lane)
    {
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl)
#pragma unroll
            for (int j = 0; j < 4; ++j)
                part[((warp * TPW + tl) * 4 + j) * 32 + lane] = y[tl][j];
    }

    // Sum the K-slice partials of the cluster's CTAs in rank order 0..S-1 and
    // write Y; each CTA writes 1/S of the block's outputs.
    static __device__ void cluster_reduce(const VerifyParams& p, float* part)
    {
        cg::cluster_group cl = cg::this_cluster();
        cl.sync();
        const int S = p.splits;
        const int V = NW * TPW * 4 * 32;
        const int per = (V + S - 1) / S;
        const int rank = (int)cl.block_rank();
        const int vend = min(V, (rank + 1) * per);
        for (int v = rank * per + (int)threadIdx.x; v < vend; v += NW * 32) {
            float acc = 0.f;
            for (int q = 0; q < S; ++q)
                acc += cl.map_shared_rank(part, q)[v];
            const int ln = v & 31, j = (v >> 5) & 3, wt = v >> 7;   // wt = warp*TPW + tl
            const int w_ = wt / TPW, tl = wt - w_ * TPW;
            const int tile = (blockIdx.y * NW + w_) * TPW + tl;
            const int n = tile * 16 + (ln >> 2) + 8 * (j >> 1);
            const int m = 2 * (ln & 3) + (j & 1);
            if (tile < p.ntiles && n < p.N && m < p.M)
                p.Y[(size_t)m * p.ldy + n] = acc;
        }
        cl.sync();
    }
};

template <int FMT, int XT, int GROUP, int NW, int TPW>
__global__ void __launch_bounds__(NW * 32) lbv_verify_kernel(const VerifyParams p)
{
    extern __shared__ __align__(16) unsigned char smem[];
    VerifyKernel<FMT, XT, GROUP, NW, TPW>::run(p, smem);
}

// ---------------------------------------------------------------------------
// Host side: launch / smem / occupancy for one (FMT, XT, GROUP)

template <int FMT, int GROUP>
inline size_t smem_bytes_t(int warps, int tpw, int cps)
{
    using T = Traits<FMT, GROUP>;
    size_t b = smem_xf_bytes(T::KT, cps);
    b += (size_t)cps * T::GPC * 8 * sizeof(float) * (T::AFFINE ? 2 : 1);
    b += (size_t)warps * tpw * 4 * 32 * sizeof(float);
    return b;
}

template <int FMT, int XT, int GROUP>
inline void* kernel_ptr(int warps, int tpw)
{
    if (warps == 4 && tpw == 1) return (void*)lbv_verify_kernel<FMT, XT, GROUP, 4, 1>;
    if (warps == 4 && tpw == 2) return (void*)lbv_verify_kernel<FMT, XT, GROUP, 4, 2>;
    if (warps == 8 && tpw == 1) return (void*)lbv_verify_kernel<FMT, XT, GROUP, 8, 1>;
    if (warps == 8 && tpw == 2) return (void*)lbv_verify_kernel<FMT, XT, GROUP, 8, 2>;
    return nullptr;
}

template <int FMT, int XT, int GROUP>
inline cudaError_t launch_t(const Shape& sh, const VerifyParams& p, const LaunchOpts& o,
                            cudaStream_t st)
{
    void* k = kernel_ptr<FMT, XT, GROUP>(sh.warps, sh.tpw);
    if (!k)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)sh.splits, (unsigned)sh.ctas_n, 1u);
    cfg.blockDim = dim3((unsigned)(sh.warps * 32), 1u, 1u);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    unsigned na = 0;
    if (sh.splits > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)sh.splits;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (o.pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
    void* args[] = {const_cast<VerifyParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, k, args);
}

template <int FMT, int XT, int GROUP>
inline cudaError_t prepare_t(const Shape& sh)
{
    void* k = kernel_ptr<FMT, XT, GROUP>(sh.warps, sh.tpw);
    if (!k)
        return cudaErrorInvalidValue;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)sh.smem);
    if (e != cudaSuccess)
        return e;
    if (sh.splits > 1)
        e = cudaFuncSetAttribute(k, cudaFuncAttributeNonPortableClusterSizeAllowed, 0);
    return e;
}

template <int FMT, int XT, int GROUP>
inline int occupancy_t(const Shape& sh)
{
    void* k = kernel_ptr<FMT, XT, GROUP>(sh.warps, sh.tpw);
    int n = 0;
    if (!k || cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, sh.warps * 32, sh.smem) !=
                  cudaSuccess)
        return 0;
    return n;
}

}  // namespace lbv
