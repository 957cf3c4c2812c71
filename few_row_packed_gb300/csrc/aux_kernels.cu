// aux_kernels.cu -- the blockwise FWHT-128 activation rotation, the 1-row
// (GEMV) path and the dense fp16 dequant test export.
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lbv_internal.h"

namespace lbv {

// ---------------------------------------------------------------------------
// FWHT-128: one warp per 128-element block; lane holds elements 4*lane + i.
// Butterflies in fp64 are exact for fp16 inputs (and for bf16 blocks whose
// magnitudes span less than 2^45), so the only rounding is the IEEE division
// by sqrt(128) and the final round to nearest even in the output dtype.
// dflash-mlx-bonsai2 README, "What this fork adds" (sign, Hadamard prep);
// Sylvester natural order: H[i][j] = (-1)^popcount(i & j).

template <int DT>
__device__ __forceinline__ double to_f64(uint16_t b)
{
    if constexpr (DT == LBV_F16)
        return (double)__half2float(__ushort_as_half(b));
    else
        return (double)__bfloat162float(__ushort_as_bfloat16(b));
}

template <int DT>
__device__ __forceinline__ uint16_t from_f64(double v)
{
    if constexpr (DT == LBV_F16)
        return __half_as_ushort(__double2half(v));
    else
        return __bfloat16_as_ushort(__double2bfloat16(v));
}

template <int DT>
__global__ void __launch_bounds__(256) lbv_fwht128_kernel(const uint16_t* X, uint16_t* Xr, int M,
                                                           int K, const uint32_t* signs)
{
    const int lane = threadIdx.x & 31;
    const int nb = K / 128;
    const int blk = blockIdx.x * 8 + (threadIdx.x >> 5);
    if (blk >= M * nb)
        return;
    const int row = blk / nb, b = blk - row * nb;
    const size_t base = (size_t)row * K + (size_t)b * 128 + 4 * lane;
    double v[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        double x = to_f64<DT>(X[base + i]);
        if (signs) {
            const int k = b * 128 + 4 * lane + i;
            if ((signs[k >> 5] >> (k & 31)) & 1u)
                x = -x;
        }
        v[i] = x;
    }
    // h = 1, 2: within the lane
#pragma unroll
    for (int h = 1; h <= 2; h <<= 1)
#pragma unroll
        for (int i = 0; i < 4; ++i)
            if (!(i & h)) {
                const double a = v[i], c = v[i + h];
                v[i] = a + c;
                v[i + h] = a - c;
            }
    // h = 4 .. 64: partner lane = lane ^ (h / 4)
#pragma unroll
    for (int lm = 1; lm <= 16; lm <<= 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const double o = __shfl_xor_sync(0xffffffffu, v[i], lm);
            v[i] = (lane & lm) ? (o - v[i]) : (v[i] + o);
        }
    }
    __syncwarp();
    const double norm = sqrt(128.0);
#pragma unroll
    for (int i = 0; i < 4; ++i)
        Xr[base + i] = from_f64<DT>(v[i] / norm);
}

cudaError_t launch_fwht128(const void* X, void* Xr, int M, int K, lbv_dtype dt,
                           const uint32_t* signs, cudaStream_t st)
{
    const int nblk = M * (K / 128);
    const dim3 grid((unsigned)((nblk + 7) / 8));
    if (dt == LBV_F16)
        lbv_fwht128_kernel<LBV_F16><<<grid, 256, 0, st>>>((const uint16_t*)X, (uint16_t*)Xr, M,
                                                           K, signs);
    else
        lbv_fwht128_kernel<LBV_BF16><<<grid, 256, 0, st>>>((const uint16_t*)X, (uint16_t*)Xr,
                                                            M, K, signs);
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// Per-format constants of the device layout (see layout.h).

template <int FMT, int GROUP>
struct AuxTraits;
template <>
struct AuxTraits<LBV_FMT_SIGN1_G128, 128> {
    static constexpr int CK = 128, CB = 16, SB = 2, W = 1, GK = 128;
};
template <int G>
struct AuxTraits<LBV_FMT_AFFINE2, G> {
    static constexpr int CK = G == 128 ? 128 : 64, CB = G == 128 ? 32 : 16, SB = G == 32 ? 8 : 4,
                         W = 2, GK = G;
};
template <>
struct AuxTraits<LBV_FMT_Q4_0, 32> {
    static constexpr int CK = 64, CB = 32, SB = 4, W = 4, GK = 32;
};

template <int FMT, int GROUP>
struct AuxGeo {
    using A = AuxTraits<FMT, GROUP>;
    static constexpr int PPW = 16 / A::W, NWORD = A::CB / 4, GPC = A::CK / A::GK;
    static constexpr int REC = 128 * (A::CB + A::SB);
};

__device__ __forceinline__ float h2f(uint16_t b)
{
    return __half2float(__ushort_as_half(b));
}

// The codes words and side values of column c (0..127) of one record.
template <int FMT, int GROUP>
__device__ __forceinline__ void read_column(const uint8_t* rec, int c,
                                            uint32_t (&wv)[AuxGeo<FMT, GROUP>::NWORD],
                                            uint16_t (&sv)[AuxTraits<FMT, GROUP>::SB / 2])
{
    using A = AuxTraits<FMT, GROUP>;
#pragma unroll
    for (int h = 0; h < A::CB / 16; ++h) {
        const uint4 v = *reinterpret_cast<const uint4*>(rec + h * 2048 + c * 16);
        wv[4 * h + 0] = v.x;
        wv[4 * h + 1] = v.y;
        wv[4 * h + 2] = v.z;
        wv[4 * h + 3] = v.w;
    }
#pragma unroll
    for (int i = 0; i < A::SB / 2; ++i)
        sv[i] = reinterpret_cast<const uint16_t*>(rec + 128 * A::CB + c * A::SB)[i];
}

// Code of pair-element (p, h) of a column: k = 2p + h within the chunk.
template <int FMT, int GROUP>
__device__ __forceinline__ uint32_t code_at(const uint32_t (&wv)[AuxGeo<FMT, GROUP>::NWORD], int p,
                                            int h)
{
    using A = AuxTraits<FMT, GROUP>;
    using Gm = AuxGeo<FMT, GROUP>;
    return (wv[p / Gm::PPW] >> ((p % Gm::PPW) * A::W + 16 * h)) & ((1u << A::W) - 1u);
}

// ---------------------------------------------------------------------------
// Dense fp16 dequant (test export): one thread per (tile, chunk, column).
// sign1: +-s exactly; affine: s*q + b exact in fp64, rounded once; Q4_0:
// d*(q-8) exact in fp32, rounded once.

template <int FMT, int GROUP>
__global__ void __launch_bounds__(128) lbv_dequant_kernel(const uint8_t* Wp, int K, int N,
                                                          int ntiles, int nchunks, uint16_t* W)
{
    using A = AuxTraits<FMT, GROUP>;
    using Gm = AuxGeo<FMT, GROUP>;
    const long long tc = blockIdx.x;                     // record index
    const int c = threadIdx.x;
    const int tile = (int)(tc / nchunks), chunk = (int)(tc - (long long)tile * nchunks);
    const int col = tile * 128 + c;
    if (col >= N)
        return;
    uint32_t wv[Gm::NWORD];
    uint16_t sv[A::SB / 2];
    read_column<FMT, GROUP>(Wp + (size_t)tc * Gm::REC, c, wv, sv);
    for (int kk = 0; kk < A::CK; ++kk) {
        const int k = chunk * A::CK + kk;
        if (k >= K)
            break;
        const uint32_t code = code_at<FMT, GROUP>(wv, kk >> 1, kk & 1);
        const int gi = kk / A::GK;
        uint16_t out;
        if constexpr (FMT == LBV_FMT_SIGN1_G128) {
            out = code ? sv[0] : (uint16_t)(sv[0] ^ 0x8000u);
        } else if constexpr (FMT == LBV_FMT_AFFINE2) {
            const double sc = (double)h2f(sv[2 * gi]);
            const double bi = (double)h2f(sv[2 * gi + 1]);
            out = __half_as_ushort(__double2half(sc * (double)code + bi));
        } else {
            const float d = h2f(sv[gi]);
            out = __half_as_ushort(__float2half_rn(d * (float)((int)code - 8)));
        }
        W[(size_t)k * N + col] = out;
    }
}

cudaError_t launch_dequant(lbv_format fmt, int group, const uint8_t* Wp, int K, int N,
                           int ntiles, int nchunks, uint16_t* W, cudaStream_t st)
{
    const dim3 grid((unsigned)((long long)ntiles * nchunks));
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        lbv_dequant_kernel<LBV_FMT_SIGN1_G128, 128><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        break;
    case LBV_FMT_AFFINE2:
        if (group == 32)
            lbv_dequant_kernel<LBV_FMT_AFFINE2, 32><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        else if (group == 64)
            lbv_dequant_kernel<LBV_FMT_AFFINE2, 64><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        else
            lbv_dequant_kernel<LBV_FMT_AFFINE2, 128><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        break;
    case LBV_FMT_Q4_0:
        lbv_dequant_kernel<LBV_FMT_Q4_0, 32><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        break;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// 1-row path (the plain decode step): one thread per output column over all
// of K, fp32 FMAs on the FMA pipe, run once per row.  A warp reads 32
// consecutive columns' records (coalesced); X is read through the L1 cache.

template <int DT>
__device__ __forceinline__ float x_at(const uint16_t* x, int k)
{
    if constexpr (DT == LBV_F16)
        return __half2float(__ushort_as_half(x[k]));
    else
        return __bfloat162float(__ushort_as_bfloat16(x[k]));
}

template <int FMT, int DT, int GROUP>
__global__ void __launch_bounds__(128) lbv_gemv_kernel(const VerifyParams p, int row)
{
    using A = AuxTraits<FMT, GROUP>;
    using Gm = AuxGeo<FMT, GROUP>;
    const int tile = blockIdx.x, c = threadIdx.x;
    const int col = tile * 128 + c;
    const uint16_t* x = reinterpret_cast<const uint16_t*>(p.X) + (size_t)row * p.ldx;
    float y = 0.f;
    for (int chunk = 0; chunk < p.nchunks; ++chunk) {
        uint32_t wv[Gm::NWORD];
        uint16_t sv[A::SB / 2];
        read_column<FMT, GROUP>(p.W + ((size_t)tile * p.nchunks + chunk) * Gm::REC, c, wv, sv);
#pragma unroll
        for (int gi = 0; gi < Gm::GPC; ++gi) {
            float a = 0.f, r = 0.f;
#pragma unroll 8
            for (int kk = gi * A::GK; kk < (gi + 1) * A::GK; ++kk) {
                const int k = chunk * A::CK + kk;
                const float xv = k < p.K ? x_at<DT>(x, k) : 0.f;
                const uint32_t code = code_at<FMT, GROUP>(wv, kk >> 1, kk & 1);
                if constexpr (FMT == LBV_FMT_SIGN1_G128)
                    a += code ? xv : -xv;
                else if constexpr (FMT == LBV_FMT_AFFINE2) {
                    a = fmaf((float)code, xv, a);
                    r += xv;
                } else
                    a = fmaf((float)((int)code - 8), xv, a);
            }
            if constexpr (FMT == LBV_FMT_AFFINE2)
                y = fmaf(h2f(sv[2 * gi]), a, fmaf(h2f(sv[2 * gi + 1]), r, y));
            else
                y = fmaf(h2f(sv[gi]), a, y);
        }
    }
    if (col < p.N)
        p.Y[(size_t)row * p.ldy + col] = y;
}

template <int FMT, int GROUP>
static cudaError_t gemv_t(lbv_dtype xt, const VerifyParams& p, int row, cudaStream_t st)
{
    const dim3 grid((unsigned)p.ntiles);
    if (xt == LBV_F16)
        lbv_gemv_kernel<FMT, LBV_F16, GROUP><<<grid, 128, 0, st>>>(p, row);
    else
        lbv_gemv_kernel<FMT, LBV_BF16, GROUP><<<grid, 128, 0, st>>>(p, row);
    return cudaGetLastError();
}

cudaError_t launch_gemv(lbv_format fmt, lbv_dtype xt, int group, const VerifyParams& p, int row,
                        cudaStream_t st)
{
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        return gemv_t<LBV_FMT_SIGN1_G128, 128>(xt, p, row, st);
    case LBV_FMT_AFFINE2:
        if (group == 32)
            return gemv_t<LBV_FMT_AFFINE2, 32>(xt, p, row, st);
        if (group == 64)
            return gemv_t<LBV_FMT_AFFINE2, 64>(xt, p, row, st);
        return gemv_t<LBV_FMT_AFFINE2, 128>(xt, p, row, st);
    case LBV_FMT_Q4_0:
        return gemv_t<LBV_FMT_Q4_0, 32>(xt, p, row, st);
    }
    return cudaErrorInvalidValue;
}

}  // namespace lbv
