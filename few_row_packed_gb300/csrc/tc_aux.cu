// tc_aux.cu -- kernels that read the 128-column record layout (tc_layout.h)
// other than the few-row verify kernel itself: the fp16 dequant export used by
// the bit-exact tests of LBV_PLAN_TCGEN05 plans.
#include <cuda_fp16.h>

#include "tc_internal.h"

namespace lbv {

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
__global__ void __launch_bounds__(128) lbv_tc_dequant_kernel(const uint8_t* Wp, int K, int N,
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

cudaError_t tc_launch_dequant(lbv_format fmt, int group, const uint8_t* Wp, int K, int N,
                           int ntiles, int nchunks, uint16_t* W, cudaStream_t st)
{
    const dim3 grid((unsigned)((long long)ntiles * nchunks));
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        lbv_tc_dequant_kernel<LBV_FMT_SIGN1_G128, 128><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        break;
    case LBV_FMT_AFFINE2:
        if (group == 32)
            lbv_tc_dequant_kernel<LBV_FMT_AFFINE2, 32><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        else if (group == 64)
            lbv_tc_dequant_kernel<LBV_FMT_AFFINE2, 64><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        else
            lbv_tc_dequant_kernel<LBV_FMT_AFFINE2, 128><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        break;
    case LBV_FMT_Q4_0:
        lbv_tc_dequant_kernel<LBV_FMT_Q4_0, 32><<<grid, 128, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        break;
    }
    return cudaGetLastError();
}

}  // namespace lbv
