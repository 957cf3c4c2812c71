// aux_kernels.cu -- the blockwise FWHT-128 activation rotation, the 1-row
// (GEMV) path and the dense fp16 dequant test export.
#include <algorithm>

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "lbv_internal.h"
#include "verify_kernel.cuh"

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
    static constexpr int CK = 256, KT = 16, W = 1, SLOTS = 16, GK = 128, SIDE_W = 2;
    static constexpr int REC = 512 + 8 * SIDE_W * 4;
};
template <int G>
struct AuxTraits<LBV_FMT_AFFINE2, G> {
    static constexpr int CK = 128, KT = 8, W = 2, SLOTS = 8, GK = G, SIDE_W = 2 * (128 / G);
    static constexpr int REC = 512 + 8 * SIDE_W * 4;
};
template <>
struct AuxTraits<LBV_FMT_Q4_0, 32> {
    static constexpr int CK = 64, KT = 4, W = 4, SLOTS = 4, GK = 32, SIDE_W = 2;
    static constexpr int REC = 512 + 8 * SIDE_W * 4;
};

// fp16 of one scale/bias half of a side word: lo half = column g, hi = g + 8.
__device__ __forceinline__ uint16_t side_half(uint32_t word, int hi)
{
    return hi ? (uint16_t)(word >> 16) : (uint16_t)(word & 0xFFFFu);
}

__device__ __forceinline__ float h2f(uint16_t b)
{
    return __half2float(__ushort_as_half(b));
}

// ---------------------------------------------------------------------------
// Dense fp16 dequant (test export): one thread per (tile, chunk, lane).
// sign1: +-s exactly; affine: s*q + b exact in fp64, rounded once; Q4_0:
// d*(q-8) exact in fp32, rounded once.

template <int FMT, int GROUP>
__global__ void __launch_bounds__(256) lbv_dequant_kernel(const uint8_t* Wp, int K, int N,
                                                          int ntiles, int nchunks, uint16_t* W)
{
    using A = AuxTraits<FMT, GROUP>;
    const long long idx = (long long)blockIdx.x * blockDim.x + threadIdx.x;
    const long long total = (long long)ntiles * nchunks * 32;
    if (idx >= total)
        return;
    const int lane = (int)(idx & 31);
    const long long tc = idx >> 5;
    const int tile = (int)(tc / nchunks), chunk = (int)(tc - (long long)tile * nchunks);
    const int g = lane >> 2, t = lane & 3;
    const uint8_t* rec = Wp + (size_t)tc * A::REC;
    const uint4 q = reinterpret_cast<const uint4*>(rec)[lane];
    const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
    const uint32_t* sw = reinterpret_cast<const uint32_t*>(rec + 512 + g * (A::SIDE_W * 4));
    for (int wi = 0; wi < 4; ++wi) {
        const int col = tile * 16 + g + 8 * (wi & 1);
        const int hi = wi & 1;
        const int half = wi >> 1;
        if (col >= N)
            continue;
        for (int s = 0; s < A::SLOTS; ++s) {
            const int kt = half * (A::KT / 2) + (s >> 1);
            const int k0 = chunk * A::CK + 16 * kt + 8 * (s & 1) + 2 * t;
            const int gi = (16 * kt) / A::GK;        // group within the chunk
            for (int h = 0; h < 2; ++h) {
                const int k = k0 + h;
                if (k >= K)
                    continue;
                const uint32_t code = (wv[wi] >> (s * A::W + 16 * h)) & ((1u << A::W) - 1u);
                uint16_t out;
                if constexpr (FMT == LBV_FMT_SIGN1_G128) {
                    const uint16_t sb = side_half(sw[gi], hi);
                    out = code ? sb : (uint16_t)(sb ^ 0x8000u);
                } else if constexpr (FMT == LBV_FMT_AFFINE2) {
                    const double sc = (double)h2f(side_half(sw[2 * gi], hi));
                    const double bi = (double)h2f(side_half(sw[2 * gi + 1], hi));
                    out = __half_as_ushort(__double2half(sc * (double)code + bi));
                } else {
                    const float d = h2f(side_half(sw[gi], hi));
                    out = __half_as_ushort(__float2half_rn(d * (float)((int)code - 8)));
                }
                W[(size_t)k * N + col] = out;
            }
        }
    }
}

cudaError_t launch_dequant(lbv_format fmt, int group, const uint8_t* Wp, int K, int N,
                           int ntiles, int nchunks, uint16_t* W, cudaStream_t st)
{
    const long long total = (long long)ntiles * nchunks * 32;
    const dim3 grid((unsigned)((total + 255) / 256));
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        lbv_dequant_kernel<LBV_FMT_SIGN1_G128, 128>
            <<<grid, 256, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        break;
    case LBV_FMT_AFFINE2:
        if (group == 32)
            lbv_dequant_kernel<LBV_FMT_AFFINE2, 32>
                <<<grid, 256, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        else if (group == 64)
            lbv_dequant_kernel<LBV_FMT_AFFINE2, 64>
                <<<grid, 256, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        else
            lbv_dequant_kernel<LBV_FMT_AFFINE2, 128>
                <<<grid, 256, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        break;
    case LBV_FMT_Q4_0:
        lbv_dequant_kernel<LBV_FMT_Q4_0, 32>
            <<<grid, 256, 0, st>>>(Wp, K, N, ntiles, nchunks, W);
        break;
    }
    return cudaGetLastError();
}

// ---------------------------------------------------------------------------
// 1-row path (the plain decode step), run once per row on the FMA pipe.  A CTA
// stages the row of X in shared memory as fp32 (plain 2-byte loads: X need
// only be 2-byte aligned), then its warps walk 16-column tiles (grid-stride,
// a warp per tile over all of K).  Per chunk one 16-byte load per lane gives
// the same codes the few-row kernel's lane reads (columns g and g + 8, k
// pairs of its fragment); each code meets its activation with one fp32 add
// or FMA (a sign weight flips the activation's sign bit), the group's scale
// (and bias times the group's row sum) is applied per group, and the 4 lanes
// of a column pair reduce by shuffles.

template <int FMT, int DT, int GROUP>
__global__ void __launch_bounds__(256) lbv_gemv_kernel(const VerifyParams p, int row)
{
    using A = AuxTraits<FMT, GROUP>;
    constexpr int KTG = A::GK / 16;                  // k-tiles per scale group
    extern __shared__ float xrow[];                  // [nchunks * CK] fp32, zero past K
    const int lane = threadIdx.x & 31, g = lane >> 2, t = lane & 3;
    const uint16_t* x = reinterpret_cast<const uint16_t*>(p.X) + (size_t)row * p.ldx;
    const int kpad = p.nchunks * A::CK;
#ifdef LBV_CHECKED
    {
        // checked build: the fp32 row fits the launch's shared memory and the
        // row lies inside X's rows
        uint32_t dyn;
        asm volatile("mov.u32 %0, %%dynamic_smem_size;\n" : "=r"(dyn));
        if ((size_t)kpad * sizeof(float) > dyn || row < 0 || row >= p.M || kpad < p.K) {
            if (threadIdx.x == 0)
                atomicOr(p.err, 2u);
            return;
        }
    }
#endif
    for (int k = threadIdx.x; k < kpad; k += blockDim.x) {
        float v = 0.f;
        if (k < p.K) {
            if constexpr (DT == LBV_F16)
                v = __half2float(__ushort_as_half(x[k]));
            else
                v = __bfloat162float(__ushort_as_bfloat16(x[k]));
        }
        xrow[k] = v;
    }
    __syncthreads();
    const int nwarps = gridDim.x * (blockDim.x >> 5);
    for (int tile = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5); tile < p.ntiles;
         tile += nwarps) {
        float y0 = 0.f, y1 = 0.f;                    // columns g and g + 8
        const uint8_t* rec = p.W + (size_t)tile * p.nchunks * A::REC;
        for (int chunk = 0; chunk < p.nchunks; ++chunk, rec += A::REC) {
            const uint4 q = __ldg(reinterpret_cast<const uint4*>(rec) + lane);
            const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
            const uint32_t* sw = reinterpret_cast<const uint32_t*>(rec + 512 + g * (A::SIDE_W * 4));
            const float* xc = xrow + chunk * A::CK;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                constexpr int span = KTG < A::KT / 2 ? KTG : A::KT / 2;
#pragma unroll
                for (int kt0 = 0; kt0 < A::KT / 2; kt0 += span) {
                    float a0 = 0.f, a1 = 0.f, r = 0.f;   // column g, column g + 8, row sum
#pragma unroll
                    for (int kk = 0; kk < span; ++kk) {
                        const int ktl = kt0 + kk;
                        const int kt = half * (A::KT / 2) + ktl;
#pragma unroll
                        for (int rr = 0; rr < 2; ++rr) {
                            const int s = 2 * ktl + rr;
                            const float2 xv =
                                *reinterpret_cast<const float2*>(xc + 16 * kt + 8 * rr + 2 * t);
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                const float xs = h ? xv.y : xv.x;
                                const int sh = s * A::W + 16 * h;
                                const uint32_t w0 = wv[2 * half], w1 = wv[2 * half + 1];
                                if constexpr (FMT == LBV_FMT_SIGN1_G128) {
                                    // bit 1 -> +x, bit 0 -> -x: flip the sign bit of x
                                    const uint32_t xb = __float_as_uint(xs);
                                    a0 += __uint_as_float(xb ^ ((~w0 << (31 - sh)) & 0x80000000u));
                                    a1 += __uint_as_float(xb ^ ((~w1 << (31 - sh)) & 0x80000000u));
                                } else if constexpr (FMT == LBV_FMT_AFFINE2) {
                                    a0 = fmaf((float)((w0 >> sh) & 3u), xs, a0);
                                    a1 = fmaf((float)((w1 >> sh) & 3u), xs, a1);
                                    r += xs;
                                } else {
                                    a0 = fmaf((float)((int)((w0 >> sh) & 15u) - 8), xs, a0);
                                    a1 = fmaf((float)((int)((w1 >> sh) & 15u) - 8), xs, a1);
                                }
                            }
                        }
                    }
                    const int gi = (16 * (half * (A::KT / 2) + kt0)) / A::GK;
                    if constexpr (FMT == LBV_FMT_AFFINE2) {
                        const uint32_t sc = sw[2 * gi], bi = sw[2 * gi + 1];
                        y0 = fmaf(h2f(side_half(sc, 0)), a0, fmaf(h2f(side_half(bi, 0)), r, y0));
                        y1 = fmaf(h2f(side_half(sc, 1)), a1, fmaf(h2f(side_half(bi, 1)), r, y1));
                    } else {
                        const uint32_t sc = sw[gi];
                        y0 = fmaf(h2f(side_half(sc, 0)), a0, y0);
                        y1 = fmaf(h2f(side_half(sc, 1)), a1, y1);
                    }
                }
            }
        }
        y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
        y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
        y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
        y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
        if (t == 0) {
            const int n0 = tile * 16 + g, n1 = n0 + 8;
            float* yr = p.Y + (size_t)row * p.ldy;
            if (n0 < p.N)
                yr[n0] = y0;
            if (n1 < p.N)
                yr[n1] = y1;
        }
    }
}

// 1-row path for the 1-bit format, by table lookup.  In the record layout a
// lane's word w of chunk c, half H (one 128-K group of one column) holds at
// bit 4i + j, i < 8, j < 4, the sign of k = 256 c + 16 (8 H + 2 (i & 3) +
// (j >> 1)) + 8 (j & 1) + 2 t + (i >> 2) for the lane's t = lane & 3 (the
// few-row kernel's fragment order).  So the 4-bit field i of w selects one of
// 16 signed sums of four activations:
//   T[c][H][i][t][v] = sum_j (bit j of v ? +x_k : -x_k),
// which each CTA tabulates once in shared memory, and a group's dot product
// is 8 table reads per word.  Warps take (tile, K quarter) items, four tiles
// per CTA at a time; each warp fetches an item's records with one bulk copy
// into one of two buffers, the next item's while it works on the current one
// (the first two are issued before the table is built), and the four
// quarters' partial sums of a tile meet in shared memory and are added in
// quarter order.  Within a (chunk, half, field) row of 272 bytes, entry
// (t, v) sits at word 16 t + v: the 16 values of one t take 16 different
// banks, so a warp's read conflicts only between lanes t and t + 2 that pick
// the same value.
constexpr int kLutWarps = 16, kLutTiles = kLutWarps / 4;
constexpr int kLutField = 272;                       // bytes per (chunk, half, field): 16 x 4 floats + pad
constexpr int kLutHalf = 8 * kLutField;
constexpr int kLutChunk = 2 * kLutHalf;

struct Sign1LutGeom {
    int kq, cpq;                                     // K quarters, chunks per quarter
    size_t table, xrow, buf, part, bars, end;        // byte offsets of the carve-up
};

__host__ __device__ inline Sign1LutGeom sign1_lut_geom(int nchunks, int K)
{
    using A = AuxTraits<LBV_FMT_SIGN1_G128, 128>;
    Sign1LutGeom gm;
    gm.kq = nchunks < 4 ? nchunks : 4;
    gm.cpq = (nchunks + gm.kq - 1) / gm.kq;
    gm.table = 0;
    gm.xrow = (size_t)nchunks * kLutChunk;
    gm.buf = gm.xrow + (((size_t)nchunks * A::CK * 2 + 15) / 16) * 16;
    gm.part = gm.buf + (size_t)kLutWarps * 2 * gm.cpq * A::REC;    // two buffers per warp
    gm.bars = gm.part + (size_t)kLutWarps * 32 * 2 * sizeof(float);
    gm.end = gm.bars + (size_t)kLutWarps * 2 * 8;
    (void)K;
    return gm;
}

// Sum of the 8 table entries that word w's fields select; tb points at the
// (chunk, half) block plus this lane's t (entries 4 bytes apart by value).
__device__ __forceinline__ float lut_word(uint32_t w, const unsigned char* tb)
{
    float e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        const uint32_t off = i == 0 ? (w << 2) & 0x3Cu : (w >> (4 * i - 2)) & 0x3Cu;
        e[i] = *reinterpret_cast<const float*>(tb + i * kLutField + off);
    }
    return ((e[0] + e[1]) + (e[2] + e[3])) + ((e[4] + e[5]) + (e[6] + e[7]));
}

template <int DT>
__global__ void __launch_bounds__(kLutWarps * 32) lbv_gemv_sign1_lut_kernel(const VerifyParams p,
                                                                             int row)
{
    using A = AuxTraits<LBV_FMT_SIGN1_G128, 128>;
    extern __shared__ __align__(128) unsigned char smem[];
    const Sign1LutGeom gm = sign1_lut_geom(p.nchunks, p.K);
#ifdef LBV_CHECKED
    {
        // checked build: the table kernel's carve-up fits the launch's shared
        // memory and the row lies inside X's rows
        uint32_t dyn;
        asm volatile("mov.u32 %0, %%dynamic_smem_size;\n" : "=r"(dyn));
        if (gm.end > dyn || row < 0 || row >= p.M) {
            if (threadIdx.x == 0)
                atomicOr(p.err, 2u);
            return;
        }
    }
#endif
    unsigned char* tbl = smem + gm.table;
    uint16_t* xs = reinterpret_cast<uint16_t*>(smem + gm.xrow);
    float* part = reinterpret_cast<float*>(smem + gm.part);
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31, g = lane >> 2, t = lane & 3;
    const int tl = warp % kLutTiles, q = warp / kLutTiles;
    const int ca = min(q * gm.cpq, p.nchunks), cz = min(ca + gm.cpq, p.nchunks);
    const uint32_t bar0 = smem_u32(smem + gm.bars) + warp * 16;       // per buffer
    unsigned char* buf0 = smem + gm.buf + (size_t)warp * 2 * gm.cpq * A::REC;
    if (lane == 0) {
        mbar_init(bar0, 1);
        mbar_init(bar0 + 8, 1);
        mbar_init_fence();
    }
    __syncwarp();
    // this warp's records of item n (tile tile0_n + tl) into buffer n & 1;
    // bit b of pend: a copy into buffer b issued and not yet waited for; bit b
    // of phase: the parity buffer b's next wait is for
    bool ok = true;
    uint32_t pend = 0u, phase = 0u;
    const int stride = gridDim.x * kLutTiles;
    auto fetch = [&](int n) {
        const int tile = blockIdx.x * kLutTiles + n * stride + tl, b = n & 1;
        if (ok && tile < p.ntiles && q < gm.kq && cz > ca) {
            if (lane == 0) {
                const uint32_t bytes = (uint32_t)(cz - ca) * A::REC;
                mbar_expect_tx(bar0 + b * 8, bytes);
                bulk_g2s_if(1u, smem_u32(buf0 + (size_t)b * gm.cpq * A::REC),
                            p.W + ((size_t)tile * p.nchunks + ca) * A::REC, bytes, bar0 + b * 8);
            }
            pend |= 1u << b;
        }
    };
    fetch(0);
    fetch(1);

    const uint16_t* x = reinterpret_cast<const uint16_t*>(p.X) + (size_t)row * p.ldx;
    for (int k = tid; k < p.nchunks * A::CK; k += kLutWarps * 32)
        xs[k] = k < p.K ? x[k] : (uint16_t)0;
    __syncthreads();
    // the table: one (chunk, half, field, t) row of 16 sums per thread and turn
    const int nrows = p.nchunks * 64;
    for (int r = tid; r < nrows; r += kLutWarps * 32) {
        const int tt = r & 3, i = (r >> 2) & 7, H = (r >> 5) & 1, c = r >> 6;
        float xv[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const int k = c * A::CK + 16 * (8 * H + 2 * (i & 3) + (j >> 1)) + 8 * (j & 1) + 2 * tt +
                          (i >> 2);
            if constexpr (DT == LBV_F16)
                xv[j] = __half2float(__ushort_as_half(xs[k]));
            else
                xv[j] = __bfloat162float(__ushort_as_bfloat16(xs[k]));
        }
        const float a[4] = {-xv[0] - xv[1], xv[0] - xv[1], -xv[0] + xv[1], xv[0] + xv[1]};
        const float b[4] = {-xv[2] - xv[3], xv[2] - xv[3], -xv[2] + xv[3], xv[2] + xv[3]};
        float* out = reinterpret_cast<float*>(tbl + (size_t)c * kLutChunk + H * kLutHalf +
                                              i * kLutField) + 16 * tt;
#pragma unroll
        for (int v = 0; v < 16; ++v)
            out[v] = a[v & 3] + b[v >> 2];
    }
    __syncthreads();

    int n = 0;
    for (int tile0 = blockIdx.x * kLutTiles; tile0 < p.ntiles; tile0 += stride, ++n) {
        const int tile = tile0 + tl, b = n & 1;
        float y0 = 0.f, y1 = 0.f;                    // columns g and g + 8
        if ((pend >> b) & 1u) {
            const uint32_t bar = bar0 + b * 8, par = (phase >> b) & 1u;
            const bool landed = mbar_try(bar, par) || mbar_wait(bar, par);
            if (__all_sync(0xffffffffu, landed)) {
                phase ^= 1u << b;
                pend &= ~(1u << b);
            } else {
                ok = false;
            }
        }
        if (ok && tile < p.ntiles && q < gm.kq && cz > ca) {
            const unsigned char* tb = tbl + (size_t)ca * kLutChunk + t * 64;
            const unsigned char* rec = buf0 + (size_t)b * gm.cpq * A::REC;
            for (int c = ca; c < cz; ++c, rec += A::REC, tb += kLutChunk) {
                const uint4 w = reinterpret_cast<const uint4*>(rec)[lane];
                const uint2 sw = *reinterpret_cast<const uint2*>(rec + 512 + g * 8);
                // x: column g, group 0; y: column g + 8, group 0; z, w: group 1
                y0 = fmaf(h2f(side_half(sw.x, 0)), lut_word(w.x, tb), y0);
                y1 = fmaf(h2f(side_half(sw.x, 1)), lut_word(w.y, tb), y1);
                y0 = fmaf(h2f(side_half(sw.y, 0)), lut_word(w.z, tb + kLutHalf), y0);
                y1 = fmaf(h2f(side_half(sw.y, 1)), lut_word(w.w, tb + kLutHalf), y1);
            }
        }
        __syncwarp();
        fence_proxy_async_if(lane == 0);                 // the buffer's reads before its refill
        fetch(n + 2);                                    // item n + 2 into this buffer
        // the 4 lanes of a column pair, then the quarters in order
        y0 += __shfl_xor_sync(0xffffffffu, y0, 1);
        y0 += __shfl_xor_sync(0xffffffffu, y0, 2);
        y1 += __shfl_xor_sync(0xffffffffu, y1, 1);
        y1 += __shfl_xor_sync(0xffffffffu, y1, 2);
        part[(warp * 32 + lane) * 2] = y0;
        part[(warp * 32 + lane) * 2 + 1] = y1;
        __syncthreads();
        if (q == 0 && t == 0 && tile < p.ntiles) {
            float s0 = 0.f, s1 = 0.f;
            for (int qq = 0; qq < gm.kq; ++qq) {
                const float* pp = part + ((qq * kLutTiles + tl) * 32 + lane) * 2;
                s0 += pp[0];
                s1 += pp[1];
            }
            const int n0 = tile * 16 + g, n1 = n0 + 8;
            float* yr = p.Y + (size_t)row * p.ldy;
            if (n0 < p.N)
                yr[n0] = s0;
            if (n1 < p.N)
                yr[n1] = s1;
        }
        __syncthreads();
    }
    for (int b = 0; b < 2; ++b)                      // a copy that did not land in time
        if ((pend >> b) & 1u)
            mbar_wait(bar0 + b * 8, (phase >> b) & 1u);
    if (!ok && lane == 0)
        atomicOr(p.err, 1u);
}

template <int FMT, int GROUP>
static cudaError_t gemv_t(lbv_dtype xt, const VerifyParams& p, int row, cudaStream_t st)
{
    using A = AuxTraits<FMT, GROUP>;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const int ctas = std::min((p.ntiles + 7) / 8, 4 * std::max(sms, 1));
    const size_t smem = (size_t)p.nchunks * A::CK * sizeof(float);
    void* k = xt == LBV_F16 ? (void*)lbv_gemv_kernel<FMT, LBV_F16, GROUP>
                            : (void*)lbv_gemv_kernel<FMT, LBV_BF16, GROUP>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)std::max<size_t>(smem, 48 * 1024));
    if (e != cudaSuccess)
        return e;
    if (xt == LBV_F16)
        lbv_gemv_kernel<FMT, LBV_F16, GROUP><<<ctas, 256, smem, st>>>(p, row);
    else
        lbv_gemv_kernel<FMT, LBV_BF16, GROUP><<<ctas, 256, smem, st>>>(p, row);
    return cudaGetLastError();
}

static cudaError_t gemv_sign1_lut(lbv_dtype xt, const VerifyParams& p, int row, cudaStream_t st)
{
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    const size_t smem = sign1_lut_geom(p.nchunks, p.K).end;
    const int ctas = std::min((p.ntiles + kLutTiles - 1) / kLutTiles, std::max(sms, 1));
    void* k = xt == LBV_F16 ? (void*)lbv_gemv_sign1_lut_kernel<LBV_F16>
                            : (void*)lbv_gemv_sign1_lut_kernel<LBV_BF16>;
    cudaError_t e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)std::max<size_t>(smem, 48 * 1024));
    if (e != cudaSuccess)
        return e;
    if (xt == LBV_F16)
        lbv_gemv_sign1_lut_kernel<LBV_F16><<<ctas, kLutWarps * 32, smem, st>>>(p, row);
    else
        lbv_gemv_sign1_lut_kernel<LBV_BF16><<<ctas, kLutWarps * 32, smem, st>>>(p, row);
    return cudaGetLastError();
}

cudaError_t launch_gemv(lbv_format fmt, lbv_dtype xt, int group, const VerifyParams& p, int row,
                        cudaStream_t st)
{
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        if (sign1_lut_geom(p.nchunks, p.K).end <= (size_t)kMaxDynSmem)
            return gemv_sign1_lut(xt, p, row, st);
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
