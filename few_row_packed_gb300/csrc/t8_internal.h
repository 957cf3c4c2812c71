// t8_internal.h -- launch parameters, constants and entry points of the e4m3
// tensor-memory kernel (plans created with LBV_PLAN_TC_E4M3, t8_kernel.cuh).
#pragma once

#include <cuda_runtime.h>

#include "lbv_internal.h"
#include "t8_layout.h"

namespace lbv {

constexpr int kT8DecodeWarps = 16;                 // 4 warpgroups x 4
constexpr int kT8Threads = (kT8DecodeWarps + 4) * 32;   // + one MMA warp per warpgroup
constexpr int kT8Stages = 6;                       // ring stages per decode warp
constexpr int kT8EarlyStages = 2;                  // issued before the prologue
constexpr int kT8MaxSmem = 227 * 1024;
// Requesting more than half of an SM's shared memory keeps two CTAs (each
// allocating all tensor memory) off one SM.
constexpr size_t kT8SmemOnePerSm = 116 * 1024;

// Groups per ring stage of a warpgroup: 4608-byte stages either way.
template <int FMT>
constexpr int kT8GroupsPerStage = FMT == LBV_FMT_SIGN1_G128 ? 2 : 1;

// Parameters of one launch (passed by value to the kernel).
struct T8Params {
    const void* X;          // [M][ldx] fp16 / bf16
    const uint8_t* W;       // packed records (t8_layout.h)
    float* Y;               // [M][ldy]
    unsigned* err;          // device status word of the plan (bounded waits)
    int ldx, ldy;
    int M, K, N;
    int ntiles, ngroups;
    int splits;             // K slices == cluster size along grid x
    int gps;                // groups per slice (the last slice may be shorter)
    int owned;              // partial-slot tiles per CTA (splits > 1)
    int x_vec;              // 1: X rows 16-byte aligned (bulk staging)
    int x_in_ring;          // 1: X staged in the ring stages issued after the prologue
    int wait_limit;         // tries of a ring wait (0: the default, ~1 s)
    // fused head (lbv_verify_fused); lbv_verify_gemm leaves rot = 0,
    // amax_keys = NULL and store_y = 1
    int rot;
    int store_y;
    const uint32_t* signs;
    unsigned long long* amax_keys;
    unsigned* amax_done;
    int* amax_idx;
    float* amax_val;
};

// Per-format entry points; each translation unit t8_<fmt>.cu instantiates one set.
struct T8Ops {
    cudaError_t (*launch)(lbv_dtype xt, const T8Shape& sh, const T8Params& p,
                          const LaunchOpts& o, cudaStream_t st);
    cudaError_t (*prepare)(lbv_dtype xt, const T8Shape& sh);
    int (*max_clusters)(lbv_dtype xt, const T8Shape& sh);
    size_t (*smem)(int gps, int splits, int owned, int x_in_ring);
    bool (*x_fits_ring)(int gps);
    cudaError_t (*dequant)(const uint8_t* Wp, int K, int N, int ntiles, int ngroups, uint16_t* W,
                           cudaStream_t st);
};

extern const T8Ops t8_sign1_ops;
extern const T8Ops t8_affine2_g128_ops;

}  // namespace lbv

// Defines the T8Ops of one format in a translation unit that includes
// t8_kernel.cuh.
#define LBV_DEFINE_T8_OPS(NAME, FMT)                                                       \
    namespace lbv {                                                                        \
    static cudaError_t NAME##_launch(lbv_dtype xt, const T8Shape& sh, const T8Params& p,   \
                                     const LaunchOpts& o, cudaStream_t st)                 \
    {                                                                                      \
        return xt == LBV_F16 ? t8_launch_t<FMT, LBV_F16>(sh, p, o, st)                     \
                             : t8_launch_t<FMT, LBV_BF16>(sh, p, o, st);                   \
    }                                                                                      \
    static cudaError_t NAME##_prepare(lbv_dtype xt, const T8Shape& sh)                     \
    {                                                                                      \
        return xt == LBV_F16 ? t8_prepare_t<FMT, LBV_F16>(sh) : t8_prepare_t<FMT, LBV_BF16>(sh); \
    }                                                                                      \
    static int NAME##_max_clusters(lbv_dtype xt, const T8Shape& sh)                        \
    {                                                                                      \
        return xt == LBV_F16 ? t8_max_clusters_t<FMT, LBV_F16>(sh)                         \
                             : t8_max_clusters_t<FMT, LBV_BF16>(sh);                       \
    }                                                                                      \
    static size_t NAME##_smem(int gps, int splits, int owned, int x_in_ring)               \
    {                                                                                      \
        return t8_smem_bytes_t<FMT>(gps, splits, owned, x_in_ring);                        \
    }                                                                                      \
    static bool NAME##_x_fits_ring(int gps) { return t8_x_fits_ring<FMT>(gps); }           \
    const T8Ops NAME##_ops = {NAME##_launch, NAME##_prepare, NAME##_max_clusters,          \
                              NAME##_smem, NAME##_x_fits_ring, t8_dequant_t<FMT>};         \
    }
