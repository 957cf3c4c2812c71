// tc_internal.h -- launch parameters, shape and entry points of the tcgen05
// few-row kernel (plans created with LBV_PLAN_TCGEN05) and of the kernels that
// read its 128-column record layout (tc_layout.h).
#pragma once

#include <cuda_runtime.h>

#include "lbv_internal.h"
#include "tc_layout.h"

namespace lbv {

// Decode warpgroups per CTA of the tcgen05 few-row kernel.
constexpr int kTcWarpgroups = 3;

// Parameters of one tcgen05 few-row launch (passed by value to the kernel).
struct TcParams {
    const void* X;          // [M][ldx] fp16 / bf16
    const uint8_t* W;       // packed records [tile][chunk] (tc_layout.h)
    float* Y;               // [M][ldy]
    unsigned* err;          // device status word of the plan (bounded waits)
    int ldx, ldy;
    int M, K, N;
    int ntiles, nchunks;
    int splits;             // K slices == cluster size along grid x
    int cps;                // chunks per slice (the last slice may be shorter)
    int wsplit;             // warpgroup split of a slice inside a CTA (divides kTcWarpgroups)
    int x_vec;              // 1: X rows 16-byte aligned (vector staging)
    unsigned zero;          // always 0 (keeps decode constants in registers)
};

// Per-(format, group) entry points of the tcgen05 few-row kernel; each
// translation unit tc_<fmt>.cu instantiates one set.
struct TcOps {
    cudaError_t (*launch)(lbv_dtype xt, const TcShape& sh, const TcParams& p,
                          const LaunchOpts& o, cudaStream_t st);
    cudaError_t (*prepare)(lbv_dtype xt, const TcShape& sh);
    int (*max_clusters)(lbv_dtype xt, const TcShape& sh);
    size_t (*smem)(int cps, int owned_max, int nparts);   // nparts = splits * wsplit
};

extern const TcOps tc_sign1_ops;
extern const TcOps tc_affine2_g32_ops;
extern const TcOps tc_affine2_g64_ops;
extern const TcOps tc_affine2_g128_ops;
extern const TcOps tc_q4_0_ops;

// Records of the 128-column layout -> fp16 W[K][N], rounded once (test export).
cudaError_t tc_launch_dequant(lbv_format fmt, int group, const uint8_t* Wp, int K, int N,
                              int ntiles, int nchunks, uint16_t* W, cudaStream_t st);

}  // namespace lbv

// Defines the TcOps of one (FMT, GROUP) in a translation unit that includes
// tc_kernel.cuh.
#define LBV_DEFINE_TC_OPS(NAME, FMT, GROUP)                                                  \
    namespace lbv {                                                                        \
    static cudaError_t NAME##_launch(lbv_dtype xt, const TcShape& sh, const TcParams& p,   \
                                     const LaunchOpts& o, cudaStream_t st)                 \
    {                                                                                      \
        return xt == LBV_F16 ? tc_launch_t<FMT, LBV_F16, GROUP>(sh, p, o, st)              \
                             : tc_launch_t<FMT, LBV_BF16, GROUP>(sh, p, o, st);            \
    }                                                                                      \
    static cudaError_t NAME##_prepare(lbv_dtype xt, const TcShape& sh)                     \
    {                                                                                      \
        return xt == LBV_F16 ? tc_prepare_t<FMT, LBV_F16, GROUP>(sh)                       \
                             : tc_prepare_t<FMT, LBV_BF16, GROUP>(sh);                     \
    }                                                                                      \
    static int NAME##_max_clusters(lbv_dtype xt, const TcShape& sh)                        \
    {                                                                                      \
        return xt == LBV_F16 ? tc_max_clusters_t<FMT, LBV_F16, GROUP>(sh)                  \
                             : tc_max_clusters_t<FMT, LBV_BF16, GROUP>(sh);                \
    }                                                                                      \
    static size_t NAME##_smem(int cps, int owned_max, int nparts)                          \
    {                                                                                      \
        return tc_smem_bytes<FMT, GROUP>(cps, owned_max, nparts);                          \
    }                                                                                      \
    const TcOps NAME##_ops = {NAME##_launch, NAME##_prepare, NAME##_max_clusters,          \
                              NAME##_smem};                                                \
    }
