// verify_ops.h -- per-(format, group) few-row kernel entry points; each
// translation unit verify_<fmt>.cu instantiates one set.
#pragma once

#include "lbv_internal.h"

namespace lbv {

struct VerifyOps {
    cudaError_t (*launch)(lbv_dtype xt, const Shape& sh, const VerifyParams& p,
                          const LaunchOpts& o, cudaStream_t st);
    cudaError_t (*prepare)(lbv_dtype xt, const Shape& sh);
    int (*max_clusters)(lbv_dtype xt, const Shape& sh);
    size_t (*smem)(int warps, int tpw, int cps, int tiles_max, int splits);
    // grouped verify (16 warps, 1 or 2 tiles per unit)
    cudaError_t (*launch_grouped)(lbv_dtype xt, const Shape& sh, const GroupedParams& gp,
                                  const LaunchOpts& o, cudaStream_t st);
    int (*max_clusters_grouped)(lbv_dtype xt, const Shape& sh);
};

extern const VerifyOps sign1_ops;
extern const VerifyOps affine2_g32_ops;
extern const VerifyOps affine2_g64_ops;
extern const VerifyOps affine2_g128_ops;
extern const VerifyOps q4_0_ops;

}  // namespace lbv

// Defines the VerifyOps of one (FMT, GROUP) in a translation unit that
// includes verify_kernel.cuh.
#define LBV_DEFINE_VERIFY_OPS(NAME, FMT, GROUP)                                             \
    namespace lbv {                                                                         \
    static cudaError_t NAME##_launch(lbv_dtype xt, const Shape& sh, const VerifyParams& p,  \
                                     const LaunchOpts& o, cudaStream_t st)                  \
    {                                                                                       \
        return xt == LBV_F16 ? launch_t<FMT, LBV_F16, GROUP>(sh, p, o, st)                  \
                             : launch_t<FMT, LBV_BF16, GROUP>(sh, p, o, st);                \
    }                                                                                       \
    static cudaError_t NAME##_prepare(lbv_dtype xt, const Shape& sh)                        \
    {                                                                                       \
        return xt == LBV_F16 ? prepare_t<FMT, LBV_F16, GROUP>(sh)                           \
                             : prepare_t<FMT, LBV_BF16, GROUP>(sh);                         \
    }                                                                                       \
    static int NAME##_max_clusters(lbv_dtype xt, const Shape& sh)                           \
    {                                                                                       \
        return xt == LBV_F16 ? max_clusters_t<FMT, LBV_F16, GROUP>(sh)                      \
                             : max_clusters_t<FMT, LBV_BF16, GROUP>(sh);                    \
    }                                                                                       \
    static size_t NAME##_smem(int warps, int tpw, int cps, int tiles_max, int splits)       \
    {                                                                                       \
        return smem_bytes_t<FMT, GROUP>(warps, tpw, cps, tiles_max, splits);                \
    }                                                                                       \
    static cudaError_t NAME##_launch_grouped(lbv_dtype xt, const Shape& sh,                 \
                                             const GroupedParams& gp, const LaunchOpts& o,  \
                                             cudaStream_t st)                               \
    {                                                                                       \
        return xt == LBV_F16 ? launch_grouped_t<FMT, LBV_F16, GROUP>(sh, gp, o, st)         \
                             : launch_grouped_t<FMT, LBV_BF16, GROUP>(sh, gp, o, st);       \
    }                                                                                       \
    static int NAME##_max_clusters_grouped(lbv_dtype xt, const Shape& sh)                   \
    {                                                                                       \
        return xt == LBV_F16 ? max_clusters_t<FMT, LBV_F16, GROUP>(sh, true)                \
                             : max_clusters_t<FMT, LBV_BF16, GROUP>(sh, true);              \
    }                                                                                       \
    const VerifyOps NAME##_ops = {NAME##_launch, NAME##_prepare, NAME##_max_clusters,       \
                                  NAME##_smem, NAME##_launch_grouped,                       \
                                  NAME##_max_clusters_grouped};                             \
    }
