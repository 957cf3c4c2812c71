// Few-row verify kernels for 2-bit affine weights in groups of 128 (Ishizuki
// README, plain MLX affine packs; dflash-mlx-bonsai2 README, 2-bit pack).
#include "verify_kernel.cuh"
#include "verify_ops.h"

LBV_DEFINE_VERIFY_OPS(affine2_g128, LBV_FMT_AFFINE2, 128)
