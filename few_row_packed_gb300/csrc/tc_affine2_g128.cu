// tcgen05 few-row verify kernels for 2-bit affine weights in groups of 128 (Ishizuki
// README, plain MLX affine packs; dflash-mlx-bonsai2 README, 2-bit pack).
#include "tc_kernel.cuh"

LBV_DEFINE_TC_OPS(tc_affine2_g128, LBV_FMT_AFFINE2, 128)
