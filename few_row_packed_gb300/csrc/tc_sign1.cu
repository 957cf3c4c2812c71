// tcgen05 few-row verify kernels for the 1-bit sign g128 format (Bonsai-27B-mlx-1bit
// model card, format description).
#include "tc_kernel.cuh"

LBV_DEFINE_TC_OPS(tc_sign1, LBV_FMT_SIGN1_G128, 128)
