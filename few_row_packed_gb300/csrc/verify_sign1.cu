// Few-row verify kernels for the 1-bit sign g128 format (Bonsai-27B-mlx-1bit
// model card, format description).
#include "verify_kernel.cuh"
#include "verify_ops.h"

LBV_DEFINE_VERIFY_OPS(sign1, LBV_FMT_SIGN1_G128, 128)
