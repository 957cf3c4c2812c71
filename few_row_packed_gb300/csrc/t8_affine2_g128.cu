// t8_affine2_g128.cu -- e4m3 tensor-memory kernel, 2-bit affine g128.
#include "t8_kernel.cuh"

LBV_DEFINE_T8_OPS(t8_affine2_g128, LBV_FMT_AFFINE2)
