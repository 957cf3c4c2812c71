// t8_sign1.cu -- e4m3 tensor-memory kernel, 1-bit sign g128.
#include "t8_kernel.cuh"

LBV_DEFINE_T8_OPS(t8_sign1, LBV_FMT_SIGN1_G128)
