// tcgen05 few-row verify kernels for GGUF Q4_0 blocks (Ishizuki README, "Credits":
// GGUF block formats read as they are).
#include "tc_kernel.cuh"

LBV_DEFINE_TC_OPS(tc_q4_0, LBV_FMT_Q4_0, 32)
