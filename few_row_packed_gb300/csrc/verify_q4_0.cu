// Few-row verify kernels for GGUF Q4_0 blocks (Ishizuki README, "Credits":
// GGUF block formats read as they are).
#include "verify_kernel.cuh"
#include "verify_ops.h"

LBV_DEFINE_VERIFY_OPS(q4_0, LBV_FMT_Q4_0, 32)
