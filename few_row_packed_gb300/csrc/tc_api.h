// tc_api.h -- host entry points of plans created with LBV_PLAN_TCGEN05
// (tc_api.cpp), used by api.cpp.
#pragma once

#include <cuda_runtime.h>

#include "lbv_internal.h"

namespace lbv {

// Fills the plan's tc_fi, tc_layout and default tc_shape; false if no launch
// shape fits the device.
bool tc_plan_setup(lbv_plan* P);

// Overrides the launch shape (K split, clusters along N; 0 = as many as fit).
bool tc_set_shape(lbv_plan* P, int splits, int ctas_n);

cudaError_t tc_verify_launch(const lbv_plan* P, const void* X, int M, int ldx, const void* Wp,
                             float* Y, int ldy, bool pdl, cudaStream_t st);

cudaError_t tc_dequant(const lbv_plan* P, const void* Wp, uint16_t* W, cudaStream_t st);

size_t tc_packed_bytes(const lbv_plan* P);

// part0..2: the canonical arrays of lbv_pack_sign_g128 (bits, scales),
// lbv_pack_affine2 (codes, scales, biases) or lbv_pack_q4_0 (blocks).
void tc_pack(const lbv_plan* P, const void* part0, const void* part1, const void* part2,
             uint8_t* out);

}  // namespace lbv
