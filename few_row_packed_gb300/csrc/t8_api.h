// t8_api.h -- host entry points of plans created with LBV_PLAN_TC_E4M3
// (t8_api.cpp), used by api.cpp.
#pragma once

#include <cuda_runtime.h>

#include "lbv_internal.h"

namespace lbv {

// Fills the plan's t8_fi, t8_layout and default t8_shape; false if the format
// is not one the kernel reads or no launch shape fits the device.
bool t8_plan_setup(lbv_plan* P);

// Overrides the launch shape (K split, clusters along N; 0 = as many as fit).
bool t8_set_shape(lbv_plan* P, int splits, int ctas_n);

// Fused-head options of a launch (lbv_verify_gemm: rot = 0, store_y = 1,
// no argmax).
struct T8Fused {
    int rot;
    int store_y;
    const uint32_t* signs;
    unsigned long long* amax_keys;
    unsigned* amax_done;
    int* amax_idx;
    float* amax_val;
};

cudaError_t t8_verify_launch(const lbv_plan* P, const void* X, int M, int ldx, const void* Wp,
                             float* Y, int ldy, const T8Fused& f, bool pdl, cudaStream_t st);

cudaError_t t8_dequant(const lbv_plan* P, const void* Wp, uint16_t* W, cudaStream_t st);

size_t t8_packed_bytes(const lbv_plan* P);

// part0..2: the canonical arrays of lbv_pack_sign_g128 (bits, scales) or
// lbv_pack_affine2 (codes, scales, biases).
void t8_pack(const lbv_plan* P, const void* part0, const void* part1, const void* part2,
             uint8_t* out);

}  // namespace lbv
