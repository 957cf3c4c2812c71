// lbv_internal.h -- plan object, launch parameters and the launcher entry
// points each kernel translation unit exports to the C-ABI layer.
#pragma once

#include <cuda_runtime.h>

#include "layout.h"

namespace lbv {

// Parameters of one few-row verify launch (passed by value to the kernel).
struct VerifyParams {
    const void* X;          // [M][ldx] fp16 / bf16
    const uint4* codes;     // codes region of the device layout
    const uint8_t* side;    // side region
    float* Y;               // [M][ldy]
    int ldx, ldy;
    int M, K, N;
    int ntiles, nchunks;
    int splits;             // K slices == cluster size along grid x
    int cps;                // chunks per slice (the last slice may be shorter)
    int x_vec;              // 1: X rows 16-byte aligned (vector staging)
};

// Launch shape of the few-row kernel.
struct Shape {
    int warps;              // 4 or 8
    int tpw;                // column tiles per warp, 1 or 2
    int splits;             // 1..8
    int ctas_n;             // CTAs along N (grid y)
    size_t smem;            // dynamic shared memory bytes
};

struct LaunchOpts {
    bool pdl;               // programmatic dependent launch
};

// Few-row kernel launcher for one (format, xdtype, group); defined in the
// per-format .cu files.  Returns a CUDA error code.
cudaError_t launch_verify(lbv_format fmt, lbv_dtype xt, int group, const Shape& sh,
                          const VerifyParams& p, const LaunchOpts& o, cudaStream_t st);
// Shared memory the few-row kernel needs for a slice of `cps` chunks.
size_t verify_smem_bytes(lbv_format fmt, int group, int warps, int tpw, int cps);
// Sets the kernel's dynamic shared memory limit (once per kernel/shape).
cudaError_t prepare_verify(lbv_format fmt, lbv_dtype xt, int group, const Shape& sh);
// Max resident CTAs per SM for the shape (0 if it does not fit).
int verify_occupancy(lbv_format fmt, lbv_dtype xt, int group, const Shape& sh);

// One-row (GEMV) path, FMA pipe, run once per row.
cudaError_t launch_gemv(lbv_format fmt, lbv_dtype xt, int group, const VerifyParams& p,
                        int row, cudaStream_t st);

cudaError_t launch_fwht128(const void* X, void* Xr, int M, int K, lbv_dtype dt,
                           const uint32_t* signs, cudaStream_t st);

cudaError_t launch_dequant(lbv_format fmt, int group, const uint4* codes, const uint8_t* side,
                           int K, int N, int ntiles, int nchunks, uint16_t* W, cudaStream_t st);

}  // namespace lbv

struct lbv_plan {
    lbv_format fmt;
    lbv_dtype xdtype;
    int K, N, group;
    unsigned flags;
    int device, sms;
    lbv::FmtInfo fi;
    lbv::Layout layout;
    lbv::Shape shape;        // few-row launch shape
    int use_gemv[9];         // per M (1..8): 1 = run the 1-row path M times
    int crossover;           // smallest M that uses the few-row kernel
    float measured_us[9][2]; // per M: [few-row, 1-row x M] (LBV_PLAN_MEASURE), else 0
};
