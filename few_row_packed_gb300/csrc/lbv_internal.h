// lbv_internal.h -- plan object, launch parameters and the launcher entry
// points each kernel translation unit exports to the C-ABI layer.
#pragma once

#include <cuda_runtime.h>

#include <atomic>

#include "layout.h"
#include "t8_layout.h"
#include "tc_layout.h"

namespace lbv {

// Parameters of one few-row verify launch (passed by value to the kernel).
struct VerifyParams {
    const void* X;          // [M][ldx] fp16 / bf16
    const uint8_t* W;       // packed records [tile][chunk] (layout.h)
    float* Y;               // [M][ldy]
    unsigned* err;          // device status word of the plan (bounded waits)
    int ldx, ldy;
    int M, K, N;
    int ntiles, nchunks;
    int splits;             // K slices == cluster size along grid x
    int cps;                // chunks per slice (the last slice may be shorter)
    int x_vec;              // 1: X rows 16-byte aligned (vector staging)
    unsigned zero;          // always 0 (keeps decode constants in registers)
    int wait_limit;         // tries of a main-loop ring wait (0: the default, ~1 s)
    int skip_q;             // ring stage the first warp of CTA 0 does not issue (-1: none)
    // fused head (lbv_verify_fused); lbv_verify_gemm leaves rot = 0,
    // amax_keys = NULL and store_y = 1
    int rot;                // 1: rotate the staged X blockwise (FWHT-128) first
    int store_y;            // 0: the logits Y are not written
    const uint32_t* signs;  // rotation: optional K-bit +-1 mask (NULL: none)
    unsigned long long* amax_keys;  // workspace [8]: running argmax keys (NULL: no argmax)
    unsigned* amax_done;    // workspace: CTAs finished with their keys
    int* amax_idx;          // [M] argmax column of each row
    float* amax_val;        // [M] its logit (NULL: not written)
};

// Grouped verify: one problem of the launch (a compact VerifyParams).
struct GroupedProblem {
    const void* X;
    const uint8_t* W;
    float* Y;
    int ldx, ldy;
    int M, K, N;            // M = 0: skipped
    int ntiles, nchunks;
    int cps;                // chunks per K slice (the launch's split)
    int x_vec;
};

// Most problems of one grouped launch (the parameters travel in the kernel's
// parameter space, about 17 KB at this size).
constexpr int kMaxGroup = 256;

struct GroupedParams {
    unsigned* err;          // device status word of the group
    int splits;             // K slices == cluster size, all problems
    int count;              // problems
    int ybegin[kMaxGroup + 1];   // cluster rows of problem i: [ybegin[i], ybegin[i + 1])
    GroupedProblem prob[kMaxGroup];
};

// Launch shape of the few-row kernel.
struct Shape {
    int warps;              // 8 or 16
    int tpw;                // column tiles per warp unit, 1 or 2
    int splits;             // K slices (cluster size), 1..8
    int ctas_n;             // clusters along N (grid y); each owns a contiguous tile range
    size_t smem;            // dynamic shared memory bytes
};

// Dynamic shared-memory limit set on every few-row kernel function: the
// largest any plan may request, so plans of one kernel with different shapes
// never lower each other's limit (the attribute is per function, not per
// launch).
constexpr int kMaxDynSmem = 220 * 1024;

struct LaunchOpts {
    bool pdl;               // programmatic dependent launch
};

// One-row (GEMV) path, FMA pipe, run once per row.
cudaError_t launch_gemv(lbv_format fmt, lbv_dtype xt, int group, const VerifyParams& p,
                        int row, cudaStream_t st);

cudaError_t launch_fwht128(const void* X, void* Xr, int M, int K, lbv_dtype dt,
                           const uint32_t* signs, cudaStream_t st);

// Test export: the fused head's rotation on its own (fused_aux.cu).
cudaError_t launch_fused_rotation(const void* X, void* Xr, int M, int K, lbv_dtype dt,
                                  const uint32_t* signs, cudaStream_t st);

// Scratch of lbv_verify_fused_noalloc in the module's device memory
// (fused_aux.cu): its size, and its address on the current device; *first is
// true on the first request for a device.
size_t noalloc_scratch_bytes();
cudaError_t noalloc_scratch(void** out, bool* needs_clear);
void noalloc_scratch_cleared();

cudaError_t launch_dequant(lbv_format fmt, int group, const uint8_t* Wp, int K, int N,
                           int ntiles, int nchunks, uint16_t* W, cudaStream_t st);

}  // namespace lbv

// Plan of a grouped verify: the problems' shapes and their launches.  Each
// problem belongs to one launch class; a class's problems share a launch
// shape (warps, tiles per unit, K split, cluster rows) and run in one launch.
namespace lbv {
constexpr int kMaxGroupLaunches = 8;
struct GroupLaunch {
    Shape shape;             // warps, tpw, splits, ctas_n = cluster rows with all active, smem
    int resident;            // clusters of the shape resident at once
    int rows_target;         // R the class's cluster rows are divided from (divide_rows)
    int tiles_max;           // most tiles of one cluster row (sizes the K-split partials)
};
}  // namespace lbv

struct lbv_group {
    lbv_format fmt;
    lbv_dtype xdtype;
    int group;
    unsigned flags;
    int device, sms;
    int count;
    lbv::FmtInfo fi;
    int nlaunch;                               // launch classes
    lbv::GroupLaunch launch[lbv::kMaxGroupLaunches];
    int cls[lbv::kMaxGroup];                   // launch class of each problem
    int rows_plan[lbv::kMaxGroup];             // its cluster rows with every problem active
    int K[lbv::kMaxGroup], N[lbv::kMaxGroup];
    int ntiles[lbv::kMaxGroup], nchunks[lbv::kMaxGroup], cps[lbv::kMaxGroup];
    double bytes[lbv::kMaxGroup];              // packed bytes of each problem
    unsigned* dev_err;
    // rows-per-call counts: [m - 1] = active problems with M = m, over the
    // calls that enqueued their launches
    mutable std::atomic<unsigned long long> rows_calls[8];
};

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
    unsigned* dev_err;       // device status word (set when a bounded wait gives up)
    float measured_us[9][2]; // per M: [few-row, 1-row x M] (LBV_PLAN_MEASURE), else 0
    // plans created with LBV_PLAN_TCGEN05: the tcgen05 kernel and its layout
    int tc;
    lbv::TcFmtInfo tc_fi;
    lbv::TcLayout tc_layout;
    lbv::TcShape tc_shape;
    // plans created with LBV_PLAN_TC_E4M3: the e4m3 tensor-memory kernel and its layout
    int t8;
    lbv::T8FmtInfo t8_fi;
    lbv::T8Layout t8_layout;
    lbv::T8Shape t8_shape;
    // rows-per-call counts: [m - 1] = verify calls with M = m that enqueued
    // their launches (the plan's own launch measurement is not counted)
    mutable std::atomic<unsigned long long> rows_calls[8];
};
