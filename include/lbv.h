/*
 * lbv.h -- few-row low-bit verify matmul for GB300 (sm_103a).
 *
 *   Y[M,N] = X[M,K] . dequant(Wp)[K,N],   1 <= M <= 8 drafted rows.
 *
 * Wp is a packed low-bit weight matrix that is consumed directly: every
 * weight is decoded once, in registers, and used against every row; it is
 * never expanded in memory.  (Ishizuki README, "Kernels written for the
 * verify": the verify kernel decodes each weight once into a matrix fragment
 * and multiplies it against every drafted row; Bonsai-27B-mlx-1bit model card:
 * packed weights are consumed directly, never expanded back to FP16.)
 *
 * Conventions for every entry point:
 *   - Plain C ABI: pointers and sizes only.  "dev" pointers are CUDA device
 *     memory of the current device, "host" pointers are host memory.
 *   - The caller owns every buffer.  The library never allocates in
 *     lbv_verify_gemm, lbv_verify_fused, lbv_verify_grouped, lbv_fwht128 or
 *     lbv_dequant_fp16.  Plans are created and
 *     destroyed by the caller and are immutable in between (safe to share
 *     between host threads).
 *   - Device work is asynchronous on the given stream; a status of LBV_OK
 *     means the work was enqueued.  Errors are returned, never aborted on; no
 *     kernel traps.  lbv_last_error() gives a thread-local message for the
 *     last failing call of the calling thread.
 *   - X rows are fp16 or bf16 (the plan's xdtype), row-major with leading
 *     dimension ldx (elements); Y is fp32 row-major with leading dimension ldy.
 *     Rows >= M of Y are never written.
 */
#ifndef LBV_H
#define LBV_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define LBV_API __attribute__((visibility("default")))
#else
#define LBV_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (binary-compatible with cudaStream_t); NULL = legacy stream. */
typedef struct CUstream_st* lbv_stream;

typedef enum {
    LBV_OK = 0,
    LBV_ERR_INVALID_ARG = 1,   /* bad pointer, size, M, dtype or leading dimension */
    LBV_ERR_UNSUPPORTED = 2,   /* valid request this build does not implement     */
    LBV_ERR_CUDA = 3,          /* a CUDA runtime call failed (message has details) */
    LBV_ERR_WORKSPACE = 4,     /* caller buffer too small                           */
    LBV_ERR_TIMEOUT = 5,       /* a bounded device wait gave up                     */
    LBV_ERR_BOUNDS = 6         /* a kernel's own range check failed (an internal
                                  error: the access was skipped, the output is wrong) */
} lbv_status;

typedef enum {
    /* 1-bit sign, one fp16 scale per 128 K-weights of a column: bit 0 -> -s,
     * bit 1 -> +s, 1.125 bits/weight.  Bonsai-27B-mlx-1bit model card,
     * format description. */
    LBV_FMT_SIGN1_G128 = 0,
    /* 2-bit affine groups, w = s*q + b, q in {0..3}, fp16 (s, b) per group of
     * 32, 64 or 128 K-weights: 2 + 32/g bits/weight.  Ishizuki README ("plain
     * MLX affine packs"); dflash-mlx-bonsai2 README ("Why"). */
    LBV_FMT_AFFINE2 = 1,
    /* GGUF Q4_0 blocks of 32: fp16 d and 16 bytes of nibbles, w = d*(q-8),
     * 4.5 bits/weight.  Ishizuki README, "Credits" (GGUF blocks read as they
     * are). */
    LBV_FMT_Q4_0 = 2
} lbv_format;

typedef enum { LBV_F16 = 0, LBV_BF16 = 1 } lbv_dtype;

/* Plan flags. */
#define LBV_PLAN_MEASURE     0x1u  /* time the candidate launch shapes (as
                                      back-to-back launches over copies of
                                      scratch weights, >= 2x L2, after an L2
                                      flush) and the 1-row path at plan
                                      creation and keep the fastest per row
                                      count (allocates and synchronises
                                      inside lbv_plan_create) */
#define LBV_PLAN_FORCE_FEWROW 0x2u /* always use the few-row kernel           */
#define LBV_PLAN_FORCE_GEMV   0x4u /* always use the 1-row path (run per row) */
#define LBV_PLAN_PDL          0x8u /* launch with programmatic dependent launch:
                                      the kernel starts streaming Wp before the
                                      previous kernel on the stream has finished
                                      (X is read and Y written only after it has).
                                      Only valid if the kernel launched just
                                      before on the stream never writes Wp. */
#define LBV_PLAN_TCGEN05     0x10u /* use the tcgen05 few-row kernel (A operand
                                      in tensor memory, 128-column tiles) for
                                      every M.  Such a plan reads its own device
                                      layout: pack with lbv_plan_pack and size
                                      buffers with lbv_plan_packed_bytes.  Not
                                      combinable with LBV_PLAN_FORCE_GEMV. */
#define LBV_PLAN_TC_E4M3      0x40u /* use the e4m3 tensor-memory kernel for every M
                                      (1-bit sign g128 and 2-bit affine g128
                                      only, K % 128 == 0; LBV_ERR_UNSUPPORTED
                                      otherwise): weights decoded to e4m3 bytes
                                      in tensor memory, the activations split
                                      exactly into three e4m3 terms per row,
                                      tcgen05.mma kind::f8f6f4, fp32
                                      accumulation.  Such a plan reads its own
                                      device layout: pack with lbv_plan_pack and
                                      size buffers with lbv_plan_packed_bytes.
                                      Not combinable with LBV_PLAN_TCGEN05,
                                      LBV_PLAN_FORCE_GEMV or
                                      LBV_PLAN_TEST_WAIT_LIMIT. */
#define LBV_PLAN_TEST_WAIT_LIMIT 0x20u /* test only: the few-row kernel's waits
                                      on its weight stages give up after 256
                                      tries, and the first warp of the first
                                      CTA leaves its second stage's copy out,
                                      so that wait runs out on purpose: the
                                      warp stops, waits (with the normal
                                      limit) for the copies it did issue and
                                      the kernel ends; the plan's device status
                                      then reports LBV_ERR_TIMEOUT and the
                                      output is incomplete.  Not combinable with
                                      LBV_PLAN_TCGEN05, LBV_PLAN_FORCE_GEMV or
                                      LBV_PLAN_MEASURE. */

/* Kernel ids reported by lbv_plan_query. */
#define LBV_KERNEL_FEWROW    1     /* mma.sync few-row kernel (default)       */
#define LBV_KERNEL_GEMV      2     /* 1-row path, run once per row           */
#define LBV_KERNEL_FEWROW_TC 3     /* tcgen05 few-row kernel (LBV_PLAN_TCGEN05) */
#define LBV_KERNEL_FEWROW_TC8 4    /* e4m3 tensor-memory kernel (LBV_PLAN_TC_E4M3) */

typedef struct lbv_plan lbv_plan;   /* opaque, library-owned */

/* ------------------------------------------------------------------------ */
/* Packing (host): canonical file layout -> the library's device layout.     */

/*
 * Size in bytes of the default device layout (the one the mma.sync few-row
 * kernel and the 1-row path read) of a K x N matrix, or 0 for an invalid
 * shape.  One record per (16-column tile, K chunk), tile-major.  For
 * N % 16 == 0 and K a multiple of the format's chunk (256 for sign1, 128 for
 * affine2, 64 for Q4_0) it equals the canonical size exactly
 * (1.125, 2 + 32/g and 4.5 bits per weight); otherwise the last column tile
 * and K chunk are padded with zero codes and zero scales, which contribute
 * exactly 0.  `group` is ignored except for LBV_FMT_AFFINE2.
 */
LBV_API size_t lbv_packed_bytes(lbv_format fmt, int K, int N, int group);

/*
 * bits: host uint32 [N][K/32], bit k%32 of word k/32 = sign bit of weight
 * (k, n) (little end first); scales: host fp16 bit patterns [N][K/128].
 * K % 128 == 0.  out: host buffer of lbv_packed_bytes() bytes.
 * Bonsai-27B-mlx-1bit model card, format description.
 */
LBV_API lbv_status lbv_pack_sign_g128(const uint32_t* bits, const uint16_t* scales, int K, int N,
                              void* out, size_t out_bytes);

/*
 * codes: host uint32 [N][K/16], code of weight (k, n) in bits 2*(k%16)..+1 of
 * word k/16 ("16 per uint32, little end first"); scales, biases: host fp16
 * bit patterns [N][K/group], group in {32, 64, 128}, K % group == 0.
 */
LBV_API lbv_status lbv_pack_affine2(const uint32_t* codes, const uint16_t* scales,
                            const uint16_t* biases, int K, int N, int group, void* out,
                            size_t out_bytes);

/*
 * blocks: host bytes [N][K/32][18] in GGUF order: d (fp16, little-endian),
 * then qs[16]; element j < 16 = qs[j] & 15, element j + 16 = qs[j] >> 4.
 * K % 32 == 0.
 */
LBV_API lbv_status lbv_pack_q4_0(const uint8_t* blocks, int K, int N, void* out, size_t out_bytes);

/* ------------------------------------------------------------------------ */
/* Plans: all kernel and launch-shape selection happens here, once per shape
 * (Ishizuki releases v0.6.1: each weight shape's kernel is set up once when
 * the model loads; the verify kernel starts at the row count where it is
 * faster, per matrix).  The activation dtype is part of the key (Ishizuki
 * releases v0.6.1, "Verify kernels no longer mix up precisions"). */

/* Creates a plan for the current device.  Returns LBV_ERR_INVALID_ARG for
 * K, N <= 0 or a K the format cannot hold, LBV_ERR_UNSUPPORTED for a group
 * other than 32/64/128 (affine2) or a K so large that no K split (at most 8
 * CTAs) leaves each CTA's slice of X room in shared memory beside its weight
 * ring: on GB300 about 44-53 thousand, by format and activation dtype.  *out
 * is NULL on failure. */
LBV_API lbv_status lbv_plan_create(lbv_format fmt, int K, int N, int group, lbv_dtype xdtype,
                           unsigned flags, lbv_plan** out);
LBV_API lbv_status lbv_plan_destroy(lbv_plan* plan);

/* Size in bytes of the device layout the plan's kernels read: equal to
 * lbv_packed_bytes() of the plan's shape, except for LBV_PLAN_TCGEN05 plans,
 * whose layout is one record per (128-column tile, K chunk) (128 K for sign1
 * and affine2 g128, 64 K otherwise), padded with zero codes and scales, and
 * LBV_PLAN_TC_E4M3 plans, whose layout is one record per (128-column tile,
 * 32-column quarter, 128-K group), padded the same way.  0 for a NULL plan. */
LBV_API size_t lbv_plan_packed_bytes(const lbv_plan* plan);

/* Packs canonical host arrays into the plan's device layout (host buffer of
 * lbv_plan_packed_bytes() bytes).  part0..part2 are the arrays of
 * lbv_pack_sign_g128 (bits, scales, unused), lbv_pack_affine2 (codes, scales,
 * biases) or lbv_pack_q4_0 (blocks, unused, unused), laid out as documented
 * there.  LBV_ERR_WORKSPACE if out_bytes is too small. */
LBV_API lbv_status lbv_plan_pack(const lbv_plan* plan, const void* part0, const void* part1,
                                 const void* part2, void* out, size_t out_bytes);

/* For a row count M (1..8): the kernel that lbv_verify_gemm will launch
 * (LBV_KERNEL_FEWROW, LBV_KERNEL_GEMV, LBV_KERNEL_FEWROW_TC or LBV_KERNEL_FEWROW_TC8), its K
 * split (cluster size) and the
 * workspace it needs (always 0 in this build).  Any output may be NULL. */
LBV_API lbv_status lbv_plan_query(const lbv_plan* plan, int M, int* kernel_id, int* splits,
                          size_t* workspace_bytes);

/* The plan's launch shape for the few-row kernel: warps per CTA, column tiles
 * (16 columns each) per warp, K split and CTAs along N.  For tests and
 * benchmarks; any output may be NULL. */
LBV_API lbv_status lbv_plan_shape(const lbv_plan* plan, int* warps, int* tiles_per_warp, int* splits,
                          int* ctas_n);

/* Overrides the few-row launch shape ((warps, tiles_per_warp) in {(8, 2),
 * (8, 4), (16, 1), (16, 2)}, splits in 1..8, ctas_n = clusters along N >= 1, or 0 for as many
 * as can be resident).  Returns
 * LBV_ERR_UNSUPPORTED if the shape does not fit the device (shared memory).
 * For tuning sweeps; not thread-safe against concurrent verify calls.
 * LBV_PLAN_TCGEN05 plans report warps = tiles_per_warp = 0 and ignore both
 * on input (their kernel has a fixed CTA: three decode warpgroups and one
 * MMA warp each); so do LBV_PLAN_TC_E4M3 plans (four warpgroups of four
 * decode warps and one MMA warp each), whose splits must be 1, 2, 4 or 8. */
LBV_API lbv_status lbv_plan_set_shape(lbv_plan* plan, int warps, int tiles_per_warp, int splits,
                              int ctas_n);

/* With LBV_PLAN_MEASURE: the measured cold-L2 time (us) of the few-row kernel
 * and of the 1-row path run M times at row count M, and the crossover (the
 * smallest M that uses the few-row kernel; 9 if none).  Zero times without
 * LBV_PLAN_MEASURE.  Any output may be NULL. */
LBV_API lbv_status lbv_plan_measured(const lbv_plan* plan, int M, float* fewrow_us, float* gemv_us,
                             int* crossover);

/* Reads (and clears) the plan's device status word: LBV_ERR_TIMEOUT if a
 * verify kernel of this plan gave up a bounded wait for its weight copies
 * since the last check (its output is then incomplete), LBV_ERR_BOUNDS if a
 * kernel found one of its copy or buffer ranges outside its bounds and skipped
 * the access (the checked build's range checks, and the e4m3 kernel's
 * shared-memory carve-up check in every build), else LBV_OK.  Synchronises
 * with the device. */
LBV_API lbv_status lbv_plan_device_status(const lbv_plan* plan);

/*
 * Rows-per-call statistics ("dflash-mlx-bonsai2" README, Commands: the fork
 * keeps a histogram of how many drafted rows each verify call carried and
 * prints it at exit on request).  counts: host array of 8; counts[m - 1] =
 * the calls of this plan with M = m (lbv_verify_gemm, lbv_verify_fused,
 * lbv_verify_fused_noalloc) that returned LBV_OK since the plan was created
 * or last reset.  Failed calls and the plan's own launch measurement are not
 * counted.  A call counts when it is enqueued: one captured into a CUDA graph
 * counts once, at capture, since the graph's replays do not pass through the
 * library.  Counting is atomic: plans stay safe to share between threads.
 * LBV_ERR_INVALID_ARG for a NULL plan or counts.
 */
LBV_API lbv_status lbv_plan_rows_histogram(const lbv_plan* plan, uint64_t* counts);
LBV_API lbv_status lbv_plan_rows_reset(lbv_plan* plan);

/* ------------------------------------------------------------------------ */
/* The verify matmul.                                                         */

/*
 * Y[m][n] = sum_k X[m][k] * w[k][n] for m < M, n < N, fp32 accumulation.
 * X: dev [M][ldx] (plan xdtype), ldx >= K; Wp: dev, the device layout from
 * lbv_pack_* (lbv_packed_bytes bytes, 16-byte aligned); Y: dev fp32 [M][ldy],
 * ldy >= N.  1 <= M <= 8, else LBV_ERR_INVALID_ARG.  workspace may be NULL
 * with workspace_bytes 0 (no plan in this build needs one).  Rows >= M cost
 * the same as a full block of 8 and are never read or written (Ishizuki
 * releases v0.6.1; dflash-mlx-bonsai2 README: 2-8-row calls are padded to 8).
 * The result of row m depends only on row m of X (bitwise).
 */
LBV_API lbv_status lbv_verify_gemm(const lbv_plan* plan, const void* X, int M, int ldx,
                           const void* Wp, float* Y, int ldy, void* workspace,
                           size_t workspace_bytes, lbv_stream stream);

/*
 * Blockwise normalized Walsh-Hadamard rotation of activation rows:
 * Xr[m][b*128 + i] = RNE( sum_j H[i][j] * sx_j / sqrt(128) ), where
 * H[i][j] = (-1)^popcount(i & j) (Sylvester, natural order), x_j = X[m][b*128+j]
 * and sx_j = -x_j where bit (b*128+j) of `signs` is set (signs: dev uint32
 * [K/32], NULL for none).  The sum is exact and the one rounding is to the
 * dtype, so the result is the correctly rounded rotation.  X, Xr: dev [M][K]
 * contiguous, K % 128 == 0, 1 <= M <= 8; in place (X == Xr) allowed.
 * dflash-mlx-bonsai2 README, "What this fork adds" (fused sign, Hadamard
 * prep); Ishizuki README (2-bit Hadamard-rotated weights).
 */
LBV_API lbv_status lbv_fwht128(const void* X, void* Xr, int M, int K, lbv_dtype dtype,
                       const uint32_t* signs, lbv_stream stream);

/* ------------------------------------------------------------------------ */
/* Fused head: the rotation as the verify's prologue and a greedy argmax as  */
/* its epilogue, in one launch of the few-row kernel.                        */

#define LBV_FUSED_ROTATE 0x1u  /* rotate X blockwise before the product        */
#define LBV_FUSED_ARGMAX 0x2u  /* per-row argmax over the N logits              */

/* Bytes of the workspace an argmax call needs (128). */
LBV_API size_t lbv_fused_workspace_bytes(void);

/*
 * Y[m][:] = X'[m][:] . dequant(Wp) for rows m < M, with in the same kernel:
 *   LBV_FUSED_ROTATE: X' is the blockwise rotation of lbv_fwht128 (signs
 *     optional, dev uint32 [K/32] or NULL), computed per CTA from the staged
 *     X tile and kept in shared memory.  Its arithmetic differs from
 *     lbv_fwht128's: fp32 sums (the 16-point stages on the tensor cores), one
 *     fp32 multiplication by 1/sqrt(128), one rounding to the dtype; a
 *     rotated element can differ from the correctly rounded one by a unit in
 *     the last place.  Without it X' = X.  Needs K % 128 == 0.
 *   LBV_FUSED_ARGMAX: argmax_idx[m] (dev int32 [M]) = the column of the
 *     largest fp32 logit of row m, the smallest such column on ties, -0 equal
 *     to +0, the first NaN if any; argmax_val[m] (dev fp32 [M], or NULL) =
 *     that logit, bit for bit the value Y would hold.  The logits need not be
 *     written: Y may then be NULL (ldy ignored).
 * dflash-mlx-bonsai2 README, "What this fork adds" (the verify GEMM with a
 * fused sign, Hadamard and row-sum prep) and "What it does to the numbers"
 * (greedy decoding; acceptance decided by the argmax, up to fp16 ties).
 *
 * The other arguments and rules are those of lbv_verify_gemm, except that
 * the few-row kernel is used at every M (never the 1-row path).
 * workspace: dev, 16-byte aligned, >= lbv_fused_workspace_bytes(), needed
 * with LBV_FUSED_ARGMAX (else ignored; LBV_ERR_WORKSPACE when missing or
 * short).  The caller zeroes it once before its first use; every call leaves
 * it zeroed when its kernel completes.  Calls that may run at the same time
 * (other streams) need distinct workspaces; calls in one stream can share one.
 * Errors: LBV_ERR_INVALID_ARG as lbv_verify_gemm, for unknown ops bits, for
 * no output (Y NULL without LBV_FUSED_ARGMAX), for argmax_idx NULL with
 * LBV_FUSED_ARGMAX and for misaligned signs, argmax_idx or argmax_val;
 * LBV_ERR_UNSUPPORTED for LBV_PLAN_TCGEN05 plans (LBV_PLAN_TC_E4M3 plans
 * support every op), for the rotation with
 * K % 128 != 0 or with K slices of the plan's launch shape that are not
 * whole 128-element blocks.  If a bounded wait in the kernel gives up, the
 * plan's device status records it (lbv_plan_device_status) and argmax_idx
 * may be -1.
 */
LBV_API lbv_status lbv_verify_fused(const lbv_plan* plan, const void* X, int M, int ldx,
                                    const void* Wp, unsigned ops, const uint32_t* signs,
                                    float* Y, int ldy, int32_t* argmax_idx, float* argmax_val,
                                    void* workspace, size_t workspace_bytes, lbv_stream stream);

/*
 * lbv_verify_fused without a caller workspace, for callers that cannot
 * allocate device memory: an engine whose memory is one arena sized at start-up
 * (nothing may call cudaMalloc after that), or host code that must not make a
 * blocking allocation on its decode path.  The argmax scratch (the 128-byte
 * workspace layout; 256 bytes reserved) is a device array of the library
 * module itself, one per device, held by every device that loads the library
 * until the process exits.  Set-up: the first call on a device looks up the
 * array's device address (cudaGetSymbolAddress) and clears it on that call's
 * stream, so make the first call on each device before any stream capture; a
 * cudaDeviceReset invalidates the looked-up address for the rest of the
 * process.  Every call leaves the scratch zero.  The library allocates
 * nothing.  M > 8 is rejected (the scratch holds 8 rows).  Other arguments,
 * rules and errors as lbv_verify_fused.  Races: the scratch is shared by every
 * call on a device, so calls that could overlap in time (other streams, other
 * host threads without ordering) must not be made; calls in one stream are
 * ordered and safe.  The pages have no counterpart of this entry point.
 */
LBV_API lbv_status lbv_verify_fused_noalloc(const lbv_plan* plan, const void* X, int M, int ldx,
                                            const void* Wp, unsigned ops,
                                            const uint32_t* signs, float* Y, int ldy,
                                            int32_t* argmax_idx, float* argmax_val,
                                            lbv_stream stream);

/* ------------------------------------------------------------------------ */
/* Grouped verify: independent problems of one format and dtype in one       */
/* launch -- a model's matrices (the Q4_0 layer stack) or routed experts,    */
/* each with its own rows.                                                   */

typedef struct lbv_group lbv_group;     /* opaque, library-owned */

/* One problem of a grouped call (the i-th shape of the group). */
typedef struct lbv_problem {
    const void* X;      /* dev [M][ldx], the group's dtype                      */
    int M;              /* rows, 0..8; 0 skips the problem (nothing is written)  */
    int ldx;            /* >= K_i                                               */
    const void* Wp;     /* dev, the default device layout of K_i x N_i
                           (lbv_pack_*, lbv_packed_bytes), 16-byte aligned      */
    float* Y;           /* dev [M][ldy] fp32, rows >= M untouched               */
    int ldy;            /* >= N_i                                               */
} lbv_problem;

/*
 * Creates a group plan for `count` (1..256) problems of shapes K[i] x N[i]
 * (host arrays, each valid for the format as in lbv_plan_create).  The
 * problems of a launch class share one launch shape: 16 warps, two tiles per
 * unit, a K split (cluster size) that suits each of them, and cluster rows
 * (at least two waves of resident clusters) divided among them in proportion
 * to their packed bytes.  There is one class when some split of 1..8 suits
 * every problem (the split needing the fewest CTAs); otherwise each problem
 * joins the class of the smallest split at which its X slice fits in shared
 * memory.  flags: LBV_PLAN_PDL and/or LBV_PLAN_MEASURE, which times, per
 * class, the default shape and one to six waves of every split from the
 * class's own up to 8 on scratch buffers (allocated and freed here, cold L2,
 * M = 8) and keeps the fastest.  LBV_ERR_UNSUPPORTED if a problem fits no
 * split of 1..8.
 * Ijah README, "What's new (v0.2)": grouped routed-expert verify, each
 * expert's weights read once per verify cycle for all the rows routed to it,
 * bit-identical output.  Ishizuki README, acknowledgements: a megakernel over
 * a model's matrices needs a grid-wide barrier; these problems are
 * independent, so their launches need none.
 */
LBV_API lbv_status lbv_group_create(lbv_format fmt, int group, lbv_dtype xdtype, int count,
                                    const int* K, const int* N, unsigned flags, lbv_group** out);
LBV_API lbv_status lbv_group_destroy(lbv_group* group);

/* Launch classes of the plan (0 for NULL), and the class of a problem (-1 if
 * out of range). */
LBV_API int lbv_group_launches(const lbv_group* group);
LBV_API int lbv_group_problem_launch(const lbv_group* group, int problem);

/* Launch shape of class `launch`: tiles per warp unit (1 or 2), K split,
 * cluster rows with every problem of the class active.  set_shape puts every
 * problem in one class with the given shape; LBV_ERR_UNSUPPORTED if the split
 * does not suit every problem or the shape does not fit. */
LBV_API lbv_status lbv_group_shape(const lbv_group* group, int launch, int* tpw, int* splits,
                                   int* rows);
LBV_API lbv_status lbv_group_set_shape(lbv_group* group, int tpw, int splits, int rows);

/*
 * Y_i[m][:] = X_i[m][:] . dequant(Wp_i) for every problem i (problems: host
 * array of `count`, read during the call), one launch per class with an
 * active problem, in order on `stream`.  Row m of problem i is bit for bit
 * what lbv_verify_gemm gives with a plan of the same shape and the K split of
 * the problem's class (lbv_plan_set_shape(plan, 16, tpw, splits, 0)).
 * Problems with M = 0 get no clusters; a call with every M = 0 launches
 * nothing.  Errors: LBV_ERR_INVALID_ARG for M outside 0..8, null or
 * misaligned pointers of an active problem, ldx < K_i or ldy < N_i.  The
 * library allocates nothing.
 */
LBV_API lbv_status lbv_verify_grouped(const lbv_group* group, const lbv_problem* problems,
                                      lbv_stream stream);

/* As lbv_plan_device_status, for the group's kernels. */
LBV_API lbv_status lbv_group_device_status(const lbv_group* group);

/* As lbv_plan_rows_histogram, per active problem of each lbv_verify_grouped
 * call that returned LBV_OK: counts[m - 1] = problems run with M = m. */
LBV_API lbv_status lbv_group_rows_histogram(const lbv_group* group, uint64_t* counts);
LBV_API lbv_status lbv_group_rows_reset(lbv_group* group);

/*
 * The same counts over every plan and group of the process since the library
 * was loaded (not reset by the calls above).  With the environment variable
 * LBV_VERIFY_STATS set (and not "0"), the library prints them to stderr when
 * the process exits: one line, "lbv: verify rows per call: 1:n1 ... 8:n8
 * (calls C, mean rows R)".
 */
LBV_API lbv_status lbv_rows_histogram(uint64_t* counts);

/*
 * Test export: X' exactly as lbv_verify_fused with LBV_FUSED_ROTATE computes
 * it inside the verify kernel (the same device code, run on its own), for
 * element-by-element checks.  Arguments as lbv_fwht128 (in place allowed).
 */
LBV_API lbv_status lbv_fused_rotation(const void* X, void* Xr, int M, int K, lbv_dtype dtype,
                                      const uint32_t* signs, lbv_stream stream);

/*
 * Test export: the dense fp16 dequantized matrix, W[k][n] (dev, [K][N]
 * row-major, ldw = N) rounded once to nearest even from the exact weight.
 * Not part of the verify path (the verify never expands weights).
 */
LBV_API lbv_status lbv_dequant_fp16(const lbv_plan* plan, const void* Wp, uint16_t* W,
                            lbv_stream stream);

/* Thread-local message of the calling thread's last failing call ("" if none). */
LBV_API const char* lbv_last_error(void);

/* Library version string. */
LBV_API const char* lbv_version(void);

/*
 * 1 in the checked build (liblbv_checked.so, compiled with LBV_CHECKED), 0 in
 * the release library.  The checked build's kernels test, before each access
 * they cannot prove in range by construction, that it lies inside its buffer:
 * the shared-memory carve-up against the launch's dynamic shared memory, every
 * weight copy against the packed matrix and its ring slot, the X slice against
 * K and its row buffer, a stage's chunks against the staged slice, the K split's
 * partial slots against their buffer.  A failed test sets the status word's
 * bounds bit (LBV_ERR_BOUNDS from lbv_plan_device_status) and skips the access;
 * the kernel still ends, and its output is then wrong.  It stands in for a
 * memory checker where none can run.
 */
LBV_API int lbv_checked_build(void);

#ifdef __cplusplus
}
#endif
#endif /* LBV_H */
