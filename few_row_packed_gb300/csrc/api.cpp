// api.cpp -- the C ABI of include/lbv.h: argument checks, host packers, plan
// selection and dispatch.  Every error is returned as an lbv_status with a
// thread-local message; nothing here aborts.
#include <cuda_runtime.h>

#include <algorithm>
#include <cmath>
#include <cstdarg>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <new>
#include <string>
#include <vector>

#include "lbv_internal.h"
#include "t8_api.h"
#include "tc_api.h"
#include "verify_ops.h"

namespace {

thread_local std::string g_err;

lbv_status fail(lbv_status st, const char* fmt, ...)
{
    char buf[512];
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(buf, sizeof buf, fmt, ap);
    va_end(ap);
    g_err = buf;
    return st;
}

lbv_status cuda_fail(cudaError_t e, const char* what)
{
    return fail(LBV_ERR_CUDA, "%s: %s (%s)", what, cudaGetErrorName(e), cudaGetErrorString(e));
}

// Rows-per-call counts of the whole process ([m - 1]: calls or active grouped
// problems with M = m), and the report at exit that LBV_VERIFY_STATS=1 asks
// for ("dflash-mlx-bonsai2" README, Commands: a rows-per-call histogram of the
// verify, printed at exit).
std::atomic<unsigned long long> g_rows[8];

void count_rows(std::atomic<unsigned long long> (&own)[8], int M)
{
    own[M - 1].fetch_add(1, std::memory_order_relaxed);
    g_rows[M - 1].fetch_add(1, std::memory_order_relaxed);
}

struct RowsReport {
    ~RowsReport()
    {
        const char* v = getenv("LBV_VERIFY_STATS");
        if (!v || !*v || strcmp(v, "0") == 0)
            return;
        unsigned long long calls = 0, rows = 0;
        for (int m = 1; m <= 8; ++m) {
            const unsigned long long c = g_rows[m - 1].load(std::memory_order_relaxed);
            calls += c;
            rows += c * (unsigned long long)m;
        }
        fprintf(stderr, "lbv: verify rows per call:");
        for (int m = 1; m <= 8; ++m)
            fprintf(stderr, " %d:%llu", m, g_rows[m - 1].load(std::memory_order_relaxed));
        fprintf(stderr, " (calls %llu, mean rows %.2f)\n", calls,
                calls ? (double)rows / (double)calls : 0.0);
    }
} g_rows_report;

const lbv::VerifyOps* ops_for(lbv_format fmt, int group)
{
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        return &lbv::sign1_ops;
    case LBV_FMT_AFFINE2:
        return group == 32 ? &lbv::affine2_g32_ops
               : group == 64 ? &lbv::affine2_g64_ops
                             : &lbv::affine2_g128_ops;
    case LBV_FMT_Q4_0:
        return &lbv::q4_0_ops;
    }
    return nullptr;
}

bool valid_fmt(int fmt)
{
    return fmt == LBV_FMT_SIGN1_G128 || fmt == LBV_FMT_AFFINE2 || fmt == LBV_FMT_Q4_0;
}

// The K granularity the canonical layout of each format can represent.
int k_quantum(lbv_format fmt, int group)
{
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        return 128;
    case LBV_FMT_AFFINE2:
        return group;          // also a multiple of 16 (codes per word)
    case LBV_FMT_Q4_0:
        return 32;
    }
    return 0;
}

// K slices of a split start at multiples of `step` chunks: whole 128-element
// blocks whenever K allows it, so the fused head can rotate each slice on its
// own (only Q4_0's 64-element chunks are shorter than a block).
int slice_step(const lbv_plan* P)
{
    return (P->K % 128 == 0 && P->fi.chunk_k < 128) ? 128 / P->fi.chunk_k : 1;
}

int shape_cps(const lbv::Shape& sh, int64_t nchunks, int step)
{
    const int cps = (int)((nchunks + sh.splits - 1) / sh.splits);
    return (cps + step - 1) / step * step;
}

// Shape bookkeeping: clamp the split so every slice has >= 1 chunk (a fixed
// point: shape_cps of the result equals the cps it was derived from).
void finish_shape(lbv::Shape& sh, int64_t nchunks, int step)
{
    const int cps = shape_cps(sh, nchunks, step);
    sh.splits = (int)((nchunks + cps - 1) / cps);
}

constexpr size_t kSmemCap = 220 * 1024;        // per CTA, of 227 KB
// Requesting more than half of an SM's shared memory keeps the scheduler from
// placing two CTAs of one grid on an SM while other SMs stay empty.
constexpr size_t kSmemOnePerSm = 116 * 1024;

// Bytes per (tile, chunk) of the device layout and X bytes per chunk staged.
size_t tile_chunk_bytes(const lbv_plan* P)
{
    return P->layout.rec_bytes;
}

// Fills sh.splits (clamped), sh.ctas_n and sh.smem for a (warps, tpw,
// splits) choice: one cluster of `splits` CTAs per `splits` SMs, as many
// clusters as can be resident at once, each owning a contiguous tile range.
// ctas_req > 0 caps the number of clusters.  Returns false if nothing fits.
bool complete_shape(const lbv_plan* P, lbv::Shape& sh, int ctas_req)
{
    const lbv::VerifyOps* ops = ops_for(P->fmt, P->group);
    finish_shape(sh, P->layout.nchunks, slice_step(P));
    const int cps = shape_cps(sh, P->layout.nchunks, slice_step(P));
    const int64_t ntiles = P->layout.ntiles;
    int64_t G = std::max<int64_t>(1, std::min<int64_t>(ntiles, P->sms / sh.splits));
    if (ctas_req > 0)
        G = std::min<int64_t>(G, ctas_req);
    for (int it = 0; it < 4; ++it) {
        const int tiles_max = (int)((ntiles + G - 1) / G);
        sh.smem = std::max(ops->smem(sh.warps, sh.tpw, cps, tiles_max, sh.splits), kSmemOnePerSm);
        if (sh.smem > kSmemCap)
            return false;
        sh.ctas_n = (int)G;
        if (ops->prepare(P->xdtype, sh) != cudaSuccess)
            return false;
        const int maxc = ops->max_clusters(P->xdtype, sh);
        if (maxc < 1)
            return false;
        if (G <= maxc)
            return true;
        G = maxc;
    }
    sh.smem = std::max(ops->smem(sh.warps, sh.tpw, cps, (int)((ntiles + G - 1) / G), sh.splits),
                       kSmemOnePerSm);
    sh.ctas_n = (int)G;
    return ops->prepare(P->xdtype, sh) == cudaSuccess;
}

// Default launch shape: 16 warps of two-tile units; the K split that
// minimises what the busiest warp of a CTA streams (its units times the
// slice) plus half the activation bytes the CTA stages.
lbv::Shape default_shape(lbv_plan* P)
{
    const int warps = 16, tpw = 2;
    lbv::Shape best = {warps, tpw, 1, 0, 0};
    double best_cost = 1e300;
    for (int s = 1; s <= 8; ++s) {
        lbv::Shape sh = {warps, tpw, s, 0, 0};
        if (!complete_shape(P, sh, 0) || sh.splits != s)
            continue;
        const int cps = shape_cps(sh, P->layout.nchunks, slice_step(P));
        const int64_t tmax = (P->layout.ntiles + sh.ctas_n - 1) / sh.ctas_n;
        const int64_t umax = ((tmax + tpw - 1) / tpw + warps - 1) / warps;
        const double cost = (double)umax * tpw * warps * cps * tile_chunk_bytes(P) +
                            0.5 * (double)cps * P->fi.chunk_k * 16.0;
        if (cost < best_cost * 0.98) {
            best_cost = cost;
            best = sh;
        }
    }
    return best;
}

}  // namespace

extern "C" {

const char* lbv_last_error(void)
{
    return g_err.c_str();
}

const char* lbv_version(void)
{
    return "lbv 0.1.0 (sm_103a)";
}

int lbv_checked_build(void)
{
#ifdef LBV_CHECKED
    return 1;
#else
    return 0;
#endif
}

size_t lbv_packed_bytes(lbv_format fmt, int K, int N, int group)
{
    lbv::FmtInfo fi;
    if (!valid_fmt(fmt) || K <= 0 || N <= 0)
        return 0;
    if (fmt != LBV_FMT_AFFINE2)
        group = fmt == LBV_FMT_SIGN1_G128 ? 128 : 32;
    if (!lbv::fmt_info(fmt, group, &fi))
        return 0;
    if (K % k_quantum(fmt, group) != 0 || (fmt == LBV_FMT_AFFINE2 && K % 16 != 0))
        return 0;
    return lbv::make_layout(fi, K, N).total;
}

// --------------------------------------------------------------------------
// Host packers.  Each walks the device layout (layout.h) and fetches the
// code of weight (k, n) from the canonical arrays.

lbv_status lbv_pack_sign_g128(const uint32_t* bits, const uint16_t* scales, int K, int N,
                              void* out, size_t out_bytes)
{
    g_err.clear();
    if (!bits || !scales || !out)
        return fail(LBV_ERR_INVALID_ARG, "lbv_pack_sign_g128: null pointer");
    const size_t need = lbv_packed_bytes(LBV_FMT_SIGN1_G128, K, N, 128);
    if (need == 0)
        return fail(LBV_ERR_INVALID_ARG, "lbv_pack_sign_g128: K=%d N=%d (need K%%128==0, N>0)", K, N);
    if (out_bytes < need)
        return fail(LBV_ERR_WORKSPACE, "lbv_pack_sign_g128: out_bytes %zu < %zu", out_bytes, need);
    lbv::FmtInfo fi;
    lbv::fmt_info(LBV_FMT_SIGN1_G128, 128, &fi);
    const lbv::Layout L = lbv::make_layout(fi, K, N);
    uint8_t* base = static_cast<uint8_t*>(out);
    const int wk = K / 32, sk = K / 128;
    auto bit = [&](int n, int k) -> uint32_t {
        if (n >= N || k >= K) return 0u;
        return (bits[(size_t)n * wk + k / 32] >> (k % 32)) & 1u;
    };
    for (int64_t tile = 0; tile < L.ntiles; ++tile)
        for (int64_t ch = 0; ch < L.nchunks; ++ch) {
            const size_t tc = (size_t)tile * L.nchunks + ch;
            uint32_t* codes = reinterpret_cast<uint32_t*>(base + tc * L.rec_bytes);
            uint16_t* side = reinterpret_cast<uint16_t*>(base + tc * L.rec_bytes + 512);
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, t = lane & 3;
                for (int wi = 0; wi < 4; ++wi) {
                    const int n = (int)tile * 16 + g + 8 * (wi & 1);
                    uint32_t w = 0;
                    for (int s = 0; s < 16; ++s) {
                        const int kt = (wi >> 1) * 8 + (s >> 1);
                        const int k0 = (int)ch * 256 + 16 * kt + 8 * (s & 1) + 2 * t;
                        w |= bit(n, k0) << s;
                        w |= bit(n, k0 + 1) << (16 + s);
                    }
                    codes[lane * 4 + wi] = w;
                }
            }
            for (int g = 0; g < 8; ++g)
                for (int j = 0; j < 2; ++j)
                    for (int hi = 0; hi < 2; ++hi) {
                        const int n = (int)tile * 16 + g + 8 * hi;
                        const int grp = (int)ch * 2 + j;
                        const bool ok = n < N && grp < sk;
                        side[g * 4 + 2 * j + hi] = ok ? scales[(size_t)n * sk + grp] : 0;
                    }
        }
    return LBV_OK;
}

lbv_status lbv_pack_affine2(const uint32_t* codes_in, const uint16_t* scales,
                            const uint16_t* biases, int K, int N, int group, void* out,
                            size_t out_bytes)
{
    g_err.clear();
    if (!codes_in || !scales || !biases || !out)
        return fail(LBV_ERR_INVALID_ARG, "lbv_pack_affine2: null pointer");
    if (group != 32 && group != 64 && group != 128)
        return fail(LBV_ERR_UNSUPPORTED, "lbv_pack_affine2: group %d (supported: 32, 64, 128)", group);
    const size_t need = lbv_packed_bytes(LBV_FMT_AFFINE2, K, N, group);
    if (need == 0)
        return fail(LBV_ERR_INVALID_ARG, "lbv_pack_affine2: K=%d N=%d group=%d (need K%%group==0)", K, N, group);
    if (out_bytes < need)
        return fail(LBV_ERR_WORKSPACE, "lbv_pack_affine2: out_bytes %zu < %zu", out_bytes, need);
    lbv::FmtInfo fi;
    lbv::fmt_info(LBV_FMT_AFFINE2, group, &fi);
    const lbv::Layout L = lbv::make_layout(fi, K, N);
    uint8_t* base = static_cast<uint8_t*>(out);
    const int wk = K / 16, gk = K / group, gpc = 128 / group;
    auto code = [&](int n, int k) -> uint32_t {
        if (n >= N || k >= K) return 0u;
        return (codes_in[(size_t)n * wk + k / 16] >> (2 * (k % 16))) & 3u;
    };
    for (int64_t tile = 0; tile < L.ntiles; ++tile)
        for (int64_t ch = 0; ch < L.nchunks; ++ch) {
            const size_t tc = (size_t)tile * L.nchunks + ch;
            uint32_t* codes = reinterpret_cast<uint32_t*>(base + tc * L.rec_bytes);
            uint16_t* side = reinterpret_cast<uint16_t*>(base + tc * L.rec_bytes + 512);
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, t = lane & 3;
                for (int wi = 0; wi < 4; ++wi) {
                    const int n = (int)tile * 16 + g + 8 * (wi & 1);
                    uint32_t w = 0;
                    for (int s = 0; s < 8; ++s) {
                        const int kt = (wi >> 1) * 4 + (s >> 1);
                        const int k0 = (int)ch * 128 + 16 * kt + 8 * (s & 1) + 2 * t;
                        w |= code(n, k0) << (2 * s);
                        w |= code(n, k0 + 1) << (16 + 2 * s);
                    }
                    codes[lane * 4 + wi] = w;
                }
            }
            for (int g = 0; g < 8; ++g)
                for (int j = 0; j < gpc; ++j)
                    for (int hi = 0; hi < 2; ++hi) {
                        const int n = (int)tile * 16 + g + 8 * hi;
                        const int grp = (int)ch * gpc + j;
                        const bool ok = n < N && grp < gk;
                        uint16_t* e = side + g * (4 * gpc) + 4 * j;
                        e[hi] = ok ? scales[(size_t)n * gk + grp] : 0;
                        e[2 + hi] = ok ? biases[(size_t)n * gk + grp] : 0;
                    }
        }
    return LBV_OK;
}

lbv_status lbv_pack_q4_0(const uint8_t* blocks, int K, int N, void* out, size_t out_bytes)
{
    g_err.clear();
    if (!blocks || !out)
        return fail(LBV_ERR_INVALID_ARG, "lbv_pack_q4_0: null pointer");
    const size_t need = lbv_packed_bytes(LBV_FMT_Q4_0, K, N, 32);
    if (need == 0)
        return fail(LBV_ERR_INVALID_ARG, "lbv_pack_q4_0: K=%d N=%d (need K%%32==0)", K, N);
    if (out_bytes < need)
        return fail(LBV_ERR_WORKSPACE, "lbv_pack_q4_0: out_bytes %zu < %zu", out_bytes, need);
    lbv::FmtInfo fi;
    lbv::fmt_info(LBV_FMT_Q4_0, 32, &fi);
    const lbv::Layout L = lbv::make_layout(fi, K, N);
    uint8_t* base = static_cast<uint8_t*>(out);
    const int nb = K / 32;
    auto nib = [&](int n, int k) -> uint32_t {
        if (n >= N || k >= K) return 0u;
        const uint8_t* blk = blocks + ((size_t)n * nb + k / 32) * 18;
        const int j = k % 32;
        return j < 16 ? (blk[2 + j] & 15u) : (uint32_t)(blk[2 + j - 16] >> 4);
    };
    for (int64_t tile = 0; tile < L.ntiles; ++tile)
        for (int64_t ch = 0; ch < L.nchunks; ++ch) {
            const size_t tc = (size_t)tile * L.nchunks + ch;
            uint32_t* codes = reinterpret_cast<uint32_t*>(base + tc * L.rec_bytes);
            uint16_t* side = reinterpret_cast<uint16_t*>(base + tc * L.rec_bytes + 512);
            for (int lane = 0; lane < 32; ++lane) {
                const int g = lane >> 2, t = lane & 3;
                for (int wi = 0; wi < 4; ++wi) {
                    const int n = (int)tile * 16 + g + 8 * (wi & 1);
                    uint32_t w = 0;
                    for (int s = 0; s < 4; ++s) {
                        const int kt = (wi >> 1) * 2 + (s >> 1);
                        const int k0 = (int)ch * 64 + 16 * kt + 8 * (s & 1) + 2 * t;
                        w |= nib(n, k0) << (4 * s);
                        w |= nib(n, k0 + 1) << (16 + 4 * s);
                    }
                    codes[lane * 4 + wi] = w;
                }
            }
            for (int g = 0; g < 8; ++g)
                for (int j = 0; j < 2; ++j)
                    for (int hi = 0; hi < 2; ++hi) {
                        const int n = (int)tile * 16 + g + 8 * hi;
                        const int b = (int)ch * 2 + j;
                        uint16_t d = 0;
                        if (n < N && b < nb) {
                            const uint8_t* blk = blocks + ((size_t)n * nb + b) * 18;
                            d = (uint16_t)(blk[0] | (blk[1] << 8));
                        }
                        side[g * 4 + 2 * j + hi] = d;
                    }
        }
    return LBV_OK;
}

// --------------------------------------------------------------------------
// Plans

lbv_status lbv_plan_create(lbv_format fmt, int K, int N, int group, lbv_dtype xdtype,
                           unsigned flags, lbv_plan** out)
{
    g_err.clear();
    if (!out)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_create: out is NULL");
    *out = nullptr;
    if (!valid_fmt(fmt))
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_create: unknown format %d", (int)fmt);
    if (xdtype != LBV_F16 && xdtype != LBV_BF16)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_create: unknown dtype %d", (int)xdtype);
    if (fmt == LBV_FMT_AFFINE2 && group != 32 && group != 64 && group != 128)
        return fail(LBV_ERR_UNSUPPORTED, "lbv_plan_create: affine group %d (supported: 32, 64, 128)", group);
    if (fmt != LBV_FMT_AFFINE2)
        group = fmt == LBV_FMT_SIGN1_G128 ? 128 : 32;
    if (K <= 0 || N <= 0 || K % k_quantum(fmt, group) != 0)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_create: K=%d N=%d not valid for the format", K, N);
    if ((flags & LBV_PLAN_FORCE_FEWROW) && (flags & LBV_PLAN_FORCE_GEMV))
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_create: both FORCE flags set");
    if ((flags & LBV_PLAN_TCGEN05) && (flags & LBV_PLAN_FORCE_GEMV))
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_create: TCGEN05 with FORCE_GEMV");
    if ((flags & LBV_PLAN_TC_E4M3) &&
        (flags & (LBV_PLAN_TCGEN05 | LBV_PLAN_FORCE_GEMV | LBV_PLAN_TEST_WAIT_LIMIT)))
        return fail(LBV_ERR_INVALID_ARG,
                    "lbv_plan_create: TC_E4M3 with TCGEN05, FORCE_GEMV or TEST_WAIT_LIMIT");
    if ((flags & LBV_PLAN_TEST_WAIT_LIMIT) &&
        (flags & (LBV_PLAN_TCGEN05 | LBV_PLAN_FORCE_GEMV | LBV_PLAN_MEASURE)))
        return fail(LBV_ERR_INVALID_ARG,
                    "lbv_plan_create: TEST_WAIT_LIMIT with TCGEN05, FORCE_GEMV or MEASURE");
    if (flags & ~(LBV_PLAN_MEASURE | LBV_PLAN_FORCE_FEWROW | LBV_PLAN_FORCE_GEMV | LBV_PLAN_PDL |
                  LBV_PLAN_TCGEN05 | LBV_PLAN_TEST_WAIT_LIMIT | LBV_PLAN_TC_E4M3))
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_create: unknown flags 0x%x", flags);

    lbv_plan* P = new (std::nothrow) lbv_plan();
    if (!P)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_create: out of host memory");
    P->fmt = fmt;
    P->xdtype = xdtype;
    P->K = K;
    P->N = N;
    P->group = group;
    P->flags = flags;
    lbv::fmt_info(fmt, group, &P->fi);
    P->layout = lbv::make_layout(P->fi, K, N);
    cudaError_t e = cudaGetDevice(&P->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&P->sms, cudaDevAttrMultiProcessorCount, P->device);
    if (e != cudaSuccess) {
        delete P;
        return cuda_fail(e, "lbv_plan_create: device query");
    }
    e = cudaMalloc((void**)&P->dev_err, 256);
    if (e == cudaSuccess)
        e = cudaMemset(P->dev_err, 0, 256);
    if (e != cudaSuccess) {
        cudaFree(P->dev_err);
        delete P;
        return cuda_fail(e, "lbv_plan_create: status word");
    }
    lbv::Shape sh = default_shape(P);
    if (!complete_shape(P, sh, 0)) {
        lbv_plan_destroy(P);
        return fail(LBV_ERR_UNSUPPORTED, "lbv_plan_create: no launch shape fits K=%d", K);
    }
    P->shape = sh;
    P->tc = (flags & LBV_PLAN_TCGEN05) ? 1 : 0;
    if (P->tc && !lbv::tc_plan_setup(P)) {
        lbv_plan_destroy(P);
        return fail(LBV_ERR_UNSUPPORTED, "lbv_plan_create: no tcgen05 launch shape fits K=%d", K);
    }
    P->t8 = (flags & LBV_PLAN_TC_E4M3) ? 1 : 0;
    if (P->t8 && !lbv::t8_plan_setup(P)) {
        lbv_plan_destroy(P);
        return fail(LBV_ERR_UNSUPPORTED,
                    "lbv_plan_create: the e4m3 tensor-memory kernel reads sign1 g128 and affine2 "
                    "g128 only, and needs a launch shape that fits K=%d", K);
    }
    for (int m = 0; m <= 8; ++m)
        P->use_gemv[m] = (flags & LBV_PLAN_FORCE_GEMV) ? 1 : 0;
    P->crossover = (flags & LBV_PLAN_FORCE_GEMV) ? 9 : 1;
    memset(P->measured_us, 0, sizeof P->measured_us);
    if (flags & LBV_PLAN_MEASURE) {
        extern lbv_status lbv_plan_measure_internal(lbv_plan * P);
        lbv_status st = lbv_plan_measure_internal(P);
        if (st != LBV_OK) {
            lbv_plan_destroy(P);
            return st;
        }
    }
    *out = P;
    return LBV_OK;
}

lbv_status lbv_plan_destroy(lbv_plan* plan)
{
    if (plan) {
        cudaFree(plan->dev_err);
        delete plan;
    }
    return LBV_OK;
}

size_t lbv_plan_packed_bytes(const lbv_plan* P)
{
    if (!P)
        return 0;
    return P->t8 ? lbv::t8_packed_bytes(P) : P->tc ? lbv::tc_packed_bytes(P) : P->layout.total;
}

lbv_status lbv_plan_pack(const lbv_plan* P, const void* part0, const void* part1,
                         const void* part2, void* out, size_t out_bytes)
{
    g_err.clear();
    if (!P || !part0 || !out)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_pack: null argument");
    if ((P->fmt == LBV_FMT_SIGN1_G128 && !part1) || (P->fmt == LBV_FMT_AFFINE2 && (!part1 || !part2)))
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_pack: missing scales or biases");
    const size_t need = lbv_plan_packed_bytes(P);
    if (out_bytes < need)
        return fail(LBV_ERR_WORKSPACE, "lbv_plan_pack: out_bytes %zu < %zu", out_bytes, need);
    if (P->t8) {
        lbv::t8_pack(P, part0, part1, part2, static_cast<uint8_t*>(out));
        return LBV_OK;
    }
    if (P->tc) {
        lbv::tc_pack(P, part0, part1, part2, static_cast<uint8_t*>(out));
        return LBV_OK;
    }
    switch (P->fmt) {
    case LBV_FMT_SIGN1_G128:
        return lbv_pack_sign_g128(static_cast<const uint32_t*>(part0),
                                  static_cast<const uint16_t*>(part1), P->K, P->N, out, out_bytes);
    case LBV_FMT_AFFINE2:
        return lbv_pack_affine2(static_cast<const uint32_t*>(part0),
                                static_cast<const uint16_t*>(part1),
                                static_cast<const uint16_t*>(part2), P->K, P->N, P->group, out,
                                out_bytes);
    case LBV_FMT_Q4_0:
        return lbv_pack_q4_0(static_cast<const uint8_t*>(part0), P->K, P->N, out, out_bytes);
    }
    return fail(LBV_ERR_INVALID_ARG, "lbv_plan_pack: unknown format");
}

lbv_status lbv_plan_device_status(const lbv_plan* P)
{
    g_err.clear();
    if (!P)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_device_status: plan is NULL");
    unsigned v = 0;
    cudaError_t e = cudaMemcpy(&v, P->dev_err, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "lbv_plan_device_status");
    if (v) {
        cudaMemset(P->dev_err, 0, sizeof v);
        if (v & 2u)
            return fail(LBV_ERR_BOUNDS, "a kernel of this plan found a copy or buffer range "
                                        "outside its bounds and skipped it");
        return fail(LBV_ERR_TIMEOUT, "a verify kernel gave up waiting for its weight copies");
    }
    return LBV_OK;
}

lbv_status lbv_plan_rows_histogram(const lbv_plan* P, uint64_t* counts)
{
    g_err.clear();
    if (!P || !counts)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_rows_histogram: NULL plan or counts");
    for (int m = 0; m < 8; ++m)
        counts[m] = P->rows_calls[m].load(std::memory_order_relaxed);
    return LBV_OK;
}

lbv_status lbv_plan_rows_reset(lbv_plan* P)
{
    g_err.clear();
    if (!P)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_rows_reset: plan is NULL");
    for (int m = 0; m < 8; ++m)
        P->rows_calls[m].store(0, std::memory_order_relaxed);
    return LBV_OK;
}

lbv_status lbv_plan_query(const lbv_plan* P, int M, int* kernel_id, int* splits,
                          size_t* workspace_bytes)
{
    g_err.clear();
    if (!P)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_query: plan is NULL");
    if (M < 1 || M > 8)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_query: M=%d outside 1..8", M);
    if (kernel_id)
        *kernel_id = P->t8 ? LBV_KERNEL_FEWROW_TC8
                     : P->tc ? LBV_KERNEL_FEWROW_TC
                     : P->use_gemv[M] ? LBV_KERNEL_GEMV : LBV_KERNEL_FEWROW;
    if (splits)
        *splits = P->t8 ? P->t8_shape.splits
                  : P->tc ? P->tc_shape.splits : P->use_gemv[M] ? 1 : P->shape.splits;
    if (workspace_bytes)
        *workspace_bytes = 0;
    return LBV_OK;
}

lbv_status lbv_plan_shape(const lbv_plan* P, int* warps, int* tpw, int* splits, int* ctas_n)
{
    g_err.clear();
    if (!P)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_shape: plan is NULL");
    if (P->t8) {
        if (warps) *warps = 0;
        if (tpw) *tpw = 0;
        if (splits) *splits = P->t8_shape.splits;
        if (ctas_n) *ctas_n = P->t8_shape.ctas_n;
        return LBV_OK;
    }
    if (P->tc) {
        if (warps) *warps = 0;
        if (tpw) *tpw = 0;
        if (splits) *splits = P->tc_shape.splits;
        if (ctas_n) *ctas_n = P->tc_shape.ctas_n;
        return LBV_OK;
    }
    if (warps) *warps = P->shape.warps;
    if (tpw) *tpw = P->shape.tpw;
    if (splits) *splits = P->shape.splits;
    if (ctas_n) *ctas_n = P->shape.ctas_n;
    return LBV_OK;
}

lbv_status lbv_plan_set_shape(lbv_plan* P, int warps, int tpw, int splits, int ctas_n)
{
    g_err.clear();
    if (!P)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_set_shape: plan is NULL");
    if (P->t8) {
        if ((splits != 1 && splits != 2 && splits != 4 && splits != 8) || ctas_n < 0)
            return fail(LBV_ERR_INVALID_ARG, "lbv_plan_set_shape: splits=%d ctas_n=%d", splits, ctas_n);
        if (!lbv::t8_set_shape(P, splits, ctas_n) || P->t8_shape.splits != splits)
            return fail(LBV_ERR_UNSUPPORTED, "lbv_plan_set_shape: shape does not fit (smem, occupancy or K)");
        return LBV_OK;
    }
    if (P->tc) {
        if (splits < 1 || splits > 8 || ctas_n < 0)
            return fail(LBV_ERR_INVALID_ARG, "lbv_plan_set_shape: splits=%d ctas_n=%d", splits, ctas_n);
        if (!lbv::tc_set_shape(P, splits, ctas_n))
            return fail(LBV_ERR_UNSUPPORTED, "lbv_plan_set_shape: shape does not fit (smem or occupancy)");
        return LBV_OK;
    }
    const bool shape_ok = (warps == 8 && (tpw == 2 || tpw == 4)) ||
                          (warps == 16 && (tpw == 1 || tpw == 2));
    if (!shape_ok || splits < 1 || splits > 8 ||
        ctas_n < 0)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_set_shape: warps=%d tpw=%d splits=%d ctas_n=%d",
                    warps, tpw, splits, ctas_n);
    lbv::Shape sh = {warps, tpw, splits, 0, 0};
    if (!complete_shape(P, sh, ctas_n))
        return fail(LBV_ERR_UNSUPPORTED, "lbv_plan_set_shape: shape does not fit (smem or occupancy)");
    P->shape = sh;
    return LBV_OK;
}

// --------------------------------------------------------------------------
// Verify

static lbv_status check_verify_args(const char* fn, const lbv_plan* P, const void* X, int M,
                                    int ldx, const void* Wp, const float* Y, int ldy,
                                    const void* workspace, size_t workspace_bytes)
{
    if (!P)
        return fail(LBV_ERR_INVALID_ARG, "%s: plan is NULL", fn);
    if (M < 1 || M > 8)
        return fail(LBV_ERR_INVALID_ARG, "%s: M=%d outside 1..8", fn, M);
    if (!X || !Wp || !Y)
        return fail(LBV_ERR_INVALID_ARG, "%s: null X, Wp or Y", fn);
    if (ldx < P->K || ldy < P->N)
        return fail(LBV_ERR_INVALID_ARG, "%s: ldx=%d < K=%d or ldy=%d < N=%d", fn, ldx,
                    P->K, ldy, P->N);
    if ((reinterpret_cast<uintptr_t>(Wp) & 15u) != 0)
        return fail(LBV_ERR_INVALID_ARG, "%s: Wp not 16-byte aligned", fn);
    if ((reinterpret_cast<uintptr_t>(X) & 1u) != 0 || (reinterpret_cast<uintptr_t>(Y) & 3u) != 0)
        return fail(LBV_ERR_INVALID_ARG, "%s: X or Y misaligned for its element type", fn);
    if (workspace_bytes != 0 && !workspace)
        return fail(LBV_ERR_INVALID_ARG, "%s: workspace_bytes without workspace", fn);
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != P->device)
        return fail(LBV_ERR_INVALID_ARG, "%s: current device %d is not the plan's %d", fn,
                    dev, P->device);
    return LBV_OK;
}

static lbv::VerifyParams make_params(const lbv_plan* P, const void* X, int M, int ldx,
                                     const void* Wp, float* Y, int ldy)
{
    lbv::VerifyParams p;
    p.X = X;
    p.W = static_cast<const uint8_t*>(Wp);
    p.Y = Y;
    p.ldx = ldx;
    p.ldy = ldy;
    p.M = M;
    p.K = P->K;
    p.N = P->N;
    p.ntiles = (int)P->layout.ntiles;
    p.nchunks = (int)P->layout.nchunks;
    p.splits = P->shape.splits;
    p.cps = shape_cps(P->shape, P->layout.nchunks, slice_step(P));
    p.x_vec = ((reinterpret_cast<uintptr_t>(X) & 15u) == 0 && (ldx % 8) == 0) ? 1 : 0;
    p.err = P->dev_err;
    p.zero = 0;
    const bool wait_test = (P->flags & LBV_PLAN_TEST_WAIT_LIMIT) != 0;
    p.wait_limit = wait_test ? 256 : 0;
    p.skip_q = wait_test ? 1 : -1;
    p.rot = 0;
    p.store_y = 1;
    p.signs = nullptr;
    p.amax_keys = nullptr;
    p.amax_done = nullptr;
    p.amax_idx = nullptr;
    p.amax_val = nullptr;
    return p;
}

// Internal: launch a given path (used by the plan measurement as well).
lbv_status lbv_verify_launch_internal(const lbv_plan* P, const void* X, int M, int ldx,
                                      const void* Wp, float* Y, int ldy, bool gemv,
                                      cudaStream_t st)
{
    cudaError_t e;
    if (P->t8) {
        const lbv::T8Fused f = {0, 1, nullptr, nullptr, nullptr, nullptr, nullptr};
        e = lbv::t8_verify_launch(P, X, M, ldx, Wp, Y, ldy, f, (P->flags & LBV_PLAN_PDL) != 0, st);
        if (e != cudaSuccess)
            return cuda_fail(e, "lbv_verify_gemm: launch");
        return LBV_OK;
    }
    if (P->tc) {
        e = lbv::tc_verify_launch(P, X, M, ldx, Wp, Y, ldy, (P->flags & LBV_PLAN_PDL) != 0, st);
        if (e != cudaSuccess)
            return cuda_fail(e, "lbv_verify_gemm: launch");
        return LBV_OK;
    }
    const lbv::VerifyParams p = make_params(P, X, M, ldx, Wp, Y, ldy);
    if (gemv) {
        e = cudaSuccess;
        for (int r = 0; r < M && e == cudaSuccess; ++r)
            e = lbv::launch_gemv(P->fmt, P->xdtype, P->group, p, r, st);
    } else {
        lbv::LaunchOpts o;
        o.pdl = (P->flags & LBV_PLAN_PDL) != 0;
        e = ops_for(P->fmt, P->group)->launch(P->xdtype, P->shape, p, o, st);
    }
    if (e != cudaSuccess)
        return cuda_fail(e, "lbv_verify_gemm: launch");
    return LBV_OK;
}

lbv_status lbv_verify_gemm(const lbv_plan* P, const void* X, int M, int ldx, const void* Wp,
                           float* Y, int ldy, void* workspace, size_t workspace_bytes,
                           lbv_stream stream)
{
    g_err.clear();
    lbv_status st = check_verify_args("lbv_verify_gemm", P, X, M, ldx, Wp, Y, ldy, workspace,
                                      workspace_bytes);
    if (st != LBV_OK)
        return st;
    st = lbv_verify_launch_internal(P, X, M, ldx, Wp, Y, ldy, P->use_gemv[M] != 0,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (st == LBV_OK)
        count_rows(P->rows_calls, M);
    return st;
}

// --------------------------------------------------------------------------
// Fused head

// Argmax keys (8 x 8 bytes) and the count of finished CTAs, padded.
static constexpr size_t kFusedWorkspace = 128;

size_t lbv_fused_workspace_bytes(void)
{
    return kFusedWorkspace;
}

lbv_status lbv_verify_fused(const lbv_plan* P, const void* X, int M, int ldx, const void* Wp,
                            unsigned ops, const uint32_t* signs, float* Y, int ldy,
                            int32_t* argmax_idx, float* argmax_val, void* workspace,
                            size_t workspace_bytes, lbv_stream stream)
{
    g_err.clear();
    if (!P)
        return fail(LBV_ERR_INVALID_ARG, "lbv_verify_fused: plan is NULL");
    if (ops & ~(LBV_FUSED_ROTATE | LBV_FUSED_ARGMAX))
        return fail(LBV_ERR_INVALID_ARG, "lbv_verify_fused: unknown ops bits 0x%x", ops);
    const bool argmax = (ops & LBV_FUSED_ARGMAX) != 0, rotate = (ops & LBV_FUSED_ROTATE) != 0;
    if (!Y && !argmax)
        return fail(LBV_ERR_INVALID_ARG, "lbv_verify_fused: no output (Y NULL without argmax)");
    // the checks of lbv_verify_gemm, with Y optional
    float dummy_y[1];
    lbv_status st = check_verify_args("lbv_verify_fused", P, X, M, ldx, Wp, Y ? Y : dummy_y,
                                      Y ? ldy : P->N, nullptr, 0);
    if (st != LBV_OK)
        return st;
    if (P->tc)
        return fail(LBV_ERR_UNSUPPORTED, "lbv_verify_fused: not available on LBV_PLAN_TCGEN05 plans");
    if (rotate) {
        if (P->K % 128 != 0)
            return fail(LBV_ERR_UNSUPPORTED, "lbv_verify_fused: rotation needs K %% 128 == 0 (K=%d)",
                        P->K);
        const int cps = shape_cps(P->shape, P->layout.nchunks, slice_step(P));
        if (!P->t8 && P->shape.splits > 1 && (cps * P->fi.chunk_k) % 128 != 0)
            return fail(LBV_ERR_UNSUPPORTED,
                        "lbv_verify_fused: the plan's K slices (%d elements) are not whole "
                        "128-element blocks", cps * P->fi.chunk_k);
        if (reinterpret_cast<uintptr_t>(signs) & 3u)
            return fail(LBV_ERR_INVALID_ARG, "lbv_verify_fused: signs not 4-byte aligned");
    }
    if (argmax) {
        if (!argmax_idx)
            return fail(LBV_ERR_INVALID_ARG, "lbv_verify_fused: argmax without argmax_idx");
        if ((reinterpret_cast<uintptr_t>(argmax_idx) & 3u) ||
            (reinterpret_cast<uintptr_t>(argmax_val) & 3u))
            return fail(LBV_ERR_INVALID_ARG, "lbv_verify_fused: argmax outputs misaligned");
        if (!workspace || workspace_bytes < kFusedWorkspace ||
            (reinterpret_cast<uintptr_t>(workspace) & 15u))
            return fail(LBV_ERR_WORKSPACE,
                        "lbv_verify_fused: argmax needs a 16-byte aligned, zero-initialised "
                        "workspace of %zu bytes", kFusedWorkspace);
    }
    if (P->t8) {
        lbv::T8Fused f = {rotate ? 1 : 0, Y ? 1 : 0, rotate ? signs : nullptr, nullptr, nullptr,
                          nullptr, nullptr};
        if (argmax) {
            f.amax_keys = static_cast<unsigned long long*>(workspace);
            f.amax_done = reinterpret_cast<unsigned*>(static_cast<unsigned char*>(workspace) + 64);
            f.amax_idx = argmax_idx;
            f.amax_val = argmax_val;
        }
        const cudaError_t e = lbv::t8_verify_launch(P, X, M, ldx, Wp, Y, Y ? ldy : P->N, f,
                                                    (P->flags & LBV_PLAN_PDL) != 0,
                                                    reinterpret_cast<cudaStream_t>(stream));
        if (e != cudaSuccess)
            return cuda_fail(e, "lbv_verify_fused: launch");
        count_rows(P->rows_calls, M);
        return LBV_OK;
    }
    lbv::VerifyParams p = make_params(P, X, M, ldx, Wp, Y, Y ? ldy : P->N);
    p.rot = rotate ? 1 : 0;
    p.signs = rotate ? signs : nullptr;
    p.store_y = Y ? 1 : 0;
    if (argmax) {
        p.amax_keys = static_cast<unsigned long long*>(workspace);
        p.amax_done = reinterpret_cast<unsigned*>(static_cast<unsigned char*>(workspace) + 64);
        p.amax_idx = argmax_idx;
        p.amax_val = argmax_val;
    }
    lbv::LaunchOpts o;
    o.pdl = (P->flags & LBV_PLAN_PDL) != 0;
    const cudaError_t e = ops_for(P->fmt, P->group)
                              ->launch(P->xdtype, P->shape, p, o,
                                       reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "lbv_verify_fused: launch");
    count_rows(P->rows_calls, M);
    return LBV_OK;
}

lbv_status lbv_verify_fused_noalloc(const lbv_plan* P, const void* X, int M, int ldx,
                                    const void* Wp, unsigned ops, const uint32_t* signs, float* Y,
                                    int ldy, int32_t* argmax_idx, float* argmax_val,
                                    lbv_stream stream)
{
    g_err.clear();
    if (!P)
        return fail(LBV_ERR_INVALID_ARG, "lbv_verify_fused_noalloc: plan is NULL");
    if (M < 1 || M > 8)
        return fail(LBV_ERR_INVALID_ARG,
                    "lbv_verify_fused_noalloc: M=%d outside 1..8 (the scratch holds 8 rows)", M);
    void* scratch = nullptr;
    if (ops & LBV_FUSED_ARGMAX) {
        if (lbv::noalloc_scratch_bytes() < kFusedWorkspace)
            return fail(LBV_ERR_WORKSPACE, "lbv_verify_fused_noalloc: scratch too small");
        bool needs_clear = false;
        cudaError_t e = lbv::noalloc_scratch(&scratch, &needs_clear);
        if (e != cudaSuccess)
            return cuda_fail(e, "lbv_verify_fused_noalloc: scratch address");
        if (needs_clear) {      // zero at load already; cleared once more on first use
            e = cudaMemsetAsync(scratch, 0, lbv::noalloc_scratch_bytes(),
                                reinterpret_cast<cudaStream_t>(stream));
            if (e != cudaSuccess)
                return cuda_fail(e, "lbv_verify_fused_noalloc: clearing the scratch");
            lbv::noalloc_scratch_cleared();
        }
    }
    return lbv_verify_fused(P, X, M, ldx, Wp, ops, signs, Y, ldy, argmax_idx, argmax_val,
                            scratch, scratch ? kFusedWorkspace : 0, stream);
}

lbv_status lbv_fused_rotation(const void* X, void* Xr, int M, int K, lbv_dtype dtype,
                              const uint32_t* signs, lbv_stream stream)
{
    g_err.clear();
    if (!X || !Xr)
        return fail(LBV_ERR_INVALID_ARG, "lbv_fused_rotation: null X or Xr");
    if (M < 1 || M > 8)
        return fail(LBV_ERR_INVALID_ARG, "lbv_fused_rotation: M=%d outside 1..8", M);
    if (K <= 0 || K % 128 != 0)
        return fail(LBV_ERR_INVALID_ARG, "lbv_fused_rotation: K=%d not a positive multiple of 128",
                    K);
    if (dtype != LBV_F16 && dtype != LBV_BF16)
        return fail(LBV_ERR_INVALID_ARG, "lbv_fused_rotation: unknown dtype %d", (int)dtype);
    if ((reinterpret_cast<uintptr_t>(X) & 1u) || (reinterpret_cast<uintptr_t>(Xr) & 1u) ||
        (reinterpret_cast<uintptr_t>(signs) & 3u))
        return fail(LBV_ERR_INVALID_ARG, "lbv_fused_rotation: misaligned pointer");
    cudaError_t e = lbv::launch_fused_rotation(X, Xr, M, K, dtype, signs,
                                               reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "lbv_fused_rotation: launch");
    return LBV_OK;
}

lbv_status lbv_fwht128(const void* X, void* Xr, int M, int K, lbv_dtype dtype,
                       const uint32_t* signs, lbv_stream stream)
{
    g_err.clear();
    if (!X || !Xr)
        return fail(LBV_ERR_INVALID_ARG, "lbv_fwht128: null X or Xr");
    if (M < 1 || M > 8)
        return fail(LBV_ERR_INVALID_ARG, "lbv_fwht128: M=%d outside 1..8", M);
    if (K <= 0 || K % 128 != 0)
        return fail(LBV_ERR_INVALID_ARG, "lbv_fwht128: K=%d not a positive multiple of 128", K);
    if (dtype != LBV_F16 && dtype != LBV_BF16)
        return fail(LBV_ERR_INVALID_ARG, "lbv_fwht128: unknown dtype %d", (int)dtype);
    if ((reinterpret_cast<uintptr_t>(X) & 1u) || (reinterpret_cast<uintptr_t>(Xr) & 1u) ||
        (reinterpret_cast<uintptr_t>(signs) & 3u))
        return fail(LBV_ERR_INVALID_ARG, "lbv_fwht128: misaligned pointer");
    cudaError_t e = lbv::launch_fwht128(X, Xr, M, K, dtype, signs,
                                        reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "lbv_fwht128: launch");
    return LBV_OK;
}

lbv_status lbv_dequant_fp16(const lbv_plan* P, const void* Wp, uint16_t* W, lbv_stream stream)
{
    g_err.clear();
    if (!P || !Wp || !W)
        return fail(LBV_ERR_INVALID_ARG, "lbv_dequant_fp16: null argument");
    if ((reinterpret_cast<uintptr_t>(Wp) & 15u) != 0 || (reinterpret_cast<uintptr_t>(W) & 1u))
        return fail(LBV_ERR_INVALID_ARG, "lbv_dequant_fp16: misaligned pointer");
    cudaError_t e =
        P->t8 ? lbv::t8_dequant(P, Wp, W, reinterpret_cast<cudaStream_t>(stream))
        : P->tc ? lbv::tc_dequant(P, Wp, W, reinterpret_cast<cudaStream_t>(stream))
              : lbv::launch_dequant(P->fmt, P->group, static_cast<const uint8_t*>(Wp), P->K, P->N,
                                    (int)P->layout.ntiles, (int)P->layout.nchunks, W,
                                    reinterpret_cast<cudaStream_t>(stream));
    if (e != cudaSuccess)
        return cuda_fail(e, "lbv_dequant_fp16: launch");
    return LBV_OK;
}

}  // extern "C"

// --------------------------------------------------------------------------
// Plan-time measurement (LBV_PLAN_MEASURE): time every launch shape that fits
// and the 1-row path on scratch buffers with a cold L2, keep the fastest
// shape, and pick per row count the faster of the few-row kernel and the
// 1-row path run M times (Ishizuki releases v0.6.1: the verify kernel starts
// at the row count where it is faster, per matrix).

namespace {

struct Scratch {
    void* w = nullptr;
    void* x = nullptr;
    float* y = nullptr;
    void* flush = nullptr;
    size_t flush_bytes = 0;
    ~Scratch()
    {
        cudaFree(w);
        cudaFree(x);
        cudaFree(y);
        cudaFree(flush);
    }
};

// Median time (us) of `reps` single launches, each after an L2 flush.
template <class F>
lbv_status time_cold(F&& launch, Scratch& s, cudaStream_t st, int reps, float* us)
{
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    std::vector<float> v;
    lbv_status rc = LBV_OK;
    for (int i = 0; i < reps + 2 && rc == LBV_OK; ++i) {
        cudaMemsetAsync(s.flush, i & 0xFF, s.flush_bytes, st);
        cudaEventRecord(a, st);
        rc = launch();
        cudaEventRecord(b, st);
        if (cudaEventSynchronize(b) != cudaSuccess) {
            rc = fail(LBV_ERR_CUDA, "plan measure: %s", cudaGetErrorString(cudaGetLastError()));
            break;
        }
        float ms = 0.f;
        cudaEventElapsedTime(&ms, a, b);
        if (i >= 2)
            v.push_back(ms * 1000.f);
    }
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (rc != LBV_OK)
        return rc;
    std::sort(v.begin(), v.end());
    *us = v[v.size() / 2];
    return LBV_OK;
}

// Median time (us) per launch of `reps` chains, each after an L2 flush: every
// chain runs launch(c, stream) for c = 0 .. n-1 twice, back to back, captured
// once in a CUDA graph (the steady state of a caller that verifies through
// many matrices; launched one by one from the host, ~10 us kernels would be
// timed at the host's launch rate).  Without graph capture: direct launches.
template <class F>
lbv_status time_chain(F&& launch, int n, Scratch& s, int reps, float* us)
{
    cudaStream_t st = nullptr;
    if (cudaStreamCreateWithFlags(&st, cudaStreamNonBlocking) != cudaSuccess)
        return fail(LBV_ERR_CUDA, "plan measure: stream");
    cudaGraph_t graph = nullptr;
    cudaGraphExec_t exec = nullptr;
    lbv_status rc = LBV_OK;
    if (cudaStreamBeginCapture(st, cudaStreamCaptureModeThreadLocal) == cudaSuccess) {
        for (int k = 0; k < 2 * n && rc == LBV_OK; ++k)
            rc = launch(k % n, st);
        const cudaError_t ec = cudaStreamEndCapture(st, &graph);
        if (rc == LBV_OK && ec == cudaSuccess &&
            cudaGraphInstantiate(&exec, graph, 0) != cudaSuccess)
            exec = nullptr;
    }
    cudaGetLastError();                           // a failed capture leaves no error behind
    cudaEvent_t a, b;
    cudaEventCreate(&a);
    cudaEventCreate(&b);
    std::vector<float> v;
    rc = LBV_OK;
    for (int i = 0; i < reps + 1 && rc == LBV_OK; ++i) {
        cudaMemsetAsync(s.flush, i & 0xFF, s.flush_bytes, st);
        cudaEventRecord(a, st);
        if (exec) {
            if (cudaGraphLaunch(exec, st) != cudaSuccess)
                rc = fail(LBV_ERR_CUDA, "plan measure: graph launch");
        } else {
            for (int k = 0; k < 2 * n && rc == LBV_OK; ++k)
                rc = launch(k % n, st);
        }
        cudaEventRecord(b, st);
        if (cudaEventSynchronize(b) != cudaSuccess) {
            rc = fail(LBV_ERR_CUDA, "plan measure: %s", cudaGetErrorString(cudaGetLastError()));
            break;
        }
        float ms = 0.f;
        cudaEventElapsedTime(&ms, a, b);
        if (i >= 1)
            v.push_back(ms * 1000.f / (2 * n));
    }
    cudaEventDestroy(a);
    cudaEventDestroy(b);
    if (exec)
        cudaGraphExecDestroy(exec);
    if (graph)
        cudaGraphDestroy(graph);
    cudaStreamDestroy(st);
    if (rc != LBV_OK)
        return rc;
    std::sort(v.begin(), v.end());
    *us = v[v.size() / 2];
    return LBV_OK;
}

}  // namespace

lbv_status lbv_verify_launch_internal(const lbv_plan* P, const void* X, int M, int ldx,
                                      const void* Wp, float* Y, int ldy, bool gemv,
                                      cudaStream_t st);

lbv_status lbv_plan_measure_internal(lbv_plan* P)
{
    Scratch s;
    int l2 = 0;
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, P->device);
    s.flush_bytes = (size_t)std::max(l2, 1 << 20) * 2;
    cudaError_t e = cudaMalloc(&s.w, lbv_plan_packed_bytes(P));
    if (e == cudaSuccess) e = cudaMalloc(&s.x, (size_t)8 * P->K * 2);
    if (e == cudaSuccess) e = cudaMalloc((void**)&s.y, (size_t)8 * P->N * 4);
    if (e == cudaSuccess) e = cudaMalloc(&s.flush, s.flush_bytes);
    if (e == cudaSuccess) e = cudaMemset(s.w, 0x5A, lbv_plan_packed_bytes(P));
    if (e == cudaSuccess) e = cudaMemset(s.x, 0x11, (size_t)8 * P->K * 2);
    if (e != cudaSuccess)
        return cuda_fail(e, "plan measure: scratch");
    cudaStream_t st = nullptr;
    const int reps = 7;

    if (P->t8) {
        // e4m3 tensor-memory plans: every K split that fits; the kernel serves every M
        lbv::T8Shape best = P->t8_shape;
        float best_us = 1e30f;
        for (int sp = 1; sp <= 8; sp <<= 1) {
            if (!lbv::t8_set_shape(P, sp, 0) || P->t8_shape.splits != sp)
                continue;
            float us = 0.f;
            lbv_status rc = time_cold(
                [&] { return lbv_verify_launch_internal(P, s.x, 8, P->K, s.w, s.y, P->N, false, st); },
                s, st, reps, &us);
            if (rc != LBV_OK)
                return rc;
            if (us < best_us) {
                best_us = us;
                best = P->t8_shape;
            }
        }
        P->t8_shape = best;
        for (int m = 1; m <= 8; ++m) {
            float few = 0.f;
            lbv_status rc = time_cold(
                [&] { return lbv_verify_launch_internal(P, s.x, m, P->K, s.w, s.y, P->N, false, st); },
                s, st, reps, &few);
            if (rc != LBV_OK)
                return rc;
            P->measured_us[m][0] = few;
        }
        return LBV_OK;
    }
    if (P->tc) {
        // tcgen05 plans: every K split that fits; the kernel serves every M
        lbv::TcShape best = P->tc_shape;
        float best_us = 1e30f;
        for (int sp = 1; sp <= 8; ++sp) {
            if (!lbv::tc_set_shape(P, sp, 0) || P->tc_shape.splits != sp)
                continue;
            float us = 0.f;
            lbv_status rc = time_cold(
                [&] { return lbv_verify_launch_internal(P, s.x, 8, P->K, s.w, s.y, P->N, false, st); },
                s, st, reps, &us);
            if (rc != LBV_OK)
                return rc;
            if (us < best_us) {
                best_us = us;
                best = P->tc_shape;
            }
        }
        lbv::tc_set_shape(P, best.splits, best.ctas_n);
        for (int m = 1; m <= 8; ++m) {
            float few = 0.f;
            lbv_status rc = time_cold(
                [&] { return lbv_verify_launch_internal(P, s.x, m, P->K, s.w, s.y, P->N, false, st); },
                s, st, reps, &few);
            if (rc != LBV_OK)
                return rc;
            P->measured_us[m][0] = few;
        }
        return LBV_OK;
    }

    // 1) few-row launch shape, timed as back-to-back launches over distinct
    //    copies of the weights (at least twice the L2 in all, at most 16)
    const size_t wbytes = lbv_plan_packed_bytes(P);
    const int ncopy = (int)std::max<size_t>(1, std::min<size_t>(16, (2 * (size_t)l2 + wbytes - 1) / wbytes));
    void* copies = nullptr;
    e = cudaMalloc(&copies, wbytes * (size_t)ncopy);
    if (e == cudaSuccess)
        e = cudaMemset(copies, 0x5A, wbytes * (size_t)ncopy);
    if (e != cudaSuccess) {
        cudaFree(copies);
        return cuda_fail(e, "plan measure: weight copies");
    }
    lbv::Shape best = P->shape;
    float best_us = 1e30f;
    const int shapes_c[][2] = {{8, 2}, {8, 4}, {16, 1}, {16, 2}};
    for (const auto& wt : shapes_c)
            for (int sp = 1; sp <= 8; ++sp) {
                lbv::Shape sh = {wt[0], wt[1], sp, 0, 0};
                if (!complete_shape(P, sh, 0) || sh.splits != sp)
                    continue;
                P->shape = sh;
                float us = 0.f;
                lbv_status rc = time_chain(
                    [&](int c, cudaStream_t cs) {
                        return lbv_verify_launch_internal(
                            P, s.x, 8, P->K, static_cast<unsigned char*>(copies) + (size_t)c * wbytes,
                            s.y, P->N, false, cs);
                    },
                    ncopy, s, 5, &us);
                if (rc != LBV_OK) {
                    cudaFree(copies);
                    return rc;
                }
                if (us < best_us) {
                    best_us = us;
                    best = sh;
                }
            }
    cudaFree(copies);
    P->shape = best;
    complete_shape(P, P->shape, 0);

    // 2) per row count: few-row vs the 1-row path run M times
    float gemv1 = 0.f;
    lbv_status rc = time_cold(
        [&] { return lbv_verify_launch_internal(P, s.x, 1, P->K, s.w, s.y, P->N, true, st); }, s,
        st, reps, &gemv1);
    if (rc != LBV_OK)
        return rc;
    P->crossover = 9;
    for (int m = 1; m <= 8; ++m) {
        float few = 0.f;
        rc = time_cold(
            [&] { return lbv_verify_launch_internal(P, s.x, m, P->K, s.w, s.y, P->N, false, st); },
            s, st, reps, &few);
        if (rc != LBV_OK)
            return rc;
        P->measured_us[m][0] = few;
        P->measured_us[m][1] = gemv1 * m;
        const bool g = !(P->flags & LBV_PLAN_FORCE_FEWROW) &&
                       ((P->flags & LBV_PLAN_FORCE_GEMV) || gemv1 * m < few);
        P->use_gemv[m] = g ? 1 : 0;
        if (!g && P->crossover == 9)
            P->crossover = m;
    }
    return LBV_OK;
}

extern "C" lbv_status lbv_plan_measured(const lbv_plan* P, int M, float* fewrow_us,
                                        float* gemv_us, int* crossover)
{
    g_err.clear();
    if (!P || M < 1 || M > 8)
        return fail(LBV_ERR_INVALID_ARG, "lbv_plan_measured: bad plan or M");
    if (fewrow_us) *fewrow_us = P->measured_us[M][0];
    if (gemv_us) *gemv_us = P->measured_us[M][1];
    if (crossover) *crossover = P->crossover;
    return LBV_OK;
}

// --------------------------------------------------------------------------
// Grouped verify: independent problems of one format, one launch per class

namespace {

// Chunks per K slice of a problem under a split: whole 128-element blocks
// where K allows it (as for plans); 0 if the problem would not have exactly
// `splits` slices.
int group_problem_cps(const lbv_group* G, int i, int splits)
{
    const int step = (G->K[i] % 128 == 0 && G->fi.chunk_k < 128) ? 128 / G->fi.chunk_k : 1;
    lbv::Shape sh = {16, 2, splits, 0, 0};
    const int cps = shape_cps(sh, G->nchunks[i], step);
    return (G->nchunks[i] + cps - 1) / cps == splits ? cps : 0;
}

// Cluster rows of each problem of class c, R in all where the bounds allow:
// in proportion to its packed bytes by largest remainders, at least 1 and at
// most its tiles; problems of other classes, and those with M[i] == 0 when M
// is given, get none.  Returns the total.
int divide_rows(const lbv_group* G, int c, int R, const int* M, int* rows)
{
    double B = 0.0;
    int n = 0;
    for (int i = 0; i < G->count; ++i)
        if (G->cls[i] == c && (!M || M[i] > 0)) {
            B += G->bytes[i];
            ++n;
        }
    double quota[lbv::kMaxGroup];
    int total = 0;
    for (int i = 0; i < G->count; ++i) {
        rows[i] = 0;
        if (G->cls[i] != c || (M && M[i] == 0))
            continue;
        quota[i] = (double)R * G->bytes[i] / B;
        rows[i] = std::max(1, std::min((int)quota[i], G->ntiles[i]));
        total += rows[i];
    }
    // one row at a time to the largest remainder (or away from the most
    // over-served) until the total is R or no problem can take or give one
    for (int step = 0; step < 4 * lbv::kMaxGroup && total != R && n > 0; ++step) {
        int pick = -1;
        double best = 0.0;
        for (int i = 0; i < G->count; ++i) {
            if (rows[i] == 0)
                continue;
            const double rem = quota[i] - rows[i];
            if (total < R && rows[i] < G->ntiles[i] && (pick < 0 || rem > best)) {
                pick = i;
                best = rem;
            }
            if (total > R && rows[i] > 1 && (pick < 0 || rem < best)) {
                pick = i;
                best = rem;
            }
        }
        if (pick < 0)
            break;
        const int d = total < R ? 1 : -1;
        rows[pick] += d;
        total += d;
    }
    return total;
}

// Records the rows of class c with every problem active (a call never gives
// an active problem fewer, so no row gets more tiles than the partials hold).
void group_commit_rows(lbv_group* G, int c)
{
    int rows[lbv::kMaxGroup];
    divide_rows(G, c, G->launch[c].rows_target, nullptr, rows);
    for (int i = 0; i < G->count; ++i)
        if (G->cls[i] == c)
            G->rows_plan[i] = rows[i];
}

int group_tiles_max(const lbv_group* G, const int* rows)
{
    int t = 1;
    for (int i = 0; i < G->count; ++i)
        if (rows[i] > 0)
            t = std::max(t, (G->ntiles[i] + rows[i] - 1) / rows[i]);
    return t;
}

// Launch shape of class c for (tpw, splits) with about R cluster rows; false
// if the split does not suit every problem of the class, or shared memory or
// occupancy rule it out.
bool group_fit(lbv_group* G, int c, int tpw, int splits, int R, lbv::GroupLaunch* out)
{
    const lbv::VerifyOps* ops = ops_for(G->fmt, G->group);
    for (int i = 0; i < G->count; ++i)
        if (G->cls[i] == c && group_problem_cps(G, i, splits) == 0)
            return false;
    std::vector<int> rows(G->count);
    lbv::GroupLaunch L;
    L.shape = {16, tpw, splits, 0, 0};
    L.shape.ctas_n = divide_rows(G, c, R, nullptr, rows.data());
    L.tiles_max = group_tiles_max(G, rows.data());
    // a CTA lays out its own problem's X slice and partials: the launch
    // needs the largest of the problems' needs, not the largest slice next
    // to the largest partials
    size_t need = 0;
    for (int i = 0; i < G->count; ++i)
        if (rows[i] > 0)
            need = std::max(need, ops->smem(16, tpw, group_problem_cps(G, i, splits),
                                            (G->ntiles[i] + rows[i] - 1) / rows[i], splits));
    L.shape.smem = std::max(need, kSmemOnePerSm);
    if (L.shape.smem > kSmemCap)
        return false;
    L.resident = ops->max_clusters_grouped(G->xdtype, L.shape);
    if (L.resident < 1)
        return false;
    L.rows_target = R;
    *out = L;
    return true;
}

// Clusters of (tpw, splits) resident at once for class c: from a shape that
// fits (one wave's rows if the partials allow, else one row per tile, the
// smallest partials); the SM count over the split if none fits.
int group_resident(lbv_group* G, int c, int tpw, int splits, int tiles)
{
    lbv::GroupLaunch probe;
    const int guess = std::max(1, G->sms / splits);
    if (group_fit(G, c, tpw, splits, std::min(guess, tiles), &probe) ||
        group_fit(G, c, tpw, splits, tiles, &probe))
        return probe.resident;
    return guess;
}

// Whole waves of resident clusters, the fewest from `waves0` up whose shape
// fits class c for (tpw, splits) (a partial last wave would leave SMs idle
// for a whole row's time).
bool group_fit_rows(lbv_group* G, int c, int tpw, int splits, int waves0, lbv::GroupLaunch* out)
{
    int tiles = 0;
    for (int i = 0; i < G->count; ++i)
        if (G->cls[i] == c)
            tiles += G->ntiles[i];
    int res = group_resident(G, c, tpw, splits, tiles);
    for (int waves = waves0; waves <= 32; ++waves) {
        const int R = std::min(res * waves, tiles);
        if (group_fit(G, c, tpw, splits, R, out))
            return true;
        if (R == tiles)
            return false;
    }
    return false;
}

// Default shape of class c: two tiles per unit; the K split from s0 up that
// needs the fewest CTAs in all (each CTA pays the prologue once), in whole
// waves of resident clusters, at least two (measured on the Q4_0 stack:
// better than one wave per split class).
bool group_fit_class(lbv_group* G, int c, int s0, lbv::GroupLaunch* out)
{
    bool found = false;
    long best_ctas = 0;
    for (int sp = s0; sp <= 8; ++sp) {
        lbv::GroupLaunch L;
        if (!group_fit_rows(G, c, 2, sp, 2, &L))
            continue;
        const long ctas = (long)L.shape.ctas_n * sp;
        if (!found || ctas < best_ctas) {
            found = true;
            best_ctas = ctas;
            *out = L;
        }
    }
    return found;
}

// Launch classes: one for all problems when a K split suits every one of
// them (problems of different lengths then share the GPU within one launch,
// which hides the long-K ones' slower streaming); otherwise each problem goes
// to the smallest split (1..8) at which its X slice fits in shared memory
// next to the ring, one class per split.
bool group_default_launches(lbv_group* G)
{
    const lbv::VerifyOps* ops = ops_for(G->fmt, G->group);
    std::fill(G->cls, G->cls + G->count, 0);
    G->nlaunch = 1;
    if (group_fit_class(G, 0, 1, &G->launch[0])) {
        for (int i = 0; i < G->count; ++i)
            G->cps[i] = group_problem_cps(G, i, G->launch[0].shape.splits);
        group_commit_rows(G, 0);
        return true;
    }
    int smin[lbv::kMaxGroup];
    for (int i = 0; i < G->count; ++i) {
        smin[i] = 0;
        for (int s = 1; s <= 8 && !smin[i]; ++s) {
            const int cp = group_problem_cps(G, i, s);
            if (cp && std::max(ops->smem(16, 2, cp, 1, s), kSmemOnePerSm) <= kSmemCap)
                smin[i] = s;
        }
        if (!smin[i])
            return false;
    }
    G->nlaunch = 0;
    std::fill(G->cls, G->cls + G->count, -1);         // no class yet
    for (int s = 1; s <= 8; ++s) {
        bool any = false;
        for (int i = 0; i < G->count; ++i)
            any |= smin[i] == s;
        if (!any)
            continue;
        const int c = G->nlaunch++;
        for (int i = 0; i < G->count; ++i)
            if (smin[i] == s)
                G->cls[i] = c;
        if (!group_fit_class(G, c, s, &G->launch[c]))
            return false;
    }
    for (int i = 0; i < G->count; ++i)
        G->cps[i] = group_problem_cps(G, i, G->launch[G->cls[i]].shape.splits);
    for (int c = 0; c < G->nlaunch; ++c)
        group_commit_rows(G, c);
    return true;
}

}  // namespace

namespace {

// One launch of class c over its problems with M[i] > 0 (none active: nothing).
lbv_status launch_class(const lbv_group* G, int c, const lbv_problem* problems, const int* M,
                        cudaStream_t stream)
{
    static thread_local lbv::GroupedParams gp;
    const lbv::GroupLaunch& L = G->launch[c];
    // cluster rows per active problem of the class, divided from the plan's R
    // and never fewer than the plan's, so that no row gets more tiles than
    // the partials were sized for; the largest rows go first, the hardware
    // fills the wave's end with the small ones
    int rows[lbv::kMaxGroup];
    divide_rows(G, c, L.rows_target, M, rows);
    for (int i = 0; i < G->count; ++i)
        if (rows[i] > 0)
            rows[i] = std::max(rows[i], G->rows_plan[i]);
    if (group_tiles_max(G, rows) > L.tiles_max)        // cannot happen (fewer active
        return fail(LBV_ERR_UNSUPPORTED,               // problems only add rows)
                    "lbv_verify_grouped: cluster rows exceed the plan's");
    int order[lbv::kMaxGroup];
    int n = 0;
    for (int i = 0; i < G->count; ++i)
        if (rows[i] > 0)
            order[n++] = i;
    if (n == 0)
        return LBV_OK;
    std::stable_sort(order, order + n, [&](int a, int b) {
        return G->bytes[a] / rows[a] > G->bytes[b] / rows[b];
    });
    gp.err = G->dev_err;
    gp.splits = L.shape.splits;
    gp.count = n;
    gp.ybegin[0] = 0;
    for (int j = 0; j < n; ++j) {
        const int i = order[j];
        const lbv_problem& q = problems[i];
        lbv::GroupedProblem& d = gp.prob[j];
        d.X = q.X;
        d.W = static_cast<const uint8_t*>(q.Wp);
        d.Y = q.Y;
        d.ldx = q.ldx;
        d.ldy = q.ldy;
        d.M = q.M;
        d.K = G->K[i];
        d.N = G->N[i];
        d.ntiles = G->ntiles[i];
        d.nchunks = G->nchunks[i];
        d.cps = G->cps[i];
        d.x_vec = ((reinterpret_cast<uintptr_t>(q.X) & 15u) == 0 && (q.ldx % 8) == 0) ? 1 : 0;
        gp.ybegin[j + 1] = gp.ybegin[j] + rows[i];
    }
    lbv::Shape sh = L.shape;
    sh.ctas_n = gp.ybegin[n];
    lbv::LaunchOpts o;
    o.pdl = (G->flags & LBV_PLAN_PDL) != 0;
    const cudaError_t e = ops_for(G->fmt, G->group)->launch_grouped(G->xdtype, sh, gp, o, stream);
    if (e != cudaSuccess)
        return cuda_fail(e, "lbv_verify_grouped: launch");
    return LBV_OK;
}

// LBV_PLAN_MEASURE: for every class, time the default shape and one to six
// waves of each K split from the class's own up to 8 (cold L2, scratch
// weights and activations of the class's shapes, M = 8); keep the fastest.
// (On the Q4_0 stack: 4 waves 180 us, 5 waves 172 us, 6 waves 181 us.)
lbv_status group_measure(lbv_group* G)
{
    std::vector<size_t> woff(G->count), xoff(G->count), yoff(G->count);
    size_t wb = 0, xb = 0, yb = 0;
    for (int i = 0; i < G->count; ++i) {
        woff[i] = wb;
        wb += ((size_t)G->bytes[i] + 255) / 256 * 256;
        xoff[i] = xb;
        xb += ((size_t)8 * G->K[i] * 2 + 255) / 256 * 256;
        yoff[i] = yb;
        yb += ((size_t)8 * G->N[i] * 4 + 255) / 256 * 256;
    }
    Scratch s;
    int l2 = 0;
    cudaDeviceGetAttribute(&l2, cudaDevAttrL2CacheSize, G->device);
    s.flush_bytes = (size_t)std::max(l2, 1 << 20) * 2;
    cudaError_t e = cudaMalloc(&s.w, wb);
    if (e == cudaSuccess) e = cudaMalloc(&s.x, xb);
    if (e == cudaSuccess) e = cudaMalloc((void**)&s.y, yb);
    if (e == cudaSuccess) e = cudaMalloc(&s.flush, s.flush_bytes);
    if (e == cudaSuccess) e = cudaMemset(s.w, 0x5A, wb);
    if (e == cudaSuccess) e = cudaMemset(s.x, 0x11, xb);
    if (e != cudaSuccess)
        return cuda_fail(e, "group measure: scratch");
    std::vector<lbv_problem> probs(G->count);
    int M[lbv::kMaxGroup];
    for (int i = 0; i < G->count; ++i) {
        probs[i].X = static_cast<unsigned char*>(s.x) + xoff[i];
        probs[i].M = 8;
        probs[i].ldx = G->K[i];
        probs[i].Wp = static_cast<unsigned char*>(s.w) + woff[i];
        probs[i].Y = reinterpret_cast<float*>(reinterpret_cast<unsigned char*>(s.y) + yoff[i]);
        probs[i].ldy = G->N[i];
        M[i] = 8;
    }
    cudaStream_t st = nullptr;
    for (int c = 0; c < G->nlaunch; ++c) {
        const int s0 = G->launch[c].shape.splits;
        int tiles = 0;
        for (int i = 0; i < G->count; ++i)
            if (G->cls[i] == c)
                tiles += G->ntiles[i];
        const lbv::GroupLaunch dflt = G->launch[c];
        lbv::GroupLaunch best = dflt;
        float best_us = 1e30f;
        for (int sp = s0; sp <= 8; ++sp) {
            const int res = group_resident(G, c, 2, sp, tiles);
            for (int waves = 0; waves <= 6; ++waves) {   // 0: the default shape
                lbv::GroupLaunch L;
                if (waves == 0) {
                    if (sp != dflt.shape.splits)
                        continue;
                    L = dflt;
                } else if (!group_fit(G, c, 2, sp, std::min(res * waves, tiles), &L)) {
                    continue;
                }
                G->launch[c] = L;
                for (int i = 0; i < G->count; ++i)
                    if (G->cls[i] == c)
                        G->cps[i] = group_problem_cps(G, i, sp);
                group_commit_rows(G, c);
                float us = 0.f;
                const lbv_status rc =
                    time_cold([&] { return launch_class(G, c, probs.data(), M, st); }, s, st, 5, &us);
                if (rc != LBV_OK)
                    return rc;
                if (us < best_us) {
                    best_us = us;
                    best = L;
                }
            }
        }
        G->launch[c] = best;
        for (int i = 0; i < G->count; ++i)
            if (G->cls[i] == c)
                G->cps[i] = group_problem_cps(G, i, best.shape.splits);
        group_commit_rows(G, c);
    }
    return LBV_OK;
}

}  // namespace

lbv_status lbv_group_create(lbv_format fmt, int group, lbv_dtype xdtype, int count, const int* K,
                            const int* N, unsigned flags, lbv_group** out)
{
    g_err.clear();
    if (!out)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_create: out is NULL");
    *out = nullptr;
    if (!valid_fmt(fmt))
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_create: unknown format %d", (int)fmt);
    if (xdtype != LBV_F16 && xdtype != LBV_BF16)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_create: unknown dtype %d", (int)xdtype);
    if (fmt == LBV_FMT_AFFINE2 && group != 32 && group != 64 && group != 128)
        return fail(LBV_ERR_UNSUPPORTED, "lbv_group_create: affine group %d (supported: 32, 64, 128)",
                    group);
    if (fmt != LBV_FMT_AFFINE2)
        group = fmt == LBV_FMT_SIGN1_G128 ? 128 : 32;
    if (count < 1 || count > lbv::kMaxGroup || !K || !N)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_create: count=%d outside 1..%d or no shapes",
                    count, lbv::kMaxGroup);
    if (flags & ~(LBV_PLAN_PDL | LBV_PLAN_MEASURE))
        return fail(LBV_ERR_INVALID_ARG,
                    "lbv_group_create: flags 0x%x (only LBV_PLAN_PDL, LBV_PLAN_MEASURE)", flags);
    for (int i = 0; i < count; ++i)
        if (K[i] <= 0 || N[i] <= 0 || K[i] % k_quantum(fmt, group) != 0)
            return fail(LBV_ERR_INVALID_ARG,
                        "lbv_group_create: problem %d: K=%d N=%d not valid for the format", i,
                        K[i], N[i]);
    lbv_group* G = new (std::nothrow) lbv_group();
    if (!G)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_create: out of host memory");
    G->fmt = fmt;
    G->xdtype = xdtype;
    G->group = group;
    G->flags = flags;
    G->count = count;
    lbv::fmt_info(fmt, group, &G->fi);
    for (int i = 0; i < count; ++i) {
        const lbv::Layout L = lbv::make_layout(G->fi, K[i], N[i]);
        G->K[i] = K[i];
        G->N[i] = N[i];
        G->ntiles[i] = (int)L.ntiles;
        G->nchunks[i] = (int)L.nchunks;
        G->bytes[i] = (double)L.total;
    }
    cudaError_t e = cudaGetDevice(&G->device);
    if (e == cudaSuccess)
        e = cudaDeviceGetAttribute(&G->sms, cudaDevAttrMultiProcessorCount, G->device);
    if (e == cudaSuccess)
        e = cudaMalloc((void**)&G->dev_err, 256);
    if (e == cudaSuccess)
        e = cudaMemset(G->dev_err, 0, 256);
    if (e != cudaSuccess) {
        cudaFree(G->dev_err);
        delete G;
        return cuda_fail(e, "lbv_group_create: device set-up");
    }
    if (!group_default_launches(G)) {
        lbv_group_destroy(G);
        return fail(LBV_ERR_UNSUPPORTED,
                    "lbv_group_create: a problem fits no K split of 1..8 in shared memory");
    }
    if (flags & LBV_PLAN_MEASURE) {
        const lbv_status st = group_measure(G);
        if (st != LBV_OK) {
            lbv_group_destroy(G);
            return st;
        }
    }
    *out = G;
    return LBV_OK;
}

lbv_status lbv_group_destroy(lbv_group* G)
{
    if (G) {
        cudaFree(G->dev_err);
        delete G;
    }
    return LBV_OK;
}

int lbv_group_launches(const lbv_group* G)
{
    return G ? G->nlaunch : 0;
}

int lbv_group_problem_launch(const lbv_group* G, int problem)
{
    return (G && problem >= 0 && problem < G->count) ? G->cls[problem] : -1;
}

lbv_status lbv_group_shape(const lbv_group* G, int launch, int* tpw, int* splits, int* rows)
{
    g_err.clear();
    if (!G)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_shape: group is NULL");
    if (launch < 0 || launch >= G->nlaunch)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_shape: launch %d of %d", launch, G->nlaunch);
    const lbv::Shape& sh = G->launch[launch].shape;
    if (tpw)
        *tpw = sh.tpw;
    if (splits)
        *splits = sh.splits;
    if (rows)
        *rows = sh.ctas_n;
    return LBV_OK;
}

lbv_status lbv_group_set_shape(lbv_group* G, int tpw, int splits, int rows)
{
    g_err.clear();
    if (!G)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_set_shape: group is NULL");
    if ((tpw != 1 && tpw != 2) || splits < 1 || splits > 8 || rows < 1)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_set_shape: tpw=%d splits=%d rows=%d", tpw,
                    splits, rows);
    int cls_saved[lbv::kMaxGroup];
    std::copy(G->cls, G->cls + G->count, cls_saved);
    std::fill(G->cls, G->cls + G->count, 0);
    lbv::GroupLaunch L;
    if (!group_fit(G, 0, tpw, splits, rows, &L)) {
        std::copy(cls_saved, cls_saved + G->count, G->cls);
        return fail(LBV_ERR_UNSUPPORTED,
                    "lbv_group_set_shape: the split does not suit every problem, or the shape "
                    "does not fit (shared memory or occupancy)");
    }
    G->nlaunch = 1;
    G->launch[0] = L;
    for (int i = 0; i < G->count; ++i)
        G->cps[i] = group_problem_cps(G, i, splits);
    group_commit_rows(G, 0);
    return LBV_OK;
}

lbv_status lbv_group_device_status(const lbv_group* G)
{
    g_err.clear();
    if (!G)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_device_status: group is NULL");
    unsigned v = 0;
    cudaError_t e = cudaMemcpy(&v, G->dev_err, sizeof v, cudaMemcpyDeviceToHost);
    if (e != cudaSuccess)
        return cuda_fail(e, "lbv_group_device_status");
    if (v) {
        cudaMemset(G->dev_err, 0, sizeof v);
        if (v & 2u)
            return fail(LBV_ERR_BOUNDS, "a grouped verify kernel found a copy or buffer range "
                                        "outside its bounds and skipped it");
        return fail(LBV_ERR_TIMEOUT, "a grouped verify kernel gave up waiting for its weight copies");
    }
    return LBV_OK;
}

lbv_status lbv_verify_grouped(const lbv_group* G, const lbv_problem* problems, lbv_stream stream)
{
    g_err.clear();
    if (!G || !problems)
        return fail(LBV_ERR_INVALID_ARG, "lbv_verify_grouped: NULL group or problems");
    int dev = -1;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != G->device)
        return fail(LBV_ERR_INVALID_ARG, "lbv_verify_grouped: current device %d is not the group's %d",
                    dev, G->device);
    int M[lbv::kMaxGroup];
    for (int i = 0; i < G->count; ++i) {
        const lbv_problem& q = problems[i];
        if (q.M < 0 || q.M > 8)
            return fail(LBV_ERR_INVALID_ARG, "lbv_verify_grouped: problem %d: M=%d outside 0..8", i,
                        q.M);
        M[i] = q.M;
        if (q.M == 0)
            continue;
        if (!q.X || !q.Wp || !q.Y)
            return fail(LBV_ERR_INVALID_ARG, "lbv_verify_grouped: problem %d: null X, Wp or Y", i);
        if (q.ldx < G->K[i] || q.ldy < G->N[i])
            return fail(LBV_ERR_INVALID_ARG,
                        "lbv_verify_grouped: problem %d: ldx=%d < K=%d or ldy=%d < N=%d", i, q.ldx,
                        G->K[i], q.ldy, G->N[i]);
        if ((reinterpret_cast<uintptr_t>(q.Wp) & 15u) || (reinterpret_cast<uintptr_t>(q.X) & 1u) ||
            (reinterpret_cast<uintptr_t>(q.Y) & 3u))
            return fail(LBV_ERR_INVALID_ARG, "lbv_verify_grouped: problem %d: misaligned pointer", i);
    }
    for (int c = 0; c < G->nlaunch; ++c) {
        const lbv_status st = launch_class(G, c, problems, M, reinterpret_cast<cudaStream_t>(stream));
        if (st != LBV_OK)
            return st;
    }
    for (int i = 0; i < G->count; ++i)
        if (M[i] > 0)
            count_rows(G->rows_calls, M[i]);
    return LBV_OK;
}

lbv_status lbv_group_rows_histogram(const lbv_group* G, uint64_t* counts)
{
    g_err.clear();
    if (!G || !counts)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_rows_histogram: NULL group or counts");
    for (int m = 0; m < 8; ++m)
        counts[m] = G->rows_calls[m].load(std::memory_order_relaxed);
    return LBV_OK;
}

lbv_status lbv_group_rows_reset(lbv_group* G)
{
    g_err.clear();
    if (!G)
        return fail(LBV_ERR_INVALID_ARG, "lbv_group_rows_reset: group is NULL");
    for (int m = 0; m < 8; ++m)
        G->rows_calls[m].store(0, std::memory_order_relaxed);
    return LBV_OK;
}

lbv_status lbv_rows_histogram(uint64_t* counts)
{
    g_err.clear();
    if (!counts)
        return fail(LBV_ERR_INVALID_ARG, "lbv_rows_histogram: counts is NULL");
    for (int m = 0; m < 8; ++m)
        counts[m] = g_rows[m].load(std::memory_order_relaxed);
    return LBV_OK;
}
