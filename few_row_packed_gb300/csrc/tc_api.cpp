// tc_api.cpp -- host side of plans created with LBV_PLAN_TCGEN05: launch-shape
// selection for the tcgen05 few-row kernel, its launch, and the packer of its
// 128-column record layout (tc_layout.h).  Called from api.cpp.
#include <string.h>

#include <algorithm>

#include "tc_internal.h"
#include "tc_api.h"

namespace lbv {

namespace {

const TcOps* tc_ops_for(lbv_format fmt, int group)
{
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        return &tc_sign1_ops;
    case LBV_FMT_AFFINE2:
        return group == 32 ? &tc_affine2_g32_ops : group == 64 ? &tc_affine2_g64_ops
                                                               : &tc_affine2_g128_ops;
    case LBV_FMT_Q4_0:
        return &tc_q4_0_ops;
    }
    return nullptr;
}

constexpr size_t kSmemCap = 220 * 1024;        // per CTA, of 227 KB
// Requesting more than half of an SM's shared memory keeps the scheduler from
// placing two CTAs of one grid on an SM (each allocates all tensor memory).
constexpr size_t kSmemOnePerSm = 116 * 1024;

int tc_cps(const TcShape& sh, int64_t nchunks)
{
    return (int)((nchunks + sh.splits - 1) / sh.splits);
}

// Work of the busiest warpgroup, in (tile, chunk) records, for `tpc` tiles
// per cluster, `cps` chunks per slice and a warpgroup split `sw`.
int64_t wg_load(int64_t tpc, int cps, int sw)
{
    const int64_t lanes = kTcWarpgroups / sw;
    return ((tpc + lanes - 1) / lanes) * ((cps + sw - 1) / sw);
}

// Fills sh.smem and sh.wsplit for sh.splits and sh.ctas_n: the warpgroup
// split with the least work per warpgroup whose partial buffers fit.
bool fit_shape(const lbv_plan* P, TcShape& sh, int cps)
{
    const TcOps* ops = tc_ops_for(P->fmt, P->group);
    const int64_t tpc = (P->tc_layout.ntiles + sh.ctas_n - 1) / sh.ctas_n;
    const int owned = (int)((tpc + sh.splits - 1) / sh.splits);
    int64_t best = -1;
    for (int sw = 1; sw <= kTcWarpgroups; ++sw) {
        if (kTcWarpgroups % sw != 0 || (sw > 1 && sw > cps))
            continue;
        const size_t smem = std::max(ops->smem(cps, owned, sh.splits * sw), kSmemOnePerSm);
        if (smem > kSmemCap)
            continue;
        const int64_t load = wg_load(tpc, cps, sw);
        if (best < 0 || load < best) {
            best = load;
            sh.wsplit = sw;
            sh.smem = smem;
        }
    }
    return best >= 0;
}

// Fills sh.splits (clamped so every slice has >= 1 chunk), sh.ctas_n,
// sh.wsplit and sh.smem: one cluster of `splits` CTAs per `splits` SMs, as
// many clusters as can be resident, each owning a contiguous tile range.
// ctas_req > 0 caps the number of clusters.  False if nothing fits.
bool complete_shape(const lbv_plan* P, TcShape& sh, int ctas_req)
{
    const TcOps* ops = tc_ops_for(P->fmt, P->group);
    const int64_t nchunks = P->tc_layout.nchunks;
    int cps = tc_cps(sh, nchunks);
    sh.splits = (int)((nchunks + cps - 1) / cps);
    cps = tc_cps(sh, nchunks);
    const int64_t ntiles = P->tc_layout.ntiles;
    int64_t G = std::max<int64_t>(1, std::min<int64_t>(ntiles, P->sms / sh.splits));
    if (ctas_req > 0)
        G = std::min<int64_t>(G, ctas_req);
    for (int it = 0; it < 4; ++it) {
        sh.ctas_n = (int)G;
        if (!fit_shape(P, sh, cps) || ops->prepare(P->xdtype, sh) != cudaSuccess)
            return false;
        const int maxc = ops->max_clusters(P->xdtype, sh);
        if (maxc < 1)
            return false;
        if (G <= maxc)
            return true;
        G = maxc;
    }
    sh.ctas_n = (int)G;
    return fit_shape(P, sh, cps) && ops->prepare(P->xdtype, sh) == cudaSuccess;
}

// Generic packer: code(n, k) -> W-bit code (0 outside the matrix), side(n,
// chunk, i) -> the i-th fp16 side value of column n in that chunk.
template <class CodeF, class SideF>
void pack_records(const TcFmtInfo& fi, int K, int N, uint8_t* out, CodeF code, SideF side)
{
    const TcLayout L = tc_make_layout(fi, K, N);
    const int W = fi.code_bits, PPW = 16 / W, NWORD = fi.code_bytes / 4;
    const int nside = fi.side_bytes / 2;
    for (int64_t tile = 0; tile < L.ntiles; ++tile)
        for (int64_t ch = 0; ch < L.nchunks; ++ch) {
            uint8_t* rec = out + ((size_t)tile * L.nchunks + ch) * L.rec_bytes;
            for (int c = 0; c < kTcTileN; ++c) {
                const int n = (int)tile * kTcTileN + c;
                for (int j = 0; j < NWORD; ++j) {
                    uint32_t w = 0;
                    for (int s = 0; s < PPW; ++s) {
                        const int k0 = (int)ch * fi.chunk_k + 2 * (PPW * j + s);
                        w |= code(n, k0) << (s * W);
                        w |= code(n, k0 + 1) << (16 + s * W);
                    }
                    memcpy(rec + (j / 4) * 2048 + c * 16 + (j % 4) * 4, &w, 4);
                }
                uint16_t* sd = reinterpret_cast<uint16_t*>(rec + kTcTileN * fi.code_bytes +
                                                           c * fi.side_bytes);
                for (int i = 0; i < nside; ++i)
                    sd[i] = n < N ? side(n, (int)ch, i) : (uint16_t)0;
            }
        }
}

}  // namespace

bool tc_plan_setup(lbv_plan* P)
{
    tc_fmt_info(P->fmt, P->group, &P->tc_fi);
    P->tc_layout = tc_make_layout(P->tc_fi, P->K, P->N);
    // default: the K split that minimises what the busiest warpgroup streams
    // plus half the activation bytes a CTA stages
    TcShape best = {0, 0, 1, 0};
    double best_cost = 1e300;
    for (int s = 1; s <= 8; ++s) {
        TcShape sh = {s, 0, 1, 0};
        if (!complete_shape(P, sh, 0) || sh.splits != s)
            continue;
        const int cps = tc_cps(sh, P->tc_layout.nchunks);
        const int64_t tpc = (P->tc_layout.ntiles + sh.ctas_n - 1) / sh.ctas_n;
        const double cost = (double)wg_load(tpc, cps, sh.wsplit) * P->tc_layout.rec_bytes +
                            0.5 * (double)cps * P->tc_fi.chunk_k * 16.0;
        if (cost < best_cost * 0.98) {
            best_cost = cost;
            best = sh;
        }
    }
    if (best.splits == 0)
        return false;
    P->tc_shape = best;
    return true;
}

bool tc_set_shape(lbv_plan* P, int splits, int ctas_n)
{
    TcShape sh = {splits, 0, 1, 0};
    if (!complete_shape(P, sh, ctas_n))
        return false;
    P->tc_shape = sh;
    return true;
}

cudaError_t tc_verify_launch(const lbv_plan* P, const void* X, int M, int ldx, const void* Wp,
                             float* Y, int ldy, bool pdl, cudaStream_t st)
{
    TcParams p;
    p.X = X;
    p.W = static_cast<const uint8_t*>(Wp);
    p.Y = Y;
    p.err = P->dev_err;
    p.ldx = ldx;
    p.ldy = ldy;
    p.M = M;
    p.K = P->K;
    p.N = P->N;
    p.ntiles = (int)P->tc_layout.ntiles;
    p.nchunks = (int)P->tc_layout.nchunks;
    p.splits = P->tc_shape.splits;
    p.cps = tc_cps(P->tc_shape, P->tc_layout.nchunks);
    p.wsplit = P->tc_shape.wsplit;
    p.x_vec = ((reinterpret_cast<uintptr_t>(X) & 15u) == 0 && (ldx % 8) == 0) ? 1 : 0;
    p.zero = 0;
    LaunchOpts o;
    o.pdl = pdl;
    return tc_ops_for(P->fmt, P->group)->launch(P->xdtype, P->tc_shape, p, o, st);
}

cudaError_t tc_dequant(const lbv_plan* P, const void* Wp, uint16_t* W, cudaStream_t st)
{
    return tc_launch_dequant(P->fmt, P->group, static_cast<const uint8_t*>(Wp), P->K, P->N,
                             (int)P->tc_layout.ntiles, (int)P->tc_layout.nchunks, W, st);
}

size_t tc_packed_bytes(const lbv_plan* P)
{
    return P->tc_layout.total;
}

void tc_pack(const lbv_plan* P, const void* part0, const void* part1, const void* part2,
             uint8_t* out)
{
    const int K = P->K, N = P->N, group = P->group;
    const TcFmtInfo& fi = P->tc_fi;
    if (P->fmt == LBV_FMT_SIGN1_G128) {
        const uint32_t* bits = static_cast<const uint32_t*>(part0);
        const uint16_t* scales = static_cast<const uint16_t*>(part1);
        const int wk = K / 32, sk = K / 128;
        pack_records(
            fi, K, N, out,
            [&](int n, int k) -> uint32_t {
                if (n >= N || k >= K) return 0u;
                return (bits[(size_t)n * wk + k / 32] >> (k % 32)) & 1u;
            },
            [&](int n, int ch, int) -> uint16_t {
                return ch < sk ? scales[(size_t)n * sk + ch] : (uint16_t)0;
            });
    } else if (P->fmt == LBV_FMT_AFFINE2) {
        const uint32_t* codes = static_cast<const uint32_t*>(part0);
        const uint16_t* scales = static_cast<const uint16_t*>(part1);
        const uint16_t* biases = static_cast<const uint16_t*>(part2);
        const int wk = K / 16, gk = K / group, gpc = fi.chunk_k / group;
        pack_records(
            fi, K, N, out,
            [&](int n, int k) -> uint32_t {
                if (n >= N || k >= K) return 0u;
                return (codes[(size_t)n * wk + k / 16] >> (2 * (k % 16))) & 3u;
            },
            [&](int n, int ch, int i) -> uint16_t {
                const int grp = ch * gpc + i / 2;
                if (grp >= gk) return 0;
                return (i % 2 ? biases : scales)[(size_t)n * gk + grp];
            });
    } else {
        const uint8_t* blocks = static_cast<const uint8_t*>(part0);
        const int nb = K / 32;
        pack_records(
            fi, K, N, out,
            [&](int n, int k) -> uint32_t {
                if (n >= N || k >= K) return 0u;
                const uint8_t* blk = blocks + ((size_t)n * nb + k / 32) * 18;
                const int j = k % 32;
                return j < 16 ? (blk[2 + j] & 15u) : (uint32_t)(blk[2 + j - 16] >> 4);
            },
            [&](int n, int ch, int i) -> uint16_t {
                const int b = ch * 2 + i;
                if (b >= nb) return 0;
                const uint8_t* blk = blocks + ((size_t)n * nb + b) * 18;
                return (uint16_t)(blk[0] | (blk[1] << 8));
            });
    }
}

}  // namespace lbv
