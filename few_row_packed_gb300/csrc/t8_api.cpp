// t8_api.cpp -- host side of plans created with LBV_PLAN_TC_E4M3: launch-shape
// selection for the e4m3 tensor-memory kernel, its launch, and the packer of
// its record layout (t8_layout.h).  Called from api.cpp.
#include <string.h>

#include <algorithm>

#include "t8_api.h"
#include "t8_internal.h"

namespace lbv {

namespace {

const T8Ops* t8_ops_for(lbv_format fmt)
{
    return fmt == LBV_FMT_SIGN1_G128 ? &t8_sign1_ops : &t8_affine2_g128_ops;
}

int t8_gps(int splits, int64_t ngroups)
{
    return (int)((ngroups + splits - 1) / splits);
}

// Completes sh for sh.splits: groups per slice (every slice non-empty, so the
// split may shrink), clusters along N (one CTA per SM, as many as can be
// resident; ctas_req > 0 caps them), the owner slots and the shared memory.
bool complete_shape(const lbv_plan* P, T8Shape& sh, int ctas_req)
{
    const T8Ops* ops = t8_ops_for(P->fmt);
    const int64_t ngroups = P->t8_layout.ngroups, ntiles = P->t8_layout.ntiles;
    sh.gps = t8_gps(sh.splits, ngroups);
    sh.splits = (int)((ngroups + sh.gps - 1) / sh.gps);
    int64_t G = std::max<int64_t>(1, std::min<int64_t>(ntiles, P->sms / sh.splits));
    if (ctas_req > 0)
        G = std::min<int64_t>(G, ctas_req);
    for (int it = 0; it < 4; ++it) {
        sh.ctas_n = (int)G;
        sh.tpc = (int)((ntiles + G - 1) / G);
        sh.owned = sh.splits > 1 ? (sh.tpc + sh.splits - 1) / sh.splits : 0;
        sh.x_in_ring = ops->x_fits_ring(sh.gps) ? 1 : 0;
        sh.smem = std::max(ops->smem(sh.gps, sh.splits, sh.owned, sh.x_in_ring), kT8SmemOnePerSm);
        if (sh.smem > (size_t)kT8MaxSmem)
            return false;
        if (ops->prepare(P->xdtype, sh) != cudaSuccess)
            return false;
        const int maxc = ops->max_clusters(P->xdtype, sh);
        if (maxc < 1)
            return false;
        if (G <= maxc)
            return true;
        G = maxc;
    }
    return false;
}

// Busiest warpgroup's groups plus the prologue's share (per group of the
// slice: staging, split into B, row sums), in group-iteration units.
double shape_cost(const T8Shape& sh)
{
    return (double)((sh.tpc + 3) / 4) * sh.gps + 0.3 * sh.gps;
}

}  // namespace

bool t8_plan_setup(lbv_plan* P)
{
    if (!t8_fmt_info(P->fmt, P->group, &P->t8_fi) || P->K % kT8GroupK != 0)
        return false;
    P->t8_layout = t8_make_layout(P->t8_fi, P->K, P->N);
    T8Shape best = {};
    double best_cost = 1e300;
    for (int s = 1; s <= 8; s <<= 1) {
        T8Shape sh = {};
        sh.splits = s;
        if (!complete_shape(P, sh, 0) || sh.splits != s)
            continue;
        const double c = shape_cost(sh);
        if (c < best_cost * 0.98) {
            best_cost = c;
            best = sh;
        }
    }
    if (best.splits == 0)
        return false;
    P->t8_shape = best;
    return true;
}

bool t8_set_shape(lbv_plan* P, int splits, int ctas_n)
{
    if (splits != 1 && splits != 2 && splits != 4 && splits != 8)
        return false;
    T8Shape sh = {};
    sh.splits = splits;
    if (!complete_shape(P, sh, ctas_n))
        return false;
    P->t8_shape = sh;
    return true;
}

cudaError_t t8_verify_launch(const lbv_plan* P, const void* X, int M, int ldx, const void* Wp,
                             float* Y, int ldy, const T8Fused& f, bool pdl, cudaStream_t st)
{
    T8Params p;
    p.X = X;
    p.W = static_cast<const uint8_t*>(Wp);
    p.Y = Y;
    p.err = P->dev_err;
    p.ldx = ldx;
    p.ldy = ldy;
    p.M = M;
    p.K = P->K;
    p.N = P->N;
    p.ntiles = (int)P->t8_layout.ntiles;
    p.ngroups = (int)P->t8_layout.ngroups;
    p.splits = P->t8_shape.splits;
    p.gps = P->t8_shape.gps;
    p.owned = P->t8_shape.owned;
    p.x_vec = ((reinterpret_cast<uintptr_t>(X) & 15u) == 0 && (ldx % 8) == 0) ? 1 : 0;
    p.x_in_ring = P->t8_shape.x_in_ring;
    p.wait_limit = 0;
    p.rot = f.rot;
    p.store_y = f.store_y;
    p.signs = f.signs;
    p.amax_keys = f.amax_keys;
    p.amax_done = f.amax_done;
    p.amax_idx = f.amax_idx;
    p.amax_val = f.amax_val;
    LaunchOpts o;
    o.pdl = pdl;
    return t8_ops_for(P->fmt)->launch(P->xdtype, P->t8_shape, p, o, st);
}

cudaError_t t8_dequant(const lbv_plan* P, const void* Wp, uint16_t* W, cudaStream_t st)
{
    return t8_ops_for(P->fmt)->dequant(static_cast<const uint8_t*>(Wp), P->K, P->N,
                                       (int)P->t8_layout.ntiles, (int)P->t8_layout.ngroups, W, st);
}

size_t t8_packed_bytes(const lbv_plan* P)
{
    return P->t8_layout.total;
}

void t8_pack(const lbv_plan* P, const void* part0, const void* part1, const void* part2,
             uint8_t* out)
{
    const int K = P->K, N = P->N;
    const T8FmtInfo& fi = P->t8_fi;
    const T8Layout& L = P->t8_layout;
    const int W = fi.code_bits, CB = fi.code_bytes, SB = fi.side_bytes;
    const int gk = K / kT8GroupK;
    const bool sign = P->fmt == LBV_FMT_SIGN1_G128;
    const uint32_t* words = static_cast<const uint32_t*>(part0);
    const uint16_t* scales = static_cast<const uint16_t*>(part1);
    const uint16_t* biases = static_cast<const uint16_t*>(part2);
    const int wk = sign ? K / 32 : K / 16;                   // canonical words per column
    memset(out, 0, L.total);
    uint32_t cw[8];
    for (int64_t tile = 0; tile < L.ntiles; ++tile)
        for (int64_t g = 0; g < L.ngroups; ++g)
            for (int q = 0; q < 4; ++q) {
                uint8_t* rec = out + (((size_t)tile * L.ngroups + g) * 4 + q) * L.rec_bytes;
                for (int lane = 0; lane < 32; ++lane) {
                    const int n = (int)tile * kT8TileN + q * 32 + lane;
                    if (n >= N)
                        continue;                            // zero codes and scales
                    memset(cw, 0, sizeof cw);
                    for (int k = 0; k < kT8GroupK; ++k) {
                        const int kg = (int)g * kT8GroupK + k;
                        uint32_t code;
                        if (sign)
                            code = (words[(size_t)n * wk + kg / 32] >> (kg % 32)) & 1u;
                        else
                            code = (words[(size_t)n * wk + kg / 16] >> (2 * (kg % 16))) & 3u;
                        int wi, bit;
                        t8_code_pos(W, k, &wi, &bit);
                        cw[wi] |= code << bit;
                    }
                    for (int i = 0; i < CB / 4; ++i)
                        memcpy(rec + (i / 4) * 512 + lane * 16 + (i % 4) * 4, &cw[i], 4);
                    uint16_t* sd = reinterpret_cast<uint16_t*>(rec + 32 * CB + lane * SB);
                    sd[0] = scales[(size_t)n * gk + g];
                    if (!sign)
                        sd[1] = biases[(size_t)n * gk + g];
                }
            }
}

}  // namespace lbv
