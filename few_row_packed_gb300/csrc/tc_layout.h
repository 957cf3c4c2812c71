// tc_layout.h -- the 128-column record layout read by the tcgen05 few-row
// kernel (plans created with LBV_PLAN_TCGEN05), shared by its host packer
// (api.cpp) and its kernels.  Lossless: the same bits as the
// canonical file layout, rearranged so that one thread owns one output column
// and finds a chunk of that column's codes in 16 or 32 contiguous bytes.
//
// Terms
//   tile   128 output columns n = 128*tile .. 128*tile+127: the M side of one
//          tcgen05 MMA (the M <= 8 activation rows are the N side).
//   chunk  CK consecutive K values of a column: 128 (sign1), 64 (affine2 g32
//          and g64, Q4_0) or 128 (affine2 g128).  CB = 16 or 32 code bytes.
//   pair   the two weights k = 2p and 2p + 1 of a column: one 32-bit register
//          of two fp16/bf16 values in the MMA's A operand.
//
// Records: one record of REC = 128 * (CB + SB) bytes per (tile, chunk), in
// tile-major order (record index tile * nchunks + chunk):
//   codes: [CB / 16][128 columns][16 bytes].  The CB bytes of a column are
//          CB / 4 little-endian words; word j holds pairs p = PPW*j + s for
//          s = 0..PPW-1 (PPW = 16 / W pairs per word, W = bits per code): the
//          code of k = 2p sits at bit s*W of the low half-word and the code of
//          k = 2p + 1 at bit 16 + s*W.
//   side:  [128 columns][SB bytes] of fp16 bit patterns, per scale group j of
//          the chunk: sign1: scale (SB = 2); affine2: scale, bias (4 bytes per
//          group; SB = 4, or 8 for g32); Q4_0: d (2 bytes per block, SB = 4).
// Padding columns (n >= N) and K positions (k >= K) have zero codes and zero
// scales, so they contribute exactly 0.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/lbv.h"

namespace lbv {

constexpr int kTcTileN = 128;

struct TcFmtInfo {
    int chunk_k;      // K per chunk (CK)
    int code_bytes;   // code bytes per column and chunk (CB)
    int side_bytes;   // side bytes per column and chunk (SB)
    int code_bits;    // W
    int group_k;      // K per scale group
};

inline bool tc_fmt_info(lbv_format fmt, int group, TcFmtInfo* fi)
{
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        *fi = {128, 16, 2, 1, 128};
        return true;
    case LBV_FMT_AFFINE2:
        if (group == 32) { *fi = {64, 16, 8, 2, 32}; return true; }
        if (group == 64) { *fi = {64, 16, 4, 2, 64}; return true; }
        if (group == 128) { *fi = {128, 32, 4, 2, 128}; return true; }
        return false;
    case LBV_FMT_Q4_0:
        *fi = {64, 32, 4, 4, 32};
        return true;
    }
    return false;
}

struct TcLayout {
    int64_t ntiles;        // ceil(N / 128)
    int64_t nchunks;       // ceil(K / chunk_k)
    size_t rec_bytes;      // 128 * (CB + SB)
    size_t total;          // ntiles * nchunks * rec_bytes
};

inline TcLayout tc_make_layout(const TcFmtInfo& fi, int K, int N)
{
    TcLayout L;
    L.ntiles = (N + kTcTileN - 1) / kTcTileN;
    L.nchunks = (K + fi.chunk_k - 1) / fi.chunk_k;
    L.rec_bytes = (size_t)kTcTileN * (size_t)(fi.code_bytes + fi.side_bytes);
    L.total = (size_t)L.ntiles * (size_t)L.nchunks * L.rec_bytes;
    return L;
}

// Launch shape of the tcgen05 few-row kernel.
struct TcShape {
    int splits;             // K slices (cluster size), 1..8
    int ctas_n;             // clusters along N (grid y); each owns a contiguous tile range
    int wsplit;             // warpgroups sharing one tile inside a CTA (split of the slice)
    size_t smem;            // dynamic shared memory bytes
};

}  // namespace lbv
