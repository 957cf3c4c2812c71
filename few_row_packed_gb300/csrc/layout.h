// layout.h -- the library's device layout of packed weights, shared by the
// host packer (pack.cpp) and the kernels.  Lossless: the same bits as the
// canonical file layout, rearranged so that one 16-byte load per lane gives a
// warp exactly the mma.sync m16n8k16 A-fragment bits of one 16-column tile.
//
// Terms
//   tile   16 output columns n = 16*tile .. 16*tile+15 (the m16 side of the
//          tensor-core tile; the M <= 8 activation rows are the n8 side).
//   chunk  the K range one 16-byte load per lane covers for one tile:
//          256 K (sign1), 128 K (affine2), 64 K (Q4_0); 512 bytes per tile.
//   lane   warp lane = 4*g + t, g = lane >> 2 in 0..7, t = lane & 3.
//
// Records: one record of REC = 512 + 8 * SB bytes per (tile, chunk), in
// tile-major order (record index tile * nchunks + chunk), so the chunks of a
// tile are contiguous.  A record holds
//   codes: uint4 [32 lanes] (512 bytes).  Word wi (0..3) of lane (g, t)
//          belongs to column 16*tile + g + 8*(wi & 1) and covers the chunk's
//          k-tiles (wi >> 1) * KT/2 .. + KT/2 - 1 (KT = chunk / 16).  Slot s
//          of that word is k-tile ktl = s >> 1 of the half and r = s & 1,
//          i.e. the two weights k0 = 16*kt + 8*r + 2*t and k0 + 1 -- the
//          element pair the A-fragment register for (column, kt, r) holds.
//          The code of k0 sits at bit s*W (W = 1, 2, 4 bits) of the low
//          half-word and the code of k0 + 1 at bit 16 + s*W.
//   side:  uint8 [8 g][SB] of fp16 bit patterns:
//          sign1   : per group j (2 per chunk): scale(col g), scale(col g+8)
//          affine2 : per group j (128/g per chunk): scale(g), scale(g+8),
//                    bias(g), bias(g+8)
//          Q4_0    : per block j (2 per chunk): d(col g), d(col g+8)
// Padding columns (n >= N) and K positions (k >= K) have zero codes and zero
// scales, so they contribute exactly 0.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/lbv.h"

namespace lbv {

struct FmtInfo {
    int chunk_k;      // K per chunk
    int kt;           // k-tiles (16 K) per chunk
    int code_bits;    // bits per code
    int slots;        // slots per 32-bit word
    int group_k;      // K per scale group
    int groups;       // scale groups per chunk
    int side_bytes;   // side bytes per (tile, chunk, g)
};

inline bool fmt_info(lbv_format fmt, int group, FmtInfo* fi)
{
    switch (fmt) {
    case LBV_FMT_SIGN1_G128:
        *fi = {256, 16, 1, 16, 128, 2, 8};
        return true;
    case LBV_FMT_AFFINE2:
        if (group != 32 && group != 64 && group != 128)
            return false;
        *fi = {128, 8, 2, 8, group, 128 / group, (128 / group) * 8};
        return true;
    case LBV_FMT_Q4_0:
        *fi = {64, 4, 4, 4, 32, 2, 8};
        return true;
    }
    return false;
}

struct Layout {
    int64_t ntiles;        // ceil(N / 16)
    int64_t nchunks;       // ceil(K / chunk_k)
    size_t rec_bytes;      // 512 + 8 * side_bytes
    size_t total;          // ntiles * nchunks * rec_bytes
};

inline Layout make_layout(const FmtInfo& fi, int K, int N)
{
    Layout L;
    L.ntiles = (N + 15) / 16;
    L.nchunks = (K + fi.chunk_k - 1) / fi.chunk_k;
    L.rec_bytes = 512u + 8u * (size_t)fi.side_bytes;
    L.total = (size_t)L.ntiles * (size_t)L.nchunks * L.rec_bytes;
    return L;
}

}  // namespace lbv
