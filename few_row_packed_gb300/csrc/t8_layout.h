// t8_layout.h -- the record layout read by the e4m3 tensor-memory kernel
// (plans created with LBV_PLAN_TC_E4M3), shared by its host packer
// (t8_api.cpp) and its kernels.  Lossless: the same bits as the canonical file
// layout, rearranged so that one thread owns one output column and turns a
// group's codes into e4m3 bytes with one LOP3 per four weights.
//
// Terms
//   tile     128 output columns n = 128*tile .. 128*tile+127: the M side of
//            one tcgen05 MMA (the <= 8 activation rows are its N side).
//   quarter  32 columns 32q .. 32q+31 of a tile: the columns of one decode
//            warp (it owns tensor-memory lanes 32q .. 32q+31).
//   group    128 consecutive K values: one scale group of the g128 formats
//            and one A slot of the kernel (32 tensor-memory columns of four
//            e4m3 values each).
//
// Records: one record of REC = 32 * (CB + SB) bytes per (tile, group,
// quarter), in the order ((tile * ngroups + group) * 4 + quarter), so the
// four quarters of a group, and consecutive groups of a tile, are contiguous:
//   codes: [CB / 16][32 columns][16 bytes].  The CB bytes of a column are
//          CB / 4 little-endian words:
//            affine2 (W = 2, CB = 32): word i holds k = 16i + 4j + b
//              (j, b = 0..3) at bits 8b + 2j .. 8b + 2j + 1;
//            sign1 (W = 1, CB = 16): word i holds k = 32i + 4j + b
//              (j = 0..7, b = 0..3) at bit 8b + j.
//          So (word >> 4s) & (mask << f) with mask = 0x01010101 * (2^W - 1)
//          puts four codes in the low bits of four bytes, shifted left by f:
//          e4m3 subnormals (and, past 7, the normals that continue them)
//          worth code * 2^(f - 9), exactly.
//   side:  [32 columns][SB bytes] of fp16 bit patterns: sign1 the scale
//          (SB = 2); affine2 scale then bias (SB = 4).
// Padding columns (n >= N) and groups past K have zero codes and zero
// scales (and biases), so they contribute exactly 0.
#pragma once

#include <stddef.h>
#include <stdint.h>

#include "../../include/lbv.h"

namespace lbv {

constexpr int kT8TileN = 128;
constexpr int kT8GroupK = 128;

struct T8FmtInfo {
    int code_bytes;   // CB: code bytes per column and group
    int side_bytes;   // SB: side bytes per column and group
    int code_bits;    // W
};

// Formats the kernel reads: 1-bit sign g128 and 2-bit affine g128.
inline bool t8_fmt_info(lbv_format fmt, int group, T8FmtInfo* fi)
{
    if (fmt == LBV_FMT_SIGN1_G128) {
        *fi = {16, 2, 1};
        return true;
    }
    if (fmt == LBV_FMT_AFFINE2 && group == 128) {
        *fi = {32, 4, 2};
        return true;
    }
    return false;
}

struct T8Layout {
    int64_t ntiles;        // ceil(N / 128)
    int64_t ngroups;       // K / 128
    size_t rec_bytes;      // 32 * (CB + SB)
    size_t total;          // ntiles * 4 * ngroups * rec_bytes
};

inline T8Layout t8_make_layout(const T8FmtInfo& fi, int K, int N)
{
    T8Layout L;
    L.ntiles = (N + kT8TileN - 1) / kT8TileN;
    L.ngroups = (K + kT8GroupK - 1) / kT8GroupK;
    L.rec_bytes = (size_t)32 * (size_t)(fi.code_bytes + fi.side_bytes);
    L.total = (size_t)L.ntiles * 4 * (size_t)L.ngroups * L.rec_bytes;
    return L;
}

// Bit position of the code of group-local k inside its word, and the word.
inline void t8_code_pos(int code_bits, int k, int* word, int* bit)
{
    if (code_bits == 2) {
        const int kk = k % 16;
        *word = k / 16;
        *bit = 8 * (kk % 4) + 2 * (kk / 4);
    } else {
        const int kk = k % 32;
        *word = k / 32;
        *bit = 8 * (kk % 4) + (kk / 4);
    }
}

// Launch shape of the e4m3 tensor-memory kernel.
struct T8Shape {
    int splits;             // K slices (cluster size): 1, 2, 4 or 8
    int ctas_n;             // clusters along N (grid y); each owns a contiguous tile range
    int gps;                // groups per slice (the last slice may be shorter)
    int tpc;                // most tiles of one cluster
    int owned;              // most tiles of a cluster one rank owns (tile i: rank i % splits)
    int x_in_ring;          // 1: X is staged in the ring stages issued after the prologue
    size_t smem;            // dynamic shared memory bytes
};

}  // namespace lbv
