// verify_kernel.cuh -- the few-row verify kernel, Y[M,N] = X[M,K] . W[K,N],
// M <= 8, for the packed formats of layout.h.
//
// Design (GB300, sm_103a):
//   * Persistent grid of thread-block clusters.  Cluster y owns a contiguous,
//     balanced range of 16-column tiles; the S CTAs of a cluster split K into
//     slices, and their partial sums are reduced through distributed shared
//     memory in rank order (deterministic, no workspace).
//   * Each CTA stages its K slice of X once, row-major, with one 1-D bulk copy
//     per row (padded rows, so ldmatrix reads the B fragments without bank
//     conflicts), then computes the per-group corrections (below).  X is read
//     only after griddepcontrol.wait; the packed weights, which no kernel
//     writes, start streaming before it.
//   * Each warp streams its tiles' packed codes and scales through a private
//     ring of shared-memory stages filled by 1-D bulk async copies (TMA engine)
//     and tracked by mbarriers, so 75-110 KB per SM stay in flight with no
//     registers held; a stage carries two to four chunks of each tile.  Every
//     wait is bounded; a wait that gives up sets the plan's status word and
//     the warp stops.
//   * Decode is one LOP3 per A-fragment register: (word_variant & mask) ^ base
//     places a code in the mantissa/exponent field of an fp16 or bf16 whose
//     value is  code_value + c  for a small integer c fixed by the bit position
//     (the "codes turned into exact halves with 0x6400 less 1024" idea of the
//     Ishizuki README credits, extended to every position of the word); 1-3
//     shifts per 32-bit word bring the remaining positions into place.
//   * mma.sync m16n8k16 (fp16 or bf16 in, fp32 accumulate): 16 weight columns
//     are the M side and the M <= 8 activation rows the N side (rows >= M are
//     zero), so each decoded weight meets every drafted row at once (Ishizuki
//     README, "Kernels written for the verify").  The k-tiles of a chunk are
//     visited alternately from its two halves (two interleaved accumulator
//     chains for groups of 64 or fewer), and each tile of a unit has its own.
//   * The offsets c enter each group's accumulator as its initial value
//     -sum_k c_k x_k, computed once per CTA from the staged activations on the
//     tensor cores (the "row-sum prep" of the dflash-mlx-bonsai2 README); the
//     group scale (and bias * row sum for affine) is applied in fp32 once per
//     group, so every tensor-core operand is an exact small integer.
#pragma once

#include <cooperative_groups.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include <utility>

#include "lbv_internal.h"

namespace lbv {

namespace cg = cooperative_groups;

template <int FMT, int GROUP>
struct Traits;

template <>
struct Traits<LBV_FMT_SIGN1_G128, 128> {
    static constexpr int CHUNK_K = 256, KT = 16, W = 1, GPC = 2, KTG = 8, SIDE_W = 2;
    static constexpr bool AFFINE = false;
};
template <int G>
struct Traits<LBV_FMT_AFFINE2, G> {
    static constexpr int CHUNK_K = 128, KT = 8, W = 2, GPC = 128 / G, KTG = G / 16,
                         SIDE_W = 2 * (128 / G);
    static constexpr bool AFFINE = true;
};
template <>
struct Traits<LBV_FMT_Q4_0, 32> {
    static constexpr int CHUNK_K = 64, KT = 4, W = 4, GPC = 2, KTG = 2, SIDE_W = 2;
    static constexpr bool AFFINE = false;
};

// ---------------------------------------------------------------------------
// Decode specification of slot s of a word: shift the word (positive = left),
// then keep the W-bit field at `target` (and target + 16) and XOR `base`.
// The resulting fp16/bf16 value is  code_value + c.
struct DecSpec {
    int shift;
    int target;
    uint32_t base;   // 16-bit pattern, replicated into both halves
    int c;
    int bid;         // index of `base` among the format's distinct bases
};

// 1-bit sign: value = w + c with w = +-1 (bit 1 -> +1).
//   fp16 targets: 15 (base -1.0, c 0), 14 (0, 1), 10 (2.0, 3), 9..5 (2^(11-j), 2^(11-j)+1)
//   bf16 targets: 15 (-1.0, 0), 14 (0, 1), 7 (2.0, 3), 6..2 (2^(8-j), 2^(8-j)+1)
__host__ __device__ constexpr DecSpec sign1_spec(int xt, int s)
{
    if (xt == LBV_F16) {
        // two shifts per word: slots 0-4 -> 5-9 (left 5), 11-13 -> 8-10 (right 3)
        const int sh = (s <= 4) ? 5 : (s >= 11 && s <= 13) ? -3 : 0;
        const int j = s + sh;
        return j == 15   ? DecSpec{sh, j, 0xBC00u, 0, 0}
               : j == 14 ? DecSpec{sh, j, 0x0000u, 1, 1}
               : j == 10 ? DecSpec{sh, j, 0x4000u, 3, 2}
               : j == 9  ? DecSpec{sh, j, 0x4400u, 5, 3}
               : j == 8  ? DecSpec{sh, j, 0x4800u, 9, 4}
               : j == 7  ? DecSpec{sh, j, 0x4C00u, 17, 5}
               : j == 6  ? DecSpec{sh, j, 0x5000u, 33, 6}
                         : DecSpec{sh, j, 0x5400u, 65, 7};   // j == 5
    } else {
        const int sh = (s <= 1) ? 5 : (s >= 8 && s <= 13) ? -6 : 0;
        const int j = s + sh;
        return j == 15   ? DecSpec{sh, j, 0xBF80u, 0, 0}
               : j == 14 ? DecSpec{sh, j, 0x0000u, 1, 1}
               : j == 7  ? DecSpec{sh, j, 0x4000u, 3, 2}
               : j == 6  ? DecSpec{sh, j, 0x4080u, 5, 3}
               : j == 5  ? DecSpec{sh, j, 0x4100u, 9, 4}
               : j == 4  ? DecSpec{sh, j, 0x4180u, 17, 5}
               : j == 3  ? DecSpec{sh, j, 0x4200u, 33, 6}
                         : DecSpec{sh, j, 0x4280u, 65, 7};   // j == 2
    }
}

// 2-bit affine code q at bits 2s: value = q + c.  A field at mantissa bit j
// under a base of 2^(m - j) (m = 10 for fp16, 7 for bf16) reads as q + base.
//   fp16: targets 0, 2, 4, 6, 8 (bases 1024, 256, 64, 16, 4): slots 0-4 in
//         place, slots 5-7 shifted right by 6 onto 4, 6, 8
//   bf16: targets 0, 2, 4 (bases 128, 32, 8): slots 0-2 in place, slots 3-5
//         shifted right by 6 and slots 6-7 by 12 onto them
// (one shifted copy of a word for fp16, two for bf16)
__host__ __device__ constexpr DecSpec affine2_spec(int xt, int s)
{
    if (xt == LBV_F16) {
        const int sh = (s <= 4) ? 0 : -6;
        const int j = 2 * s + sh;
        return j == 0   ? DecSpec{sh, j, 0x6400u, 1024, 0}
               : j == 2 ? DecSpec{sh, j, 0x5C00u, 256, 1}
               : j == 4 ? DecSpec{sh, j, 0x5400u, 64, 2}
               : j == 6 ? DecSpec{sh, j, 0x4C00u, 16, 3}
                        : DecSpec{sh, j, 0x4400u, 4, 4};     // j == 8
    } else {
        const int sh = (s <= 2) ? 0 : (s <= 5) ? -6 : -12;
        const int j = 2 * s + sh;
        return j == 0   ? DecSpec{sh, j, 0x4300u, 128, 0}
               : j == 2 ? DecSpec{sh, j, 0x4200u, 32, 1}
                        : DecSpec{sh, j, 0x4100u, 8, 2};     // j == 4
    }
}

// Q4_0 nibble q at bits 4s: value = q + c.
//   fp16: targets 0 (base 1024) and 4 (base 64): slots 0-1 in place, slots
//         2-3 shifted right by 8 onto them (one shifted copy of a word)
//   bf16: target 0 (base 128): slot s shifted right by 4s
__host__ __device__ constexpr DecSpec q4_0_spec(int xt, int s)
{
    if (xt == LBV_F16) {
        const int sh = s <= 1 ? 0 : -8;
        return 4 * s + sh == 0 ? DecSpec{sh, 0, 0x6400u, 1024, 0}
                               : DecSpec{sh, 4, 0x5400u, 64, 1};
    }
    return DecSpec{-4 * s, 0, 0x4300u, 128, 0};
}

template <int FMT>
__host__ __device__ constexpr DecSpec dec_spec(int xt, int s)
{
    return FMT == LBV_FMT_SIGN1_G128 ? sign1_spec(xt, s)
           : FMT == LBV_FMT_AFFINE2  ? affine2_spec(xt, s)
                                     : q4_0_spec(xt, s);
}

// Value of a 16-bit fp16 / bf16 pattern (finite), for the compile-time check
// below.
__host__ __device__ constexpr double half_bits_value(int xt, uint32_t h)
{
    const int mbits = xt == LBV_F16 ? 10 : 7, ebits = xt == LBV_F16 ? 5 : 8;
    const int bias = (1 << (ebits - 1)) - 1;
    const uint32_t mant = h & ((1u << mbits) - 1u);
    const int e = (int)((h >> mbits) & ((1u << ebits) - 1u));
    double v = e ? (double)((1u << mbits) + mant) : (double)mant;
    int p = (e ? e : 1) - bias - mbits;
    for (; p > 0; --p)
        v *= 2.0;
    for (; p < 0; ++p)
        v *= 0.5;
    return (h >> 15) ? -v : v;
}

// Distinct XOR bases of a format and activation dtype (kept in registers:
// one LOP3 per decode).
template <int FMT, int XT>
__host__ __device__ constexpr int num_bases()
{
    return FMT == LBV_FMT_SIGN1_G128 ? 8
           : FMT == LBV_FMT_AFFINE2  ? (XT == LBV_F16 ? 5 : 3)
                                     : (XT == LBV_F16 ? 2 : 1);
}

template <int FMT>
__host__ __device__ constexpr uint32_t base_of(int xt, int bid)
{
    uint32_t b = 0;
    for (int s = 0; s < 16; ++s)
        if (dec_spec<FMT>(xt, s).bid == bid)
            b = dec_spec<FMT>(xt, s).base;
    return b | (b << 16);
}

template <int FMT, int XT, int S>
__device__ __forceinline__ uint32_t decode(uint32_t w, const uint32_t (&bases)[num_bases<FMT, XT>()])
{
    constexpr DecSpec d = dec_spec<FMT>(XT, S);
    constexpr int W = Traits<FMT, FMT == LBV_FMT_SIGN1_G128 ? 128 : FMT == LBV_FMT_Q4_0 ? 32 : 64>::W;
    constexpr uint32_t field = (1u << W) - 1u;
    constexpr uint32_t mask = (field << d.target) | (field << (d.target + 16));
    constexpr int shl = d.shift > 0 ? (d.shift > 31 ? 31 : d.shift) : 0;
    constexpr int shr = d.shift < 0 ? (-d.shift > 31 ? 31 : -d.shift) : 0;
    const uint32_t v = shl ? (w << shl) : shr ? (w >> shr) : w;
    // (v & mask) ^ base as one LOP3 with an immediate mask: written in C, the
    // compiler splits it into two logic operations.
    uint32_t r;
    asm("lop3.b32 %0, %1, %2, %3, 0x6A;\n" : "=r"(r) : "r"(v), "n"(mask), "r"(bases[d.bid]));
    return r;
}


// Every slot of every decode table, emulated for every code value in both
// halves of a word: shift, mask, XOR with the slot's base must read as
// value + c (value = +-1 for a sign bit, q for 2- and 4-bit codes).
template <int FMT, int XT>
__host__ __device__ constexpr bool decode_tables_ok()
{
    constexpr int W = FMT == LBV_FMT_SIGN1_G128 ? 1 : FMT == LBV_FMT_AFFINE2 ? 2 : 4;
    constexpr int slots = 16 / W;
    for (int s = 0; s < slots; ++s) {
        const DecSpec d = dec_spec<FMT>(XT, s);
        const uint32_t field = (1u << W) - 1u;
        const uint32_t mask = (field << d.target) | (field << (d.target + 16));
        uint32_t base = 0;
        for (int i = 0; i < 16; ++i)
            if (dec_spec<FMT>(XT, i).bid == d.bid)
                base = dec_spec<FMT>(XT, i).base;
        if (base != d.base || d.bid >= num_bases<FMT, XT>())
            return false;
        for (uint32_t q = 0; q <= field; ++q) {
            const uint32_t w = (q << (W * s)) | (q << (16 + W * s));
            const uint32_t v = d.shift > 0 ? w << d.shift : d.shift < 0 ? w >> -d.shift : w;
            const uint32_t r = (v & mask) ^ (base | (base << 16));
            const double want = (FMT == LBV_FMT_SIGN1_G128 ? (q ? 1.0 : -1.0) : (double)q) + d.c;
            if (half_bits_value(XT, r & 0xFFFFu) != want || half_bits_value(XT, r >> 16) != want)
                return false;
        }
    }
    return true;
}

static_assert(decode_tables_ok<LBV_FMT_SIGN1_G128, LBV_F16>() &&
                  decode_tables_ok<LBV_FMT_SIGN1_G128, LBV_BF16>() &&
                  decode_tables_ok<LBV_FMT_AFFINE2, LBV_F16>() &&
                  decode_tables_ok<LBV_FMT_AFFINE2, LBV_BF16>() &&
                  decode_tables_ok<LBV_FMT_Q4_0, LBV_F16>() &&
                  decode_tables_ok<LBV_FMT_Q4_0, LBV_BF16>(),
              "a decode table slot does not read as value + c");

// ---------------------------------------------------------------------------
// Device helpers

template <int XT>
__device__ __forceinline__ void mma16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                         uint32_t a3, uint32_t b0, uint32_t b1)
{
    if constexpr (XT == LBV_F16) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%0,%1,%2,%3};\n"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
}

// D = A.B + C with C in other registers (starts an accumulator chain from
// initial values without moving them into D first; c is the C fragment as
// one register quad).
template <int XT>
__device__ __forceinline__ void mma16816_c(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                           uint32_t a3, uint32_t b0, uint32_t b1, float4 c)
{
    if constexpr (XT == LBV_F16) {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y),
              "f"(c.z), "f"(c.w));
    } else {
        asm("mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 {%0,%1,%2,%3}, "
            "{%4,%5,%6,%7}, {%8,%9}, {%10,%11,%12,%13};\n"
            : "=f"(d[0]), "=f"(d[1]), "=f"(d[2]), "=f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1), "f"(c.x), "f"(c.y),
              "f"(c.z), "f"(c.w));
    }
}

__device__ __forceinline__ void griddep_wait()
{
    asm volatile("griddepcontrol.wait;\n" ::: "memory");
}

__device__ __forceinline__ void griddep_launch_dependents()
{
    asm volatile("griddepcontrol.launch_dependents;\n" ::: "memory");
}

__device__ __forceinline__ uint32_t smem_u32(const void* p)
{
    return (uint32_t)__cvta_generic_to_shared(p);
}

// Four 8x8 b16 matrices from shared memory (row addresses from lanes 8i..8i+7
// for matrix i): thread (g, t) receives row g, elements 2t and 2t + 1 of each.
__device__ __forceinline__ uint4 ldsm_x4(uint32_t addr)
{
    uint4 r;
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0,%1,%2,%3}, [%4];\n"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "r"(addr));
    return r;
}

__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;\n" ::"r"(bar), "r"(count) : "memory");
}

__device__ __forceinline__ void mbar_init_fence()
{
    asm volatile("fence.mbarrier_init.release.cluster;\n" ::: "memory");
}

__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n" ::"r"(bar), "r"(bytes)
                 : "memory");
}

// 1-D bulk copy global -> this CTA's shared memory, completion on `bar`.
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes,
                                         uint32_t bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];\n"
        ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
        : "memory");
}

// Cluster barrier halves: every CTA arrives once it runs; waiting on that
// phase guarantees all peers have started before their shared memory is
// written.
__device__ __forceinline__ void cluster_arrive_relaxed()
{
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void cluster_wait()
{
    asm volatile("barrier.cluster.wait.aligned;\n" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;\n" ::: "memory");
}

// Single-lane issue without divergence: the operation runs only where
// `pred` is nonzero.
__device__ __forceinline__ void mbar_expect_tx_if(uint32_t pred, uint32_t bar, uint32_t bytes)
{
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n"
                 " @q mbarrier.arrive.expect_tx.shared::cta.b64 _, [%1], %2;\n}\n"
                 ::"r"(pred), "r"(bar), "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ void bulk_g2s_if(uint32_t pred, uint32_t dst, const void* src,
                                            uint32_t bytes, uint32_t bar)
{
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n"
                 " @q cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes"
                 " [%1], [%2], %3, [%4];\n}\n"
                 ::"r"(pred), "r"(dst), "l"(src), "r"(bytes), "r"(bar)
                 : "memory");
}

__device__ __forceinline__ void fence_proxy_async_if(uint32_t pred)
{
    asm volatile("{\n .reg .pred q;\n setp.ne.u32 q, %0, 0;\n"
                 " @q fence.proxy.async.shared::cta;\n}\n" ::"r"(pred)
                 : "memory");
}

// One try of an mbarrier phase wait (true if the phase has completed).
__device__ __forceinline__ bool mbar_try(uint32_t bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
        " selp.u32 %0, 1, 0, p;\n}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of an mbarrier.  Returns false if it did
// not complete within `limit` tries: by default (2^20 tries, sleeping 1 us
// between tries after the first 4096) roughly a second.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity,
                                          uint32_t limit = 1u << 20)
{
    constexpr uint32_t kSpin = 1u << 12;
    for (uint32_t i = 0; i < limit; ++i) {
        uint32_t ok;
        asm volatile(
            "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n"
            " selp.u32 %0, 1, 0, p;\n}\n"
            : "=r"(ok)
            : "r"(bar), "r"(parity)
            : "memory");
        if (ok)
            return true;
        if (i >= kSpin)
            __nanosleep(1000);
    }
    return false;
}

template <int XT>
__device__ __forceinline__ float2 pair_to_float2(uint32_t v)
{
    if constexpr (XT == LBV_F16) {
        __half2 h = *reinterpret_cast<__half2*>(&v);
        return __half22float2(h);
    } else {
        __nv_bfloat162 h = *reinterpret_cast<__nv_bfloat162*>(&v);
        return __bfloat1622float2(h);
    }
}

__device__ __forceinline__ float2 f16pair(uint32_t v)
{
    __half2 h = *reinterpret_cast<__half2*>(&v);
    return __half22float2(h);
}

// Two fp32 values rounded to nearest even in the X dtype, packed (lo in the
// low half).
template <int XT>
__device__ __forceinline__ uint32_t round_x2(float lo, float hi)
{
    if constexpr (XT == LBV_F16) {
        const __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    } else {
        const __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
}

// Four 8x8 b16 matrices to shared memory, transposed: thread (g, t) gives row
// g, columns 2t and 2t + 1 of matrix i in register i; lanes 8i..8i+7 give the
// addresses of the 8 stored rows of matrix i (its columns).
__device__ __forceinline__ void stsm_x4_trans(uint32_t addr, uint32_t r0, uint32_t r1, uint32_t r2,
                                              uint32_t r3)
{
    asm volatile("stmatrix.sync.aligned.m8n8.x4.trans.shared.b16 [%0], {%1, %2, %3, %4};\n"
                 ::"r"(addr), "r"(r0), "r"(r1), "r"(r2), "r"(r3)
                 : "memory");
}

// Two entries (i, j), (i, j + 1) of the 16-point Sylvester Hadamard matrix,
// H16[i][j] = (-1)^popcount(i & j), as a packed pair of the X dtype.
template <int XT>
__device__ __forceinline__ uint32_t h16_pair(int i, int j)
{
    constexpr uint32_t one = XT == LBV_F16 ? 0x3C00u : 0x3F80u;   // +1.0
    const uint32_t lo = one | ((uint32_t)(__popc(i & j) & 1) << 15);
    const uint32_t hi = one | ((uint32_t)(__popc(i & (j + 1)) & 1) << 15);
    return lo | (hi << 16);
}

// Argmax key of (logit v, column n): keys compare like the logits, and among
// equal logits the smaller column has the larger key.  -0 counts as +0, any
// NaN ranks above every number (the first NaN wins), and no key is 0, so 0
// stands for "no column yet".
__device__ __forceinline__ unsigned long long amax_key(float v, int n)
{
    uint32_t u = __float_as_uint(v);
    if ((u << 1) == 0u)
        u = 0u;
    u = (u & 0x80000000u) ? ~u : (u | 0x80000000u);
    if (v != v)
        u = 0xffffffffu;
    return ((unsigned long long)u << 32) | (unsigned long long)(0xffffffffu - (uint32_t)n);
}

__device__ __forceinline__ float amax_key_value(unsigned long long k)
{
    const uint32_t u = (uint32_t)(k >> 32);
    return __uint_as_float((u & 0x80000000u) ? (u & 0x7fffffffu) : ~u);
}

// Largest key among the 8 lanes of a warp that share lane & 3 (the lanes
// holding the same rows of an m16n8 accumulator).
__device__ __forceinline__ unsigned long long warp_max_key(unsigned long long k)
{
#pragma unroll
    for (int s = 4; s <= 16; s <<= 1) {
        const unsigned long long o = __shfl_xor_sync(0xffffffffu, k, s);
        k = o > k ? o : k;
    }
    return k;
}

// ---------------------------------------------------------------------------
// Fused head prologue, on X rows staged row-major in shared memory (row m at
// xs + m * RS bytes, RS % 16 == 0, RS / 4 = 4 mod 8 for conflict-free rows).

// ldmatrix row address of this lane within the X rows: lanes 8i..8i+7 give the
// rows of matrix i, which covers K elements 8i..8i+7 of a 32-element span.
__device__ __forceinline__ uint32_t ldsm_lane_offset(int RS, int lane)
{
    return (uint32_t)((lane & 7) * RS + (lane >> 3) * 16);
}

// Flips the sign of X[m][k] (rows m < M, k < have; have % 32 == 0) where bit
// kb + k of `signs` is set.  Threads tid = 0, nthreads, ... share the work.
__device__ __forceinline__ void flip_signs(const uint32_t* signs, unsigned char* xs, int RS, int M,
                                           int kb, int have, int tid, int nthreads)
{
    const int words = have / 32;                       // mask words per row
    for (int i = tid; i < M * words; i += nthreads) {
        const int m = i / words, wi = i - m * words;
        const uint32_t sg = signs[(kb >> 5) + wi];
        uint32_t* e = reinterpret_cast<uint32_t*>(xs + (size_t)m * RS + wi * 64);
#pragma unroll
        for (int j = 0; j < 16; ++j)
            e[j] ^= (((sg >> (2 * j)) & 1u) << 15) | (((sg >> (2 * j + 1)) & 1u) << 31);
    }
}

// Rotates blocks 0..nblk-1 of the 8 staged rows in place (warps warp,
// warp + nwarps, ... take one block each in turn):
//   x'_b = H128 x_b / sqrt(128),  H[i][j] = (-1)^popcount(i & j)  (Sylvester).
// H128 = H8 (x) H16, so with the block split into sub-blocks J of 16 elements
//   U_J = H16 x_J                  one m16n8k16 MMA per sub-block: H16 is the A
//                                  operand, the sub-block's X fragment (as the
//                                  verify main loop reads it) is B;
//   x'_(16 I + i) = sum_J H8[I][J] U_J[i]   an 8-point butterfly across the
//                                  eight accumulators each lane holds.
// fp32 sums, one multiplication by the fp32 value of 1/sqrt(128), one rounding
// to the X dtype.  A warp reads its whole block before writing it back.  All 8
// rows are rotated; a row's results depend on that row alone.
template <int XT>
__device__ __forceinline__ void rotate_x(uint32_t xs_a, int RS, int nblk, int warp, int nwarps,
                                         int lane)
{
    const int g = lane >> 2, t = lane & 3;
    const uint32_t h0 = h16_pair<XT>(g, 2 * t), h1 = h16_pair<XT>(g + 8, 2 * t);
    const uint32_t h2 = h16_pair<XT>(g, 2 * t + 8), h3 = h16_pair<XT>(g + 8, 2 * t + 8);
    const uint32_t xa = xs_a + ldsm_lane_offset(RS, lane);
    constexpr float kInvSqrt128 = 0.08838834764831845f;
#pragma unroll 1
    for (int b = warp; b < nblk; b += nwarps) {
        float u[8][4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
            const uint4 r = ldsm_x4(xa + b * 256 + q * 64);     // sub-blocks 2q, 2q + 1
#pragma unroll
            for (int e = 0; e < 4; ++e)
                u[2 * q][e] = u[2 * q + 1][e] = 0.f;
            mma16816<XT>(u[2 * q], h0, h1, h2, h3, r.x, r.y);
            mma16816<XT>(u[2 * q + 1], h0, h1, h2, h3, r.z, r.w);
        }
#pragma unroll
        for (int h = 1; h < 8; h <<= 1)
#pragma unroll
            for (int J = 0; J < 8; ++J)
                if (!(J & h))
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                        const float a = u[J][e], c = u[J + h][e];
                        u[J][e] = a + c;
                        u[J + h][e] = a - c;
                    }
        // u[I][e] is element 16 I + g + 8 (e >> 1) of row 2 t + (e & 1): per I
        // two 8x8 matrices (elements 16 I + 0..7 and + 8..15 by rows), whose
        // transposes are the rows' elements, written with stmatrix .trans.
        // Lane 8j + r gives row r's address in matrix j of each store.
        const int mj = lane >> 3, mr = lane & 7;
#pragma unroll
        for (int k = 0; k < 4; ++k) {                    // tiles I = 2k, 2k + 1
            const int I = 2 * k + (mj >> 1), half = mj & 1;
            const uint32_t addr = xs_a + (uint32_t)(mr * RS + (b * 128 + 16 * I + 8 * half) * 2);
            stsm_x4_trans(addr,
                          round_x2<XT>(u[2 * k][0] * kInvSqrt128, u[2 * k][1] * kInvSqrt128),
                          round_x2<XT>(u[2 * k][2] * kInvSqrt128, u[2 * k][3] * kInvSqrt128),
                          round_x2<XT>(u[2 * k + 1][0] * kInvSqrt128, u[2 * k + 1][1] * kInvSqrt128),
                          round_x2<XT>(u[2 * k + 1][2] * kInvSqrt128, u[2 * k + 1][3] * kInvSqrt128));
        }
    }
}

// ---------------------------------------------------------------------------
// Chunks of each tile per ring stage.  A stage's fixed work (the barrier
// wait, the copy issue, the cursor) is spread over TPW * STAGE_CHUNKS * KT
// MMAs: three chunks per stage with two-tile units (rings of ~110 KB; two
// where a record has more than four side words, whose registers would
// spill), four with one-tile units (~80 KB), two with four-tile units.
template <int FMT, int GROUP, int TPW>
__host__ __device__ constexpr int stage_chunks()
{
    return TPW == 1 ? 4 : (TPW == 2 && Traits<FMT, GROUP>::SIDE_W <= 4) ? 3 : 2;
}

// Compile-time geometry of one (format, group, warps, tiles per warp, chunks
// per stage) kernel.
template <int FMT, int GROUP, int NW, int TPW, int STAGE_CHUNKS>
struct Geometry {
    using T = Traits<FMT, GROUP>;
    static constexpr int SIDE_B = T::SIDE_W * 4;              // side bytes per (record, g)
    static constexpr int REC = 512 + 8 * SIDE_B;              // record bytes (tile, chunk)
    static_assert(REC % 16 == 0 && (SIDE_B == 8 || SIDE_B % 16 == 0),
                  "records and side words stay aligned for 8/16-byte shared loads");
    static constexpr int CPS = STAGE_CHUNKS;                  // chunks per ring stage
    static constexpr int SLOT_B = TPW * CPS * REC;            // one ring stage
    static constexpr int STAGES_RAW = 98304 / (NW * SLOT_B);
    static constexpr int STAGES = STAGES_RAW < 2 ? 2 : STAGES_RAW > 8 ? 8 : STAGES_RAW;
    static constexpr size_t RING_B = (size_t)NW * STAGES * SLOT_B;
    // + the X barrier and a flag word (16), the CTA's argmax keys of the fused
    // head (64)
    static constexpr size_t BAR_B = (size_t)NW * STAGES * 8 + 16 + 64;
};

// Bytes between X rows in shared memory: the slice plus 16 bytes, so the 8
// row addresses of an ldmatrix hit distinct bank groups.
template <int FMT, int GROUP>
__host__ __device__ constexpr int x_row_stride(int cps)
{
    return cps * Traits<FMT, GROUP>::CHUNK_K * 2 + 16;
}

// Shared memory carve-up (bytes):
//   ring | mbarriers (+ X barrier, flag, argmax keys) | xs (X rows) | corr |
//   rsum (affine) | part (K split)
template <int FMT, int GROUP, int NW, int TPW, int STAGE_CHUNKS>
__host__ __device__ inline size_t smem_bytes_for(int cps, int tiles_max, int splits)
{
    using G = Geometry<FMT, GROUP, NW, TPW, STAGE_CHUNKS>;
    using T = Traits<FMT, GROUP>;
    size_t b = G::RING_B + G::BAR_B;
    b += 8 * x_row_stride<FMT, GROUP>(cps);
    b += (size_t)cps * T::GPC * 16 * 4;                       // corrections (C quads)
    if (T::AFFINE)
        b += (size_t)cps * T::GPC * 8 * 4;                    // row sums
    if (splits > 1)
        b += (size_t)((tiles_max + splits - 1) / splits) * splits * 512u;
    return b;
}

// ---------------------------------------------------------------------------

template <int FMT, int XT, int GROUP, int NW, int TPW, int STAGE_CHUNKS>
struct VerifyKernel {
    using T = Traits<FMT, GROUP>;
    using G = Geometry<FMT, GROUP, NW, TPW, STAGE_CHUNKS>;
    static constexpr int STAGES = G::STAGES;
    static constexpr int NSET = T::GPC;                     // accumulator chains per tile

    // Load cursor of a warp: the record of its next (unit, stage), tracked
    // incrementally by every lane; lane 0 issues.  A stage holds up to CPS
    // consecutive chunks of each of the unit's tiles.
    struct Cursor {
        const uint8_t* rec;     // record (tile0, first chunk of the stage)
        int nvalid;             // tiles of the unit inside the cluster range
        int nc;                 // chunks in this stage
        int unit, stage;
    };

    static __device__ __forceinline__ void cursor_set(const VerifyParams& p, int t0, int t1,
                                                      int c0, int nch, Cursor& c)
    {
        const int tile0 = t0 + c.unit * TPW;
        const int ch = c.stage * G::CPS;
        c.rec = p.W + ((size_t)tile0 * p.nchunks + c0 + ch) * G::REC;
        c.nvalid = min(TPW, t1 - tile0);
        c.nc = min(G::CPS, nch - ch);
    }

    // Next stage: within a unit the record pointer just moves on by a
    // stage's chunks; only a new unit recomputes it.
    static __device__ __forceinline__ void cursor_next(const VerifyParams& p, int t0, int t1,
                                                       int c0, int nch, int nstage, Cursor& c)
    {
        if (++c.stage == nstage) {
            c.stage = 0;
            c.unit += NW;
            cursor_set(p, t0, t1, c0, nch, c);
        } else {
            c.rec += G::CPS * G::REC;
            c.nc = min(G::CPS, nch - c.stage * G::CPS);
        }
    }

    // tstride: bytes between the records of consecutive tiles (nchunks * REC).
    // leader = 0 issues nothing (the lanes that do not issue, and the stage a
    // wait-limit test leaves out).
    static __device__ __forceinline__ void issue(const Cursor& c, size_t tstride,
                                                 uint32_t leader, uint32_t ring_w,
                                                 uint32_t bars_w, int slot)
    {
        const uint32_t bar = bars_w + slot * 8;
        const uint32_t dst = ring_w + slot * G::SLOT_B;
        const uint32_t bytes = (uint32_t)c.nc * G::REC;
        mbar_expect_tx_if(leader, bar, (uint32_t)c.nvalid * bytes);
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl)
            bulk_g2s_if(leader && tl < c.nvalid, dst + tl * G::CPS * G::REC,
                        c.rec + tl * tstride, bytes, bar);
    }

    static constexpr int NB = num_bases<FMT, XT>();

    // One k-tile of every tile of the unit into the chain of its group.  The
    // chains run in the order the k-tile pairs are visited (0, KT/2, 1, ...),
    // so a group's lowest k-tile comes first and starts its chain from the
    // group's correction (init) instead of from zero.
    template <int HALF, int KTL>
    static __device__ __forceinline__ void ktile(const uint4 (&w)[TPW], uint32_t b0, uint32_t b1,
                                                 const uint32_t (&bases)[NB],
                                                 const float4 (&init)[NSET],
                                                 float (&acc)[TPW][NSET][4])
    {
        constexpr int kt = HALF * (T::KT / 2) + KTL;
        constexpr int set = kt / T::KTG;
        constexpr bool first = kt % T::KTG == 0;
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl) {
            const uint32_t wa = HALF ? w[tl].z : w[tl].x;
            const uint32_t wb = HALF ? w[tl].w : w[tl].y;
            const uint32_t a0 = decode<FMT, XT, 2 * KTL>(wa, bases);
            const uint32_t a1 = decode<FMT, XT, 2 * KTL>(wb, bases);
            const uint32_t a2 = decode<FMT, XT, 2 * KTL + 1>(wa, bases);
            const uint32_t a3 = decode<FMT, XT, 2 * KTL + 1>(wb, bases);
            if constexpr (first)
                mma16816_c<XT>(acc[tl][set], a0, a1, a2, a3, b0, b1, init[set]);
            else
                mma16816<XT>(acc[tl][set], a0, a1, a2, a3, b0, b1);
        }
    }

    // k-tile pair P of both halves, alternating between the two halves'
    // accumulator chains.
    template <int... P>
    static __device__ __forceinline__ void pairs(std::integer_sequence<int, P...>,
                                                 const uint4 (&w)[TPW], uint32_t xa,
                                                 const uint32_t (&bases)[NB],
                                                 const float4 (&init)[NSET],
                                                 float (&acc)[TPW][NSET][4])
    {
        (
            [&] {
                const uint4 q0 = ldsm_x4(xa + P * 64);                    // k-tiles 2P, 2P + 1
                const uint4 q1 = ldsm_x4(xa + (T::KT / 4 + P) * 64);      // the second half's
                ktile<0, 2 * P>(w, q0.x, q0.y, bases, init, acc);
                ktile<1, 2 * P>(w, q1.x, q1.y, bases, init, acc);
                ktile<0, 2 * P + 1>(w, q0.z, q0.w, bases, init, acc);
                ktile<1, 2 * P + 1>(w, q1.z, q1.w, bases, init, acc);
            }(),
            ...);
    }

    template <int... GI>
    static __device__ __forceinline__ void epilogue(std::integer_sequence<int, GI...>,
                                                    const uint32_t (&sd)[TPW][T::SIDE_W],
                                                    const float* corr_c, const float* rsum_c,
                                                    float (&acc)[TPW][NSET][4],
                                                    float (&y)[TPW][4], int t)
    {
        (
            [&] {
                constexpr int gi = GI;
#pragma unroll
                for (int tl = 0; tl < TPW; ++tl) {
                    const float (&a)[4] = acc[tl][gi];
                    if constexpr (T::AFFINE) {
                        const float2 sc = f16pair(sd[tl][2 * gi]);
                        const float2 bi = f16pair(sd[tl][2 * gi + 1]);
                        const float2 R = *reinterpret_cast<const float2*>(rsum_c + gi * 8 + 2 * t);
                        y[tl][0] = fmaf(sc.x, a[0], fmaf(bi.x, R.x, y[tl][0]));
                        y[tl][1] = fmaf(sc.x, a[1], fmaf(bi.x, R.y, y[tl][1]));
                        y[tl][2] = fmaf(sc.y, a[2], fmaf(bi.y, R.x, y[tl][2]));
                        y[tl][3] = fmaf(sc.y, a[3], fmaf(bi.y, R.y, y[tl][3]));
                    } else {
                        const float2 sc = f16pair(sd[tl][gi]);
                        y[tl][0] = fmaf(sc.x, a[0], y[tl][0]);
                        y[tl][1] = fmaf(sc.x, a[1], y[tl][1]);
                        y[tl][2] = fmaf(sc.y, a[2], y[tl][2]);
                        y[tl][3] = fmaf(sc.y, a[3], y[tl][3]);
                    }
                }
            }(),
            ...);
    }

    // One chunk (cl = chunk index within the slice) of a warp's unit.
    static __device__ __forceinline__ void process_chunk(const uint4 (&w)[TPW],
                                                         const uint32_t (&sd)[TPW][T::SIDE_W],
                                                         int cl, uint32_t xa,
                                                         const float* __restrict__ corr,
                                                         const float* __restrict__ rsum,
                                                         const uint32_t (&bases)[NB],
                                                         float (&y)[TPW][4], int lane)
    {
        const int t = lane & 3;
        const float* corr_c = corr + cl * T::GPC * 16;
        const float* rsum_c = rsum + cl * T::GPC * 8;
        float acc[TPW][NSET][4];
        // each group's correction as the C fragment of its chain's first MMA:
        // rows 2t, 2t + 1 for columns g and g + 8, one 16-byte load
        float4 init[NSET];
#pragma unroll
        for (int j = 0; j < NSET; ++j)
            init[j] = *reinterpret_cast<const float4*>(corr_c + j * 16 + 4 * t);
        pairs(std::make_integer_sequence<int, T::KT / 4>{}, w, xa + cl * T::CHUNK_K * 2, bases,
              init, acc);
        epilogue(std::make_integer_sequence<int, T::GPC>{}, sd, corr_c, rsum_c, acc, y, t);
    }

    // A unit's results: straight to Y (no K split), or into the shared memory
    // of the cluster CTA that owns the tile (K split).  Tile t0 + i belongs to
    // rank i % S and lands in its slot [(i / S) * S + my_rank].
    // With an argmax (fused head, no K split) the unit's best column of rows
    // 2t and 2t + 1 also updates this lane's running keys ak.
    static __device__ __forceinline__ void store_unit(const VerifyParams& p, int t1, int tile0,
                                                      const float (&y)[TPW][4], int g, int t,
                                                      float* part, int tbase, int lane,
                                                      unsigned long long (&ak)[2])
    {
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl) {
            const int tile = tile0 + tl;
            if (tile >= t1)
                continue;
            if (p.splits > 1) {
                cg::cluster_group cl = cg::this_cluster();
                const int S = p.splits;
                const int i = tile - tbase;
#ifdef LBV_CHECKED
                // the slot lies inside the owner's partial buffer
                if (i < 0 || (i / S + 1) * S > (t1 - tbase + S - 1) / S * S) {
                    atomicOr(p.err, 2u);
                    continue;
                }
#endif
                float* dst = cl.map_shared_rank(part, (unsigned)(i % S)) +
                             ((i / S) * S + (int)cl.block_rank()) * 128;
#pragma unroll
                for (int j = 0; j < 4; ++j)
                    dst[j * 32 + lane] = y[tl][j];
                continue;
            }
            if (!p.store_y)
                continue;
            const int n0 = tile * 16 + g, n1 = n0 + 8;
            const int m0 = 2 * t, m1 = 2 * t + 1;
            if (m0 < p.M) {
                if (n0 < p.N) p.Y[(size_t)m0 * p.ldy + n0] = y[tl][0];
                if (n1 < p.N) p.Y[(size_t)m0 * p.ldy + n1] = y[tl][2];
            }
            if (m1 < p.M) {
                if (n0 < p.N) p.Y[(size_t)m1 * p.ldy + n0] = y[tl][1];
                if (n1 < p.N) p.Y[(size_t)m1 * p.ldy + n1] = y[tl][3];
            }
        }
        if (p.splits == 1 && p.amax_keys) {
#pragma unroll
            for (int tl = 0; tl < TPW; ++tl) {
                const int tile = tile0 + tl;
                const int n0 = tile * 16 + g, n1 = n0 + 8;
                if (tile >= t1)
                    continue;
                if (n0 < p.N) {
                    ak[0] = max(ak[0], amax_key(y[tl][0], n0));
                    ak[1] = max(ak[1], amax_key(y[tl][1], n0));
                }
                if (n1 < p.N) {
                    ak[0] = max(ak[0], amax_key(y[tl][2], n1));
                    ak[1] = max(ak[1], amax_key(y[tl][3], n1));
                }
            }
        }
    }

#ifdef LBV_CHECKED
    // Checked build: walks a warp's whole copy schedule (the cursor the loads
    // follow) and checks that every copy reads inside the packed matrix and
    // fits its ring slot.  False (and the bounds bit set) if one does not; the
    // warp then issues nothing and does no work.
    static __device__ bool copies_in_range(const VerifyParams& p, int t0, int t1, int c0, int nch,
                                           int nstage, int nu, int warp, int lane)
    {
        const uint8_t* end = p.W + (size_t)p.ntiles * p.nchunks * G::REC;
        const size_t tstride = (size_t)p.nchunks * G::REC;
        Cursor c;
        c.unit = warp;
        c.stage = 0;
        if (nu > 0)
            cursor_set(p, t0, t1, c0, nch, c);
        for (int i = 0; i < nu * nstage; ++i) {
            const bool ok = c.nvalid >= 1 && c.nvalid <= TPW && c.nc >= 1 && c.nc <= G::CPS &&
                            c.rec >= p.W &&
                            c.rec + (size_t)(c.nvalid - 1) * tstride + (size_t)c.nc * G::REC <= end;
            if (!ok) {
                if (lane == 0)
                    atomicOr(p.err, 2u);
                return false;
            }
            cursor_next(p, t0, t1, c0, nch, nstage, c);
        }
        return true;
    }
#endif

    // Stage X[0..8) x [kb, kb + nch*CHUNK_K) in fragment order (rows >= M
    // and K >= p.K are zero).
    // X slice [kb, kb + nch * CHUNK_K) of rows m < M, row-major at xs + m * RS.
    // Aligned X: thread 0 issues one bulk copy per row (completing on xbar);
    // the others zero what lies past K in the last chunk.  Otherwise all
    // threads copy it with plain loads.  Rows >= M are left as they are: they
    // only reach output columns >= M, which are never stored.
    static __device__ __forceinline__ bool stage_x(const VerifyParams& p, unsigned char* xs, int RS,
                                                   uint32_t xbar, int c0, int nch)
    {
        const int kb = c0 * T::CHUNK_K;
        const int span = nch * T::CHUNK_K;                   // elements per row slice
#ifdef LBV_CHECKED
        // the slice starts inside K and fits the row buffer: otherwise nothing
        // is staged (the result is then wrong and the status says so)
        if (kb > p.K || nch < 1 || span * 2 + 16 > RS) {
            if (threadIdx.x == 0)
                atomicOr(p.err, 2u);
            return false;
        }
#endif
        const int have = min(span, p.K - kb);                // elements inside K (K % 16 == 0)
        const uint16_t* X = reinterpret_cast<const uint16_t*>(p.X);
        if (p.x_vec) {
            if (threadIdx.x == 0) {
                mbar_expect_tx(xbar, (uint32_t)(p.M * have * 2));
                for (int m = 0; m < p.M; ++m)
                    bulk_g2s_if(1u, smem_u32(xs + (size_t)m * RS), X + (size_t)m * p.ldx + kb,
                                (uint32_t)(have * 2), xbar);
            }
            const int tail = (span - have) / 8;              // 16-byte pieces past K, per row
            for (int i = threadIdx.x; i < p.M * tail; i += NW * 32) {
                const int m = i / tail, k8 = have + (i - m * tail) * 8;
                *reinterpret_cast<uint4*>(xs + (size_t)m * RS + k8 * 2) = make_uint4(0u, 0u, 0u, 0u);
            }
            return true;
        }
        for (int i = threadIdx.x; i < p.M * span; i += NW * 32) {
            const int m = i / span, k = i - m * span;
            reinterpret_cast<uint16_t*>(xs + (size_t)m * RS)[k] =
                k < have ? X[(size_t)m * p.ldx + kb + k] : (uint16_t)0;
        }
        return false;
    }

    // Per-group corrections of the slice, one warp per chunk, on the tensor
    // cores: for each k-tile one m16n8k16 MMA of the staged X fragments (the
    // main loop's B operands) with a constant A whose rows 0..7 hold the
    // decode offset c of each K position (Q4_0: c + 8, as w = d (q - 8)) and
    // rows 8..15 ones, chained over the group's k-tiles.  So lane (g, t) holds
    //   D[g][2t + j]     = sum_k c_k x_k   (row 2t + j of X)
    //   D[g + 8][2t + j] = sum_k x_k       (its row sum)
    // and corr = -sum_k c_k x_k, rsum = the row sum.  Every product is exact
    // (c and x are fp16/bf16 values); the sums are the tensor core's fp32.
    static __host__ __device__ constexpr uint32_t small_int_bits(int xt, int v)
    {
        // v = 0 or a positive integer exact in the X dtype
        int e = 0;
        while ((2 << e) <= v)
            ++e;
        return v == 0 ? 0u
               : xt == LBV_F16
                   ? (uint32_t)((e + 15) << 10) | (uint32_t)((v - (1 << e)) << (10 - e))
                   : (uint32_t)((e + 127) << 7) | (uint32_t)((v - (1 << e)) << (7 - e));
    }

    static __host__ __device__ constexpr uint32_t offset_pair(int slot)
    {
        const int c = dec_spec<FMT>(XT, slot).c + (FMT == LBV_FMT_Q4_0 ? 8 : 0);
        const uint32_t h = small_int_bits(XT, c);
        return h | (h << 16);
    }

    static __host__ __device__ constexpr bool offsets_exact()
    {
        for (int slot = 0; slot < T::KT; ++slot) {
            const int c = dec_spec<FMT>(XT, slot).c + (FMT == LBV_FMT_Q4_0 ? 8 : 0);
            if (half_bits_value(XT, offset_pair(slot) & 0xFFFFu) != (double)c)
                return false;
        }
        return true;
    }
    static_assert(offsets_exact(), "a decode offset is not exact in the X dtype");

    template <int... KP>
    static __device__ __forceinline__ void corr_pairs(std::integer_sequence<int, KP...>,
                                                      uint32_t xa, float (&d)[T::GPC][4])
    {
        constexpr uint32_t one = XT == LBV_F16 ? 0x3C003C00u : 0x3F803F80u;
        (
            [&] {
                const uint4 q = ldsm_x4(xa + KP * 64);            // k-tiles 2 KP, 2 KP + 1
#pragma unroll
                for (int e = 0; e < 2; ++e) {
                    const int kt = 2 * KP + e;                    // folds after unrolling
                    const int ktl = kt % (T::KT / 2);
                    const int gi = kt / T::KTG;
                    const uint32_t a0 = offset_pair(2 * ktl), a2 = offset_pair(2 * ktl + 1);
                    const uint32_t b0 = e ? q.z : q.x, b1 = e ? q.w : q.y;
                    if (kt % T::KTG == 0)
                        mma16816_c<XT>(d[gi], a0, one, a2, one, b0, b1,
                                       make_float4(0.f, 0.f, 0.f, 0.f));
                    else
                        mma16816<XT>(d[gi], a0, one, a2, one, b0, b1);
                }
            }(),
            ...);
    }

    static __device__ __forceinline__ void corrections(uint32_t xs_a, int RS, float* corr, float* rsum,
                                                       int nch, int warp, int lane)
    {
        const int g = lane >> 2, t = lane & 3;
        for (int cl = warp; cl < nch; cl += NW) {
            float d[T::GPC][4];
            corr_pairs(std::make_integer_sequence<int, T::KT / 2>{},
                       xs_a + ldsm_lane_offset(RS, lane) + cl * T::CHUNK_K * 2, d);
            if (g == 0) {
#pragma unroll
                for (int i = 0; i < T::GPC; ++i) {
                    // corr holds each group's C fragment: for lane t the quad
                    // (row 2t, row 2t + 1, row 2t, row 2t + 1)
                    const int gr = cl * T::GPC + i;
                    *reinterpret_cast<float4*>(corr + gr * 16 + 4 * t) =
                        make_float4(-d[i][0], -d[i][1], -d[i][0], -d[i][1]);
                    if constexpr (T::AFFINE)
                        *reinterpret_cast<float2*>(rsum + gr * 8 + 2 * t) =
                            make_float2(d[i][2], d[i][3]);
                }
            }
        }
    }

    // Fused head epilogue: the CTA's keys go to the workspace; the CTA that
    // finishes last turns the keys into the rows' argmax columns and logits
    // and leaves the workspace zeroed for the next call.  One thread per row
    // on every step, so the last CTA's tail is three round trips to L2: the
    // fence after the key reductions, the ticket, the exchange of the keys.
    // `last` is a shared flag word.
    static __device__ void amax_finish(const VerifyParams& p, const unsigned long long* akeys,
                                       unsigned* last)
    {
        __syncthreads();
        const int tid = (int)threadIdx.x;
        if (tid < p.M) {                        // warp 0
            const unsigned long long k = akeys[tid];
            if (k)
                atomicMax(p.amax_keys + tid, k);
            __threadfence();                    // the CTA's reductions before its ticket
        }
        __syncthreads();
        if (tid == 0) {
            const unsigned total = gridDim.x * gridDim.y;
            *last = atomicAdd(p.amax_done, 1u) == total - 1u;
        }
        __syncthreads();
        if (*last) {
            __threadfence();                    // every CTA's reductions before the reads
            if (tid < p.M) {
                const unsigned long long k = atomicExch(p.amax_keys + tid, 0ull);
                p.amax_idx[tid] = (int)(0xffffffffu - (uint32_t)k);   // -1: no column
                if (p.amax_val)
                    p.amax_val[tid] = amax_key_value(k);
            }
            if (tid == 0)
                atomicExch(p.amax_done, 0u);
        }
    }

    // Cluster row cy of ny (the clusters along N that share the problem's
    // tiles; blockIdx.x is the K slice).
    static __device__ void run(const VerifyParams& p, unsigned char* smem, int cy, int ny)
    {
        const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
        const int g = lane >> 2, t = lane & 3;
        const int S = p.splits;
        const int c0 = blockIdx.x * p.cps;
        const int nch = min(p.cps, p.nchunks - c0);          // >= 1 (host guarantees)
        const int t0 = (int)(((unsigned)p.ntiles * cy) / ny);
        const int t1 = (int)(((unsigned)p.ntiles * (cy + 1)) / ny);

        unsigned char* ring = smem;
        unsigned char* bars = ring + G::RING_B;
        unsigned char* xs = bars + G::BAR_B;
        const int RS = x_row_stride<FMT, GROUP>(p.cps);
        const uint32_t xbar = smem_u32(bars) + (uint32_t)(NW * STAGES * 8);
        float* corr = reinterpret_cast<float*>(xs + (size_t)8 * RS);
        float* rsum = corr + p.cps * T::GPC * 16;
        float* part = rsum + (T::AFFINE ? p.cps * T::GPC * 8 : 0);
#ifdef LBV_CHECKED
        // Checked build: the carve-up, with the partial slots of a K split, ends
        // inside the launch's dynamic shared memory.  The test reads only values
        // a cluster's CTAs share (the launch, t0, t1), so a cluster leaves whole
        // and no CTA is left waiting at a cluster barrier.
        {
            const size_t need = (size_t)(reinterpret_cast<unsigned char*>(part) - smem) +
                                (S > 1 ? (size_t)((t1 - t0 + S - 1) / S) * S * 512u : 0u);
            uint32_t dyn;
            asm volatile("mov.u32 %0, %%dynamic_smem_size;\n" : "=r"(dyn));
            if (need > dyn || p.M < 1 || p.M > 8 || p.cps < 1) {
                if (threadIdx.x == 0)
                    atomicOr(p.err, 2u);
                return;
            }
        }
#endif

        const uint32_t ring_w = smem_u32(ring) + warp * STAGES * G::SLOT_B;
        const uint32_t bars_w = smem_u32(bars) + warp * STAGES * 8;
        const unsigned char* ring_wp = ring + (size_t)warp * STAGES * G::SLOT_B;
        unsigned long long* akeys =
            reinterpret_cast<unsigned long long*>(bars + NW * STAGES * 8 + 16);
        if (threadIdx.x < 8)
            akeys[threadIdx.x] = 0ull;

        // this warp's units of TPW tiles within [t0, t1)
        const int nunits = (t1 - t0 + TPW - 1) / TPW;
        const int nu = warp < nunits ? (nunits - 1 - warp) / NW + 1 : 0;

        if (S > 1)
            cluster_arrive_relaxed();
        if (lane == 0) {
#pragma unroll 1
            for (int s = 0; s < STAGES; ++s)
                mbar_init(bars_w + s * 8, 1);
            if (warp == 0)
                mbar_init(xbar, 1);
            mbar_init_fence();
        }
        __syncwarp();

        // XOR bases in registers: opaque values cannot be folded back into
        // immediates, so each decode stays one LOP3.
        uint32_t bases[NB];
#pragma unroll
        for (int i = 0; i < NB; ++i)
            asm volatile("mov.b32 %0, %1;\n" : "=r"(bases[i]) : "r"(base_of<FMT>(XT, i)));

        // Packed weights are read-only: start streaming before waiting on the
        // previous kernel in the stream.
        const int nstage = (nch + G::CPS - 1) / G::CPS;
#ifdef LBV_CHECKED
        const int Q = copies_in_range(p, t0, t1, c0, nch, nstage, nu, warp, lane) ? nu * nstage : 0;
#else
        const int Q = nu * nstage;
#endif
        const uint32_t leader = lane == 0;
        // wait-limit test (LBV_PLAN_TEST_WAIT_LIMIT): the first warp of the
        // first CTA does not issue its ring stage skip_q, so its wait on that
        // stage runs out; ring waits give up after wait_limit tries
        const int skip_q = (warp == 0 && blockIdx.x == 0 && blockIdx.y == 0) ? p.skip_q : -1;
        const uint32_t wait_limit = p.wait_limit ? (uint32_t)p.wait_limit : 1u << 20;
        Cursor lcur;
        lcur.unit = warp;
        lcur.stage = 0;
        cursor_set(p, t0, t1, c0, nch, lcur);
        const size_t tstride = (size_t)p.nchunks * G::REC;
        int lq = 0;
        const int npre = min(STAGES, Q);
        // one stage before the wait on the previous kernel (it overlaps that
        // kernel's tail); the rest after this CTA's activation copies, which
        // the bulk copy engine serves in issue order
        const int nearly = min(1, npre);
#pragma unroll 1
        for (; lq < nearly; ++lq) {
            issue(lcur, tstride, leader && lq != skip_q, ring_w, bars_w, lq);
            cursor_next(p, t0, t1, c0, nch, nstage, lcur);
        }

        griddep_wait();
        const bool x_async = stage_x(p, xs, RS, xbar, c0, nch);
#pragma unroll 1
        for (; lq < npre; ++lq) {
            issue(lcur, tstride, leader && lq != skip_q, ring_w, bars_w, lq);
            cursor_next(p, t0, t1, c0, nch, nstage, lcur);
        }
        __syncthreads();               // X barrier initialised, tails zeroed (or X copied)
        bool x_ok = true;
        if (x_async && !mbar_try(xbar, 0) && !mbar_wait(xbar, 0))
            x_ok = false;
        const uint32_t xs_a = smem_u32(xs);
        if (p.rot) {
            // every thread's wait on X has ended before X is rewritten
            const int kb = c0 * T::CHUNK_K, have = min(nch * T::CHUNK_K, p.K - kb);
            if (__syncthreads_and(x_ok)) {
                if (p.signs) {
                    flip_signs(p.signs, xs, RS, p.M, kb, have, threadIdx.x, NW * 32);
                    __syncthreads();
                }
                rotate_x<XT>(xs_a, RS, have / 128, warp, NW, lane);
            }
            __syncthreads();
        }
        corrections(xs_a, RS, corr, rsum, nch, warp, lane);
        __syncthreads();
        if (S > 1)
            cluster_wait();            // all peers run: their partial buffers are live
        griddep_launch_dependents();

        float y[TPW][4];
#pragma unroll
        for (int tl = 0; tl < TPW; ++tl)
            y[tl][0] = y[tl][1] = y[tl][2] = y[tl][3] = 0.f;
        unsigned long long ak[2] = {0ull, 0ull};              // argmax keys, rows 2t, 2t + 1
        int cu = warp, cc = 0;                                // compute cursor
        const uint32_t xa_lane = xs_a + ldsm_lane_offset(RS, lane);
        bool ok = x_ok;
        int q = 0, slot = 0;
        uint32_t parity = 0;
#pragma unroll 1
        for (; q < Q; ++q) {
            const uint32_t bar = bars_w + slot * 8;
            // the whole warp leaves together (the unit store below shuffles)
            const bool landed = mbar_try(bar, parity) || mbar_wait(bar, parity, wait_limit);
            if (!__all_sync(0xffffffffu, landed)) {
                ok = false;
                break;
            }
            const int nc = min(G::CPS, nch - cc);
            uint4 w[G::CPS][TPW];
            uint32_t sd[G::CPS][TPW][T::SIDE_W];
            const unsigned char* src = ring_wp + slot * G::SLOT_B;
#pragma unroll
            for (int ci = 0; ci < G::CPS; ++ci)
#pragma unroll
                for (int tl = 0; tl < TPW; ++tl) {
                    const unsigned char* r = src + (tl * G::CPS + ci) * G::REC;
                    w[ci][tl] = reinterpret_cast<const uint4*>(r)[lane];
                    // side words of column pair g: 8, 16 or 32 bytes, as wide loads
                    // (records are 16-byte aligned, so is r + 512 + g * SIDE_B)
                    const unsigned char* sp = r + 512 + g * G::SIDE_B;
                    if constexpr (T::SIDE_W == 2) {
                        const uint2 v = *reinterpret_cast<const uint2*>(sp);
                        sd[ci][tl][0] = v.x;
                        sd[ci][tl][1] = v.y;
                    } else {
                        static_assert(T::SIDE_W % 4 == 0, "side words in 16-byte pieces");
#pragma unroll
                        for (int i = 0; i < T::SIDE_W / 4; ++i) {
                            const uint4 v = reinterpret_cast<const uint4*>(sp)[i];
                            sd[ci][tl][4 * i] = v.x;
                            sd[ci][tl][4 * i + 1] = v.y;
                            sd[ci][tl][4 * i + 2] = v.z;
                            sd[ci][tl][4 * i + 3] = v.w;
                        }
                    }
                }
            __syncwarp();
            if (lq < Q) {
                fence_proxy_async_if(leader);
                issue(lcur, tstride, leader && lq != skip_q, ring_w, bars_w, slot);
                ++lq;
                cursor_next(p, t0, t1, c0, nch, nstage, lcur);
            }
            if (++slot == STAGES) {
                slot = 0;
                parity ^= 1u;
            }
#ifdef LBV_CHECKED
            // the stage's chunks lie inside the staged X slice and its corrections
            if (nc < 1 || cc + nc > p.cps) {
                if (lane == 0)
                    atomicOr(p.err, 2u);
                ok = false;
                break;
            }
#endif
#pragma unroll
            for (int ci = 0; ci < G::CPS; ++ci)
                if (ci == 0 || ci < nc)
                    process_chunk(w[ci], sd[ci], cc + ci, xa_lane, corr, rsum, bases, y, lane);
            cc += nc;
            if (cc == nch) {
                store_unit(p, t1, t0 + cu * TPW, y, g, t, part, t0, lane, ak);
#pragma unroll
                for (int tl = 0; tl < TPW; ++tl)
                    y[tl][0] = y[tl][1] = y[tl][2] = y[tl][3] = 0.f;
                cc = 0;
                cu += NW;
            }
        }
        if (!ok) {
            if (lane == 0)
                atomicOr(p.err, 1u);
            // let the copies already issued into this warp's ring (and X) land
            for (int r = q; r < lq; ++r)
                if (r != skip_q)
                    mbar_wait(bars_w + (r % STAGES) * 8, (uint32_t)((r / STAGES) & 1));
            if (x_async && !x_ok)
                mbar_wait(xbar, 0);
        }

        if (S == 1 && p.amax_keys) {                          // the warp's keys into the CTA's
            ak[0] = warp_max_key(ak[0]);
            ak[1] = warp_max_key(ak[1]);
            if (g == 0) {
                if (2 * t < p.M && ak[0])
                    atomicMax(akeys + 2 * t, ak[0]);
                if (2 * t + 1 < p.M && ak[1])
                    atomicMax(akeys + 2 * t + 1, ak[1]);
            }
        }
        if (S > 1)
            cluster_reduce(p, part, t0, t1, akeys);
        if (p.amax_keys)
            amax_finish(p, akeys, reinterpret_cast<unsigned*>(bars + NW * STAGES * 8 + 8));
    }

    // After the cluster barrier each CTA sums, in rank order 0..S-1, the
    // partials its cluster peers stored for the tiles it owns, and writes Y.
    // With an argmax each thread's elements lie in one row (the stride NW * 32
    // is a multiple of 128), so its best key needs only a warp reduction.
    static __device__ void cluster_reduce(const VerifyParams& p, float* part, int t0, int t1,
                                          unsigned long long* akeys)
    {
        static_assert((NW * 32) % 128 == 0, "one row per thread in the reduction");
        cg::cluster_group cl = cg::this_cluster();
        cl.sync();
        const int S = p.splits;
        const int rank = (int)cl.block_rank();
        const int nown = (t1 - t0 - rank + S - 1) / S;        // tiles t0 + rank + S*k
        unsigned long long best = 0ull;
        for (int e = (int)threadIdx.x; e < nown * 128; e += NW * 32) {
            const int k = e >> 7, r = e & 127;
#ifdef LBV_CHECKED
            if ((k + 1) * S > (t1 - t0 + S - 1) / S * S) {   // inside the partial buffer
                atomicOr(p.err, 2u);
                continue;
            }
#endif
            const float* src = part + (k * S) * 128 + r;
            float acc = 0.f;
            for (int q = 0; q < S; ++q)
                acc += src[q * 128];
            const int tile = t0 + rank + S * k;
            const int j = r >> 5, ln = r & 31;
            const int n = tile * 16 + (ln >> 2) + 8 * (j >> 1);
            const int m = 2 * (ln & 3) + (j & 1);
            if (n < p.N && m < p.M) {
                if (p.store_y)
                    p.Y[(size_t)m * p.ldy + n] = acc;
                if (p.amax_keys)
                    best = max(best, amax_key(acc, n));
            }
        }
        if (p.amax_keys) {
            best = warp_max_key(best);
            const int lane = threadIdx.x & 31;
            const int m = 2 * (lane & 3) + ((threadIdx.x >> 5) & 1);
            if (lane < 4 && m < p.M && best)
                atomicMax(akeys + m, best);
        }
    }
};

template <int FMT, int XT, int GROUP, int NW, int TPW>
__global__ void __launch_bounds__(NW * 32, 1) lbv_verify_kernel(const VerifyParams p)
{
    extern __shared__ __align__(128) unsigned char smem[];
    constexpr int SC = stage_chunks<FMT, GROUP, TPW>();
    VerifyKernel<FMT, XT, GROUP, NW, TPW, SC>::run(p, smem, (int)blockIdx.y, (int)gridDim.y);
}

// Grouped verify: independent problems of one format in one launch.  Cluster
// row blockIdx.y belongs to the problem i with ybegin[i] <= y < ybegin[i + 1]
// and is its (y - ybegin[i])-th of (ybegin[i + 1] - ybegin[i]) rows; every
// problem uses the launch's K split.  Clusters of a problem with M = 0 exit
// at once.
template <int FMT, int XT, int GROUP, int NW, int TPW>
__global__ void __launch_bounds__(NW * 32, 1)
    lbv_verify_grouped_kernel(const __grid_constant__ GroupedParams gp)
{
    extern __shared__ __align__(128) unsigned char smem[];
    const int y = (int)blockIdx.y;
    int lo = 0, hi = gp.count;                               // ybegin[lo] <= y < ybegin[hi]
    while (hi - lo > 1) {
        const int mid = (lo + hi) >> 1;
        if (gp.ybegin[mid] <= y)
            lo = mid;
        else
            hi = mid;
    }
    const GroupedProblem& q = gp.prob[lo];
    if (q.M == 0)
        return;
    VerifyParams p;
    p.X = q.X;
    p.W = q.W;
    p.Y = q.Y;
    p.err = gp.err;
    p.ldx = q.ldx;
    p.ldy = q.ldy;
    p.M = q.M;
    p.K = q.K;
    p.N = q.N;
    p.ntiles = q.ntiles;
    p.nchunks = q.nchunks;
    p.splits = gp.splits;
    p.cps = q.cps;
    p.wait_limit = 0;
    p.skip_q = -1;
    p.x_vec = q.x_vec;
    p.zero = 0;
    p.rot = 0;
    p.store_y = 1;
    p.signs = nullptr;
    p.amax_keys = nullptr;
    p.amax_done = nullptr;
    p.amax_idx = nullptr;
    p.amax_val = nullptr;
    constexpr int SC = stage_chunks<FMT, GROUP, TPW>();
    VerifyKernel<FMT, XT, GROUP, NW, TPW, SC>::run(p, smem, y - gp.ybegin[lo],
                                                   gp.ybegin[lo + 1] - gp.ybegin[lo]);
}

// ---------------------------------------------------------------------------
// Host side: launch / smem / cluster occupancy for one (FMT, XT, GROUP)

template <int FMT, int XT, int GROUP>
inline void* kernel_ptr(int warps, int tpw)
{
    if (warps == 8 && tpw == 2) return (void*)lbv_verify_kernel<FMT, XT, GROUP, 8, 2>;
    if (warps == 8 && tpw == 4) return (void*)lbv_verify_kernel<FMT, XT, GROUP, 8, 4>;
    if (warps == 16 && tpw == 1) return (void*)lbv_verify_kernel<FMT, XT, GROUP, 16, 1>;
    if (warps == 16 && tpw == 2) return (void*)lbv_verify_kernel<FMT, XT, GROUP, 16, 2>;
    return nullptr;
}

// Grouped launches use 16 warps with 1 or 2 tiles per unit.
template <int FMT, int XT, int GROUP>
inline void* grouped_kernel_ptr(int warps, int tpw)
{
    if (warps == 16 && tpw == 1) return (void*)lbv_verify_grouped_kernel<FMT, XT, GROUP, 16, 1>;
    if (warps == 16 && tpw == 2) return (void*)lbv_verify_grouped_kernel<FMT, XT, GROUP, 16, 2>;
    return nullptr;
}

template <int FMT, int GROUP, int NW, int TPW>
inline size_t smem_bytes_k(int cps, int tiles_max, int splits)
{
    return smem_bytes_for<FMT, GROUP, NW, TPW, stage_chunks<FMT, GROUP, TPW>()>(cps, tiles_max,
                                                                              splits);
}

template <int FMT, int GROUP>
inline size_t smem_bytes_t(int warps, int tpw, int cps, int tiles_max, int splits)
{
    if (warps == 8 && tpw == 2) return smem_bytes_k<FMT, GROUP, 8, 2>(cps, tiles_max, splits);
    if (warps == 8 && tpw == 4) return smem_bytes_k<FMT, GROUP, 8, 4>(cps, tiles_max, splits);
    if (warps == 16 && tpw == 1) return smem_bytes_k<FMT, GROUP, 16, 1>(cps, tiles_max, splits);
    if (warps == 16 && tpw == 2) return smem_bytes_k<FMT, GROUP, 16, 2>(cps, tiles_max, splits);
    return (size_t)1 << 40;
}

inline void fill_config(cudaLaunchConfig_t& cfg, cudaLaunchAttribute (&attr)[2], const Shape& sh,
                        bool pdl, cudaStream_t st)
{
    cfg = {};
    cfg.gridDim = dim3((unsigned)sh.splits, (unsigned)sh.ctas_n, 1u);
    cfg.blockDim = dim3((unsigned)(sh.warps * 32), 1u, 1u);
    cfg.dynamicSmemBytes = sh.smem;
    cfg.stream = st;
    unsigned na = 0;
    if (sh.splits > 1) {
        attr[na].id = cudaLaunchAttributeClusterDimension;
        attr[na].val.clusterDim.x = (unsigned)sh.splits;
        attr[na].val.clusterDim.y = 1;
        attr[na].val.clusterDim.z = 1;
        ++na;
    }
    if (pdl) {
        attr[na].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[na].val.programmaticStreamSerializationAllowed = 1;
        ++na;
    }
    cfg.attrs = attr;
    cfg.numAttrs = na;
}

template <int FMT, int XT, int GROUP>
inline cudaError_t launch_t(const Shape& sh, const VerifyParams& p, const LaunchOpts& o,
                            cudaStream_t st)
{
    void* k = kernel_ptr<FMT, XT, GROUP>(sh.warps, sh.tpw);
    if (!k)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_config(cfg, attr, sh, o.pdl, st);
    void* args[] = {const_cast<VerifyParams*>(&p)};
    return cudaLaunchKernelExC(&cfg, k, args);
}

template <int FMT, int XT, int GROUP>
inline cudaError_t launch_grouped_t(const Shape& sh, const GroupedParams& gp, const LaunchOpts& o,
                                    cudaStream_t st)
{
    void* k = grouped_kernel_ptr<FMT, XT, GROUP>(sh.warps, sh.tpw);
    if (!k)
        return cudaErrorInvalidValue;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    fill_config(cfg, attr, sh, o.pdl, st);
    void* args[] = {const_cast<GroupedParams*>(&gp)};
    return cudaLaunchKernelExC(&cfg, k, args);
}

template <int FMT, int XT, int GROUP>
inline cudaError_t prepare_t(const Shape& sh, bool grouped = false)
{
    void* k = grouped ? grouped_kernel_ptr<FMT, XT, GROUP>(sh.warps, sh.tpw)
                      : kernel_ptr<FMT, XT, GROUP>(sh.warps, sh.tpw);
    if (!k)
        return cudaErrorInvalidValue;
    return cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)sh.smem > kMaxDynSmem ? (int)sh.smem : kMaxDynSmem);
}

// Clusters of the shape that can be resident at once (0 if none fits).
template <int FMT, int XT, int GROUP>
inline int max_clusters_t(const Shape& sh, bool grouped = false)
{
    void* k = grouped ? grouped_kernel_ptr<FMT, XT, GROUP>(sh.warps, sh.tpw)
                      : kernel_ptr<FMT, XT, GROUP>(sh.warps, sh.tpw);
    if (!k || prepare_t<FMT, XT, GROUP>(sh, grouped) != cudaSuccess)
        return 0;
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attr[2];
    Shape s1 = sh;
    s1.ctas_n = 1;
    fill_config(cfg, attr, s1, false, nullptr);
    int n = 0;
    if (sh.splits > 1) {
        if (cudaOccupancyMaxActiveClusters(&n, k, &cfg) != cudaSuccess)
            return 0;
        return n;
    }
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&n, k, sh.warps * 32, sh.smem) !=
        cudaSuccess)
        return 0;
    int dev = 0, sms = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
    return n * sms;
}

}  // namespace lbv
