/*
 * oracle.c -- plain fp64 CPU reference for the few-row packed-weight verify
 * matmul  y[M,N] = X[M,K] . dequant(Wp)[K,N].
 *
 * TEST INFRASTRUCTURE ONLY.  Only the tests, the smoke check and the CPU
 * baseline leg of the benchmark call into this file.  It shares no code,
 * header, table or constant with the CUDA library; it reads the weights in
 * their canonical (file) layout, never in the library's device layout.
 *
 * Everything is computed the slow, obvious way: every weight is decoded to an
 * exact fp64 value from its format definition, and the contraction is a naive
 * loop over k in fp64.  Build with -ffp-contract=off so that no product and
 * sum are fused (the same results on x86 and Arm).
 *
 * Canonical layouts (all little-endian, "per output column n, contiguous
 * along K", the out x in orientation that MLX packs and GGUF files use):
 *   sign1 g128 : bits[N][K/32] uint32, bit (k % 32) of word k/32 is the sign
 *                bit of weight (k, n);  scales[N][K/128] fp16 bit patterns.
 *   affine2    : codes[N][K/16] uint32, code q of weight (k, n) sits in bits
 *                2*(k%16) .. 2*(k%16)+1 of word k/16 ("16 per uint32, little
 *                end first");  scales[N][K/g], biases[N][K/g] fp16.
 *   q4_0       : blocks[N][K/32], 18 bytes each: d (fp16, little-endian)
 *                then qs[16]; element j < 16 is qs[j] & 15, element j + 16
 *                is qs[j] >> 4.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#define ORC_FMT_SIGN1_G128 0
#define ORC_FMT_AFFINE2 1
#define ORC_FMT_Q4_0 2

/* ------------------------------------------------------------------------ */
/* IEEE 754 binary16 / bfloat16 <-> fp64, written from the format definitions */

/* binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double orc_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 31;
    int f = h & 1023;
    double v;
    if (e == 0)
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-24 */
    else if (e == 31)
        v = f ? NAN : INFINITY;
    else
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/1024) 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 is the upper half of an IEEE binary32 word. */
double orc_bf16_to_f64(uint16_t h)
{
    uint32_t u = (uint32_t)h << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * Round an fp64 value to the nearest value of a binary format with `p`
 * significand bits (implicit bit included), `ebits` exponent bits and
 * maximum exponent `emax` (bias = emax, minimum normal exponent 1 - emax);
 * ties go to the even significand.  Returns the format's bit pattern.
 */
static uint32_t orc_round_rne(double v, int p, int ebits, int emax)
{
    const int fbits = p - 1;
    const int emin = 1 - emax;
    const uint32_t eall = (1u << ebits) - 1;              /* inf / nan exponent */
    uint32_t sbit = 0;
    if (isnan(v))
        return (eall << fbits) | (1u << (fbits - 1));
    if (signbit(v)) {
        sbit = 1u << (ebits + fbits);
        v = -v;
    }
    if (isinf(v))
        return sbit | (eall << fbits);
    if (v == 0.0)
        return sbit;
    int E;
    frexp(v, &E);                 /* v = f * 2^E, f in [0.5, 1): exponent E-1 */
    int e = E - 1;
    if (e < emin)
        e = emin;                 /* the subnormal range shares emin's quantum */
    double quantum = ldexp(1.0, e - fbits);
    double n = rint(v / quantum); /* v / quantum is exact; rint ties to even */
    double r = n * quantum;
    double maxfinite = ldexp(2.0 - ldexp(1.0, -fbits), emax);
    if (r > maxfinite)
        return sbit | (eall << fbits);
    if (r < ldexp(1.0, emin))     /* subnormal: exponent field 0 */
        return sbit | (uint32_t)(r / ldexp(1.0, emin - fbits));
    frexp(r, &E);
    e = E - 1;
    uint32_t frac = (uint32_t)((ldexp(r, -e) - 1.0) * ldexp(1.0, fbits));
    return sbit | ((uint32_t)(e + emax) << fbits) | frac;
}

/* binary16: p = 11, 5 exponent bits, emax = 15. */
uint16_t orc_f64_to_f16(double v)
{
    return (uint16_t)orc_round_rne(v, 11, 5, 15);
}

/* bfloat16: p = 8, 8 exponent bits, emax = 127. */
uint16_t orc_f64_to_bf16(double v)
{
    return (uint16_t)orc_round_rne(v, 8, 8, 127);
}

void orc_f64_to_f16_array(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_f64_to_f16(v[i]);
}

void orc_f64_to_bf16_array(const double* v, int64_t n, uint16_t* out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_f64_to_bf16(v[i]);
}

void orc_f16_to_f64_array(const uint16_t* h, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_f16_to_f64(h[i]);
}

void orc_bf16_to_f64_array(const uint16_t* h, int64_t n, double* out)
{
    for (int64_t i = 0; i < n; i++)
        out[i] = orc_bf16_to_f64(h[i]);
}

/* ------------------------------------------------------------------------ */
/* Unpacking one output column to exact fp64 weights w[0..K)                  */

/*
 * 1-bit sign, one fp16 scale per 128 consecutive K-weights of a column.
 * Bonsai-27B-mlx-1bit model card, format description: a weight is one sign
 * bit, 0 stands for -scale and 1 for +scale; each group of 128 weights shares
 * one fp16 scale (1 + 16/128 = 1.125 bits per weight).
 */
void orc_col_sign1(const uint32_t* bits, const uint16_t* scales, int K, int n, double* w)
{
    const uint32_t* col = bits + (int64_t)n * (K / 32);
    const uint16_t* sc = scales + (int64_t)n * (K / 128);
    for (int k = 0; k < K; k++) {
        int b = (col[k / 32] >> (k % 32)) & 1;
        double s = orc_f16_to_f64(sc[k / 128]);
        w[k] = b ? s : -s;
    }
}

/*
 * 2-bit affine groups: w = scale * q + bias, q in {0,1,2,3}, one fp16
 * (scale, bias) pair per `group` consecutive K-weights of a column.
 * Ishizuki README, "Reads what people actually ship" (plain MLX affine packs);
 * dflash-mlx-bonsai2 README, "Why" (the 2-bit pack).  s*q + b is exact in fp64
 * because fp16 operands span at most 40 binary orders of magnitude.
 */
void orc_col_affine2(const uint32_t* codes, const uint16_t* scales, const uint16_t* biases,
                     int K, int group, int n, double* w)
{
    const uint32_t* col = codes + (int64_t)n * (K / 16);
    const uint16_t* sc = scales + (int64_t)n * (K / group);
    const uint16_t* bi = biases + (int64_t)n * (K / group);
    for (int k = 0; k < K; k++) {
        int q = (col[k / 16] >> (2 * (k % 16))) & 3;
        double s = orc_f16_to_f64(sc[k / group]);
        double b = orc_f16_to_f64(bi[k / group]);
        w[k] = s * (double)q + b;
    }
}

/*
 * GGUF Q4_0 block, read as it is stored: 32 weights, an fp16 d and 16 bytes
 * of 4-bit codes, w = d * (q - 8).  Ishizuki README, "Credits" (the GGUF
 * block formats, read as they are) and "Reads what people actually ship".
 */
void orc_col_q4_0(const uint8_t* blocks, int K, int n, double* w)
{
    const uint8_t* col = blocks + (int64_t)n * (K / 32) * 18;
    for (int kb = 0; kb < K / 32; kb++) {
        const uint8_t* blk = col + (int64_t)kb * 18;
        uint16_t dbits = (uint16_t)(blk[0] | (blk[1] << 8));
        double d = orc_f16_to_f64(dbits);
        const uint8_t* qs = blk + 2;
        for (int j = 0; j < 32; j++) {
            int q = j < 16 ? (qs[j] & 15) : (qs[j - 16] >> 4);
            w[kb * 32 + j] = d * (double)(q - 8);
        }
    }
}

static void orc_col(int fmt, const void* p0, const void* p1, const void* p2, int K, int group,
                    int n, double* w)
{
    if (fmt == ORC_FMT_SIGN1_G128)
        orc_col_sign1((const uint32_t*)p0, (const uint16_t*)p1, K, n, w);
    else if (fmt == ORC_FMT_AFFINE2)
        orc_col_affine2((const uint32_t*)p0, (const uint16_t*)p1, (const uint16_t*)p2, K, group,
                        n, w);
    else
        orc_col_q4_0((const uint8_t*)p0, K, n, w);
}

/* Dense unpack: W[K][N] row-major fp64 (for small shapes). */
void orc_unpack(int fmt, const void* p0, const void* p1, const void* p2, int K, int N, int group,
                double* W)
{
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
    for (int n = 0; n < N; n++) {
        orc_col(fmt, p0, p1, p2, K, group, n, w);
        for (int k = 0; k < K; k++)
            W[(int64_t)k * N + n] = w[k];
    }
    free(w);
}

/*
 * Dequantized fp16 weights, rounded once from the exact value:
 * W16[k][n] = RNE_fp16(w[k][n]) for the requested columns cols[0..ncols),
 * written as out[k][j] (row-major [K][ncols]).
 */
void orc_dequant_f16(int fmt, const void* p0, const void* p1, const void* p2, int K, int group,
                     const int64_t* cols, int64_t ncols, uint16_t* out)
{
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t j = 0; j < ncols; j++) {
        orc_col(fmt, p0, p1, p2, K, group, (int)cols[j], w);
        for (int k = 0; k < K; k++)
            out[(int64_t)k * ncols + j] = orc_f64_to_f16(w[k]);
    }
    free(w);
}

/* ------------------------------------------------------------------------ */
/* Contraction                                                                */

/* Naive triple loop, fp64: Y[m][n] = sum_k X[m][k] * W[k][n], k ascending. */
void orc_gemm(const double* X, const double* W, int M, int K, int N, double* Y)
{
    for (int m = 0; m < M; m++)
        for (int n = 0; n < N; n++) {
            double acc = 0.0;
            for (int k = 0; k < K; k++)
                acc += X[(int64_t)m * K + k] * W[(int64_t)k * N + n];
            Y[(int64_t)m * N + n] = acc;
        }
}

/*
 * The verify matmul on packed input, column by column: for each requested
 * column n = cols[j], unpack w[.][n] exactly, then for every row m
 *   Y[m][j] = sum_k X[m][k] * w[k]        (fp64, k ascending)
 *   A[m][j] = sum_k |X[m][k] * w[k]|      (the tolerance scale)
 * Ishizuki README, "Kernels written for the verify": each weight is decoded
 * once and multiplied against every drafted row.  The arithmetic per (m, n)
 * is exactly orc_gemm's on the unpacked matrix.
 */
void orc_verify(int fmt, const void* p0, const void* p1, const void* p2, int group,
                const double* X, int M, int K, const int64_t* cols, int64_t ncols, double* Y,
                double* A)
{
    double* w = (double*)malloc(sizeof(double) * (size_t)K);
    for (int64_t j = 0; j < ncols; j++) {
        orc_col(fmt, p0, p1, p2, K, group, (int)cols[j], w);
        for (int m = 0; m < M; m++) {
            const double* x = X + (int64_t)m * K;
            double acc = 0.0, aacc = 0.0;
            for (int k = 0; k < K; k++) {
                double t = x[k] * w[k];
                acc += t;
                aacc += fabs(t);
            }
            Y[(int64_t)m * ncols + j] = acc;
            if (A)
                A[(int64_t)m * ncols + j] = aacc;
        }
    }
    free(w);
}

/* ------------------------------------------------------------------------ */
/* Blockwise Walsh-Hadamard rotation                                          */

static int orc_popcount(unsigned v)
{
    int c = 0;
    while (v) {
        c += v & 1u;
        v >>= 1;
    }
    return c;
}

/*
 * x' = x_b . H128 / sqrt(128) for every 128-block b of a row of length `len`
 * (len % 128 == 0), with the Sylvester (natural-order) Hadamard matrix
 * H[i][j] = (-1)^popcount(i & j).  H is symmetric, so x_b . H = H . x_b.
 * An optional sign vector (bit k of signs[k/32] set: x_k is negated before
 * the rotation; NULL for none) gives the randomized form.
 * dflash-mlx-bonsai2 README, "What this fork adds" (fused sign, Hadamard
 * prep of the verify kernel); Ishizuki README (2-bit Hadamard-rotated weights).
 * The sum over j is exact in fp64 for fp16 or bf16 inputs; the one rounding
 * is the IEEE division by sqrt(128).
 */
void orc_fwht128(const double* x, int len, const uint32_t* signs, double* out)
{
    const double norm = sqrt(128.0);
    for (int b = 0; b < len / 128; b++) {
        double xs[128];
        for (int j = 0; j < 128; j++) {
            int k = b * 128 + j;
            double v = x[k];
            if (signs && ((signs[k / 32] >> (k % 32)) & 1))
                v = -v;
            xs[j] = v;
        }
        for (int i = 0; i < 128; i++) {
            double acc = 0.0;
            for (int j = 0; j < 128; j++)
                acc += (orc_popcount((unsigned)(i & j)) & 1) ? -xs[j] : xs[j];
            out[b * 128 + i] = acc / norm;
        }
    }
}
