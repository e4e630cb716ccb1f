/*
 * oracle.c -- plain, slow, float64 CPU oracle for the weight-only quantized GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product library calls, links or
 * includes this file.  Only the test-suite, the package's smoke() check and the
 * benchmark's CPU-baseline leg may load it.  It shares no code, header, table or
 * constant with the CUDA path: every decode below is written out from the number
 * format's definition.
 *
 * What it computes (one definition per weight format):
 *
 *   out[m, n] = sum_k A[m, k] * w[n, k]            (float64, k ascending)
 *
 *   INT4 (W4A16):  w[n, k] = (q[n, k] - 8) * S[k / G, n]
 *       q is the 4-bit code; two codes per byte along K, the even k in the low
 *       nibble.  Source: "Low Bit Triton Kernels" (GPU MODE lecture 34), §03 core
 *       pattern: the gemlite-style BLOCK_K loop unpacks b_lo = (byte & 0xF) - 8 and
 *       b_hi = ((byte >> 4) & 0xF) - 8, looks up the group scale at
 *       s[k // GROUP_SIZE, n] and multiplies before the dot product.
 *
 *   FP8 (W8A16):   out[m, n] = alpha * sum_k A[m, k] * e4m3(W[n, k])  (+ bias[n])
 *       Source: "FlashInfer W8A16 GEMM (mm_bf16_fp8) analysis" (PR #7495),
 *       introduction: the per-tensor fp32 scale is applied to the fp32
 *       accumulator, no 16-bit weight copy is made.  The bias term follows the
 *       optional `bias` argument of mm_bf16_fp8 in §2 (public API).
 *
 *   INT4 codebook: w[n, k] = LUT[q[n, k]] * S[k / G, n]      (NF4-style, LUT an input)
 *       Source: "Low Bit Triton Kernels", the passage on choosing the 16 values of a
 *       4-bit weight (uniform INT4 / non-uniform NF4 / FP4) and NF4's table lookup.
 *
 *   INT2 (W2A16):  w[n, k] = (q[n, k] - 2) * S[k / G, n], four codes per byte
 *       Source: "Bitblas -- Mixed-Precision GEMM with the Ladder Compiler", hands-on
 *       sequence item 6 (W2A16); the layout and offset are the readings stated below.
 *
 *   FP4:           out[m, n] = alpha * sum_k A[m, k] * e2m1(W[n, k]) * e4m3(SF[n, k / 16])
 *       Source: "FlashInfer SM100 BF16 x FP4 GEMM" (PR #4466), §2: the weight is a
 *       uint8 [N, K/2] array (k = 2 * shape[1]) with one e4m3 scale factor per
 *       block of 16 along K (`sf_vec_size = block_size`) and a global alpha.
 *
 * Number formats, each decoded from its definition, not from a library:
 *   fp16  IEEE binary16 (1/5/10, bias 15, subnormals).
 *   bf16  bfloat16 (1/8/7, bias 127, subnormals).
 *   e4m3  OCP 8-bit E4M3 "FN": bias 7, subnormals, no infinities, S.1111.111 = NaN.
 *   e2m1  OCP MX 4-bit E2M1: bias 1, one subnormal (0.5), values 0..6.
 *
 * Every function is single-pass and plain.  OpenMP, when the compiler has it,
 * only spreads independent output columns over cores.
 */
#include <math.h>
#include <stdint.h>
#ifdef _OPENMP
#include <omp.h>
#endif
#include <stdlib.h>
#include <string.h>

#define ORACLE_API __attribute__((visibility("default")))

/* ---------------------------------------------------------------- formats */

/* IEEE binary16 bits -> value. */
ORACLE_API double oracle_f16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int m = h & 0x3ff;
    double v;
    if (e == 0)
        v = ldexp((double)m, -24);                 /* subnormal: m * 2^-24 */
    else if (e == 31)
        v = (m == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(1024 + m), e - 25);     /* 1.m * 2^(e-15) */
    return sign ? -v : v;
}

/* bfloat16 bits -> value. */
ORACLE_API double oracle_bf16_to_double(uint16_t b) {
    int sign = (b >> 15) & 1;
    int e = (b >> 7) & 0xff;
    int m = b & 0x7f;
    double v;
    if (e == 0)
        v = ldexp((double)m, -133);                /* m * 2^-126 * 2^-7 */
    else if (e == 255)
        v = (m == 0) ? INFINITY : NAN;
    else
        v = ldexp((double)(128 + m), e - 134);     /* 1.m * 2^(e-127) */
    return sign ? -v : v;
}

/* OCP E4M3 (FN variant) bits -> value. */
ORACLE_API double oracle_e4m3_to_double(uint8_t c) {
    int sign = (c >> 7) & 1;
    int e = (c >> 3) & 0xf;
    int m = c & 0x7;
    double v;
    if ((c & 0x7f) == 0x7f)
        return NAN;                                /* S.1111.111 */
    if (e == 0)
        v = ldexp((double)m, -9);                  /* 0.m * 2^-6 */
    else
        v = ldexp((double)(8 + m), e - 10);        /* 1.m * 2^(e-7) */
    return sign ? -v : v;
}

/* OCP MX E2M1 code (low 4 bits of c) -> value. */
ORACLE_API double oracle_e2m1_to_double(uint8_t c) {
    int sign = (c >> 3) & 1;
    int e = (c >> 1) & 0x3;
    int m = c & 0x1;
    double v;
    if (e == 0)
        v = 0.5 * m;                               /* 0.m * 2^0 */
    else
        v = ldexp((double)(2 + m), e - 2);         /* 1.m * 2^(e-1) */
    return sign ? -v : v;
}

/* Round-to-nearest-even of a finite double into a binary format with
 * `mbits` stored mantissa bits, exponent bias `bias` and maximum biased
 * exponent `emax_field` (all-ones is inf/NaN).  Overflow gives infinity.
 * Returns the encoded bits (sign in bit mbits+ebits). */
static uint32_t round_to_format(double x, int mbits, int ebits, int bias) {
    uint32_t sign = signbit(x) ? 1u : 0u;
    uint32_t sign_bit = sign << (mbits + ebits);
    uint32_t inf_bits = ((1u << ebits) - 1u) << mbits;
    double a = fabs(x);
    if (isnan(x))
        return sign_bit | inf_bits | (1u << (mbits - 1));
    if (a == 0.0)
        return sign_bit;
    if (isinf(a))
        return sign_bit | inf_bits;
    int E;
    frexp(a, &E);                  /* a = f * 2^E, f in [0.5, 1) */
    int e = E - 1;                 /* a in [2^e, 2^(e+1)) */
    int emin = 1 - bias;           /* smallest normal exponent */
    int qexp = (e < emin) ? (emin - mbits) : (e - mbits);   /* quantum = 2^qexp */
    double q = ldexp(a, -qexp);    /* exact: scaling by a power of two */
    double fl = floor(q);
    double diff = q - fl;
    double n = fl;
    if (diff > 0.5 || (diff == 0.5 && fmod(fl, 2.0) != 0.0))
        n = fl + 1.0;
    /* n * 2^qexp is the rounded magnitude. */
    uint64_t ni = (uint64_t)n;
    if (e < emin) {
        /* subnormal range; n == 2^mbits lands exactly on the smallest normal */
        return sign_bit | (uint32_t)ni;
    }
    if (ni == (1ull << (mbits + 1))) {   /* rounding carried into the next binade */
        ni >>= 1;
        e += 1;
    }
    int field = e + bias;
    if (field >= (1 << ebits) - 1)
        return sign_bit | inf_bits;
    return sign_bit | ((uint32_t)field << mbits) | (uint32_t)(ni - (1ull << mbits));
}

/* RN16: round-to-nearest-even to IEEE binary16, returned as bits. */
ORACLE_API uint16_t oracle_round_f16(double x) { return (uint16_t)round_to_format(x, 10, 5, 15); }

/* RN_bf: round-to-nearest-even to bfloat16, returned as bits. */
ORACLE_API uint16_t oracle_round_bf16(double x) { return (uint16_t)round_to_format(x, 7, 8, 127); }

static double act_value(const uint16_t* A, int a_is_bf16, int64_t idx) {
    return a_is_bf16 ? oracle_bf16_to_double(A[idx]) : oracle_f16_to_double(A[idx]);
}

/* The activation rows a GEMM reads, decoded once: row i of the result holds
 * A[rows[i], 0..K-1] (rows NULL: all M rows) as float64.  Only the decoding moves
 * out of the dot products; every product and every k-ascending sum below is the
 * same.  The caller frees the array. */
static double* act_rows(const uint16_t* A, int a_is_bf16, int64_t M, int64_t K, const int64_t* rows,
                        int64_t nrows) {
    double* ad = (double*)malloc(sizeof(double) * (size_t)(nrows * K > 0 ? nrows * K : 1));
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < nrows; ++i) {
        const int64_t m = rows ? rows[i] : i;
        for (int64_t k = 0; k < K; ++k) ad[i * K + k] = act_value(A, a_is_bf16, m * K + k);
    }
    (void)M;
    return ad;
}

/* ---------------------------------------------------------------- INT4 */

/* Canonical packing: byte (n, j) holds code q[n, 2j] in its low nibble and
 * q[n, 2j+1] in its high nibble.  q values must lie in 0..15. */
ORACLE_API void oracle_pack_int4(const uint8_t* q, int64_t N, int64_t K, uint8_t* w) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / 2; ++j) {
            uint8_t lo = q[n * K + 2 * j] & 0xF;
            uint8_t hi = q[n * K + 2 * j + 1] & 0xF;
            w[n * (K / 2) + j] = (uint8_t)(lo | (hi << 4));
        }
}

/* Inverse of the canonical packing. */
ORACLE_API void oracle_unpack_int4(const uint8_t* w, int64_t N, int64_t K, uint8_t* q) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) {
            uint8_t byte = w[n * (K / 2) + k / 2];
            q[n * K + k] = (k % 2 == 0) ? (byte & 0xF) : ((byte >> 4) & 0xF);
        }
}

/* Synthetic group-wise symmetric INT4 quantiser, the step upstream of the packing
 * ("Low Bit Triton Kernels", hands-on exercise 1: fp16 weight -> group-wise
 * quantize -> two nibbles per byte, checked by a round trip).  The page fixes no
 * scale rule; the reading taken is the symmetric one whose largest magnitude maps
 * to +-7:
 *   amax = max_{k in group} |W[n, k]|,   S[g, n] = RN16(amax / 7)
 *   q = clamp(rint(W[n, k] / S) + 8, 0, 15)          (rint: half to even)
 * with q = 8 throughout a group whose scale is 0.  The decisions are taken in fp32
 * (IEEE division, round half to even), the precision of the GPU kernel; both are
 * equal to the exact rational roundings: amax / 7 is never within fp32 rounding of
 * an fp16 tie, and W / S is either exactly a tie (representable) or ~3e-5 away.
 * W fp16 bits [N][K]; outputs: canonical packed codes [N][K/2] (even k in the low
 * nibble) and fp16 scale bits [K/G][N]. */
ORACLE_API void oracle_quantize_int4(const uint16_t* w_f16, int64_t N, int64_t K, int64_t G, uint8_t* w,
                                     uint16_t* s) {
    memset(w, 0, (size_t)(N * (K / 2)));
    for (int64_t n = 0; n < N; ++n)
        for (int64_t g = 0; g < K / G; ++g) {
            double amax = 0.0;
            for (int64_t k = g * G; k < (g + 1) * G; ++k) {
                const double a = fabs(oracle_f16_to_double(w_f16[n * K + k]));
                if (a > amax) amax = a;
            }
            const float amax32 = (float)amax;                     /* exact: an fp16 value */
            const uint16_t sb = oracle_round_f16((double)(amax32 / 7.0f));
            s[g * N + n] = sb;
            const float sv = (float)oracle_f16_to_double(sb);
            for (int64_t k = g * G; k < (g + 1) * G; ++k) {
                int q = 8;
                if (sv != 0.0f) {
                    const float x = (float)oracle_f16_to_double(w_f16[n * K + k]) / sv;
                    q = (int)rintf(x) + 8;
                    if (q < 0) q = 0;
                    if (q > 15) q = 15;
                }
                w[n * (K / 2) + k / 2] |= (uint8_t)((k % 2 == 0) ? q : (q << 4));
            }
        }
}

/* The 4-bit code of weight (n, k) in the canonical packing [N][K/2]. */
static int int4_code(const uint8_t* w, int64_t K, int64_t n, int64_t k) {
    uint8_t byte = w[n * (K / 2) + k / 2];
    int q = (k % 2 == 0) ? (byte & 0xF) : ((byte >> 4) & 0xF);
    return q;
}

/* One dequantized INT4 weight: (q - 8) * S[k / G, n], S fp16 [K/G][N]. */
static double int4_weight(const uint8_t* w, const uint16_t* s, int64_t N, int64_t K, int64_t G,
                          int64_t n, int64_t k) {
    int q = int4_code(w, K, n, k);
    int64_t g = k / G;
    double scale = oracle_f16_to_double(s[g * N + n]);
    return (double)(q - 8) * scale;
}

/* Dequantized weight as fp32, w_f32[n][k].  (q-8)*s has at most 4 + 11
 * significant bits, so the fp32 value is the exact product. */
ORACLE_API void oracle_dequant_int4(const uint8_t* w, const uint16_t* s, int64_t N, int64_t K,
                                    int64_t G, float* out) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = (float)int4_weight(w, s, N, K, G, n, k);
}

/* Asymmetric INT4 (zero point per group and row): (q - Z[k / G, n]) * S[k / G, n],
 * Z uint8 [K/G][N] holding integers 0..15.  The pages name group-scaled 4-bit formats
 * with zero points (GPTQ / AWQ / HQQ, "Low Bit Triton Kernels" §02) but print none;
 * the integer zero point is the reading taken. */
static double int4_weight_zp(const uint8_t* w, const uint16_t* s, const uint8_t* z, int64_t N, int64_t K,
                             int64_t G, int64_t n, int64_t k) {
    int q = int4_code(w, K, n, k);
    int64_t grp = k / G;
    double scale = oracle_f16_to_double(s[grp * N + n]);
    int zero = z[grp * N + n];
    return (double)(q - zero) * scale;
}

ORACLE_API void oracle_dequant_int4_zp(const uint8_t* w, const uint16_t* s, const uint8_t* z, int64_t N, int64_t K,
                                       int64_t G, float* out) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = (float)int4_weight_zp(w, s, z, N, K, G, n, k);
}

ORACLE_API void oracle_gemm_w4a16_zp(const uint16_t* A, int a_is_bf16, const uint8_t* w, const uint16_t* s,
                                     const uint8_t* z, int64_t M, int64_t N, int64_t K, int64_t G,
                                     const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                                     double* out) {
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    double* ad = act_rows(A, a_is_bf16, M, K, rows, nrows);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < ncols; ++j) {
        const int64_t n = cols ? cols[j] : j;
        double* wrow = (double*)malloc((size_t)K * sizeof(double));
        for (int64_t k = 0; k < K; ++k) wrow[k] = int4_weight_zp(w, s, z, N, K, G, n, k);
        for (int64_t i = 0; i < nrows; ++i) {
            const double* arow = ad + i * K;
            double dot = 0.0;
            for (int64_t k = 0; k < K; ++k) dot += wrow[k] * arow[k];
            out[i * ncols + j] = dot;
        }
        free(wrow);
    }
    free(ad);
}

/* out[i][j] = sum_k A[rows[i], k] * w[cols[j], k].  rows/cols may be NULL
 * (all rows / all columns); out is [nrows][ncols] float64. */
ORACLE_API void oracle_gemm_w4a16(const uint16_t* A, int a_is_bf16, const uint8_t* w,
                                  const uint16_t* s, int64_t M, int64_t N, int64_t K, int64_t G,
                                  const int64_t* rows, int64_t nrows, const int64_t* cols,
                                  int64_t ncols, double* out) {
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    double* ad = act_rows(A, a_is_bf16, M, K, rows, nrows);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < ncols; ++j) {
        int64_t n = cols ? cols[j] : j;
        double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
        for (int64_t k = 0; k < K; ++k)
            wrow[k] = int4_weight(w, s, N, K, G, n, k);
        for (int64_t i = 0; i < nrows; ++i) {
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += ad[i * K + k] * wrow[k];
            out[i * ncols + j] = acc;
        }
        free(wrow);
    }
    free(ad);
}

/* ---------------------------------------------------------------- INT4 codebook */

/* Non-uniform 4-bit format: the code picks one of 16 fp16 codebook values, which
 * the group scale then multiplies ("Low Bit Triton Kernels", the passage on how
 * the 16 values of a 4-bit weight are chosen -- a uniform grid (INT4), a
 * non-uniform one (NF4) or a floating-point one (FP4) -- and on NF4's dequant
 * being a table lookup held in registers).  The page prints no table, so the
 * codebook is an input:
 *   w[n, k] = LUT[q[n, k]] * S[k / G, n]      LUT fp16 [16], S fp16 [K/G][N]
 * with the codes in the canonical INT4 packing.  LUT[q] * S has at most 11 + 11
 * significant bits and stays inside the fp32 range, so its fp32 value is exact. */
static double lut4_weight(const uint8_t* w, const uint16_t* s, const uint16_t* lut, int64_t N, int64_t K,
                          int64_t G, int64_t n, int64_t k) {
    int code = int4_code(w, K, n, k);
    double entry = oracle_f16_to_double(lut[code]);
    double scale = oracle_f16_to_double(s[(k / G) * N + n]);
    return entry * scale;
}

ORACLE_API void oracle_dequant_int4_lut(const uint8_t* w, const uint16_t* s, const uint16_t* lut, int64_t N,
                                        int64_t K, int64_t G, float* out) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = (float)lut4_weight(w, s, lut, N, K, G, n, k);
}

ORACLE_API void oracle_gemm_w4a16_lut(const uint16_t* A, int a_is_bf16, const uint8_t* w, const uint16_t* s,
                                      const uint16_t* lut, int64_t M, int64_t N, int64_t K, int64_t G,
                                      const int64_t* rows, int64_t nrows, const int64_t* cols, int64_t ncols,
                                      double* out) {
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    double* ad = act_rows(A, a_is_bf16, M, K, rows, nrows);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < ncols; ++j) {
        const int64_t n = cols ? cols[j] : j;
        double* wv = (double*)malloc((size_t)K * sizeof(double));
        for (int64_t k = 0; k < K; ++k) wv[k] = lut4_weight(w, s, lut, N, K, G, n, k);
        for (int64_t i = 0; i < nrows; ++i) {
            double sum = 0.0;
            for (int64_t k = 0; k < K; ++k) sum += ad[K * i + k] * wv[k];
            out[i * ncols + j] = sum;
        }
        free(wv);
    }
    free(ad);
}

/* ---------------------------------------------------------------- INT2 */

/* W2A16: 2-bit codes ("Bitblas -- Mixed-Precision GEMM with the Ladder Compiler",
 * hands-on sequence item 6: the W2A16 (INT2 weight) dtype combination, its
 * accuracy loss and its speed-up).  The page gives no formula; the reading taken
 * follows the INT4 format one size down: four codes per byte along K, code k at
 * bits 2 (k % 4) .. 2 (k % 4) + 1 (the smallest k in the lowest bits), symmetric
 * offset 2 (half the code range, as 8 is for INT4) and fp16 group scales:
 *   w[n, k] = (q[n, k] - 2) * S[k / G, n]                 q in 0..3 */
ORACLE_API void oracle_pack_int2(const uint8_t* q, int64_t N, int64_t K, uint8_t* w) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t j = 0; j < K / 4; ++j) {
            uint8_t byte = 0;
            for (int i = 0; i < 4; ++i) byte |= (uint8_t)((q[n * K + 4 * j + i] & 0x3) << (2 * i));
            w[n * (K / 4) + j] = byte;
        }
}

static int int2_code(const uint8_t* w, int64_t K, int64_t n, int64_t k) {
    uint8_t byte = w[n * (K / 4) + k / 4];
    return (byte >> (2 * (k % 4))) & 0x3;
}

ORACLE_API void oracle_unpack_int2(const uint8_t* w, int64_t N, int64_t K, uint8_t* q) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) q[n * K + k] = (uint8_t)int2_code(w, K, n, k);
}

static double int2_weight(const uint8_t* w, const uint16_t* s, int64_t N, int64_t K, int64_t G, int64_t n,
                          int64_t k) {
    int q = int2_code(w, K, n, k);
    double scale = oracle_f16_to_double(s[(k / G) * N + n]);
    return (double)(q - 2) * scale;
}

/* (q - 2) * s has at most 2 + 11 significant bits: the fp32 value is exact. */
ORACLE_API void oracle_dequant_int2(const uint8_t* w, const uint16_t* s, int64_t N, int64_t K, int64_t G,
                                    float* out) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k) out[n * K + k] = (float)int2_weight(w, s, N, K, G, n, k);
}

ORACLE_API void oracle_gemm_w2a16(const uint16_t* A, int a_is_bf16, const uint8_t* w, const uint16_t* s,
                                  int64_t M, int64_t N, int64_t K, int64_t G, const int64_t* rows, int64_t nrows,
                                  const int64_t* cols, int64_t ncols, double* out) {
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    double* ad = act_rows(A, a_is_bf16, M, K, rows, nrows);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < ncols; ++j) {
        const int64_t n = cols ? cols[j] : j;
        double* wv = (double*)malloc((size_t)K * sizeof(double));
        for (int64_t k = 0; k < K; ++k) wv[k] = int2_weight(w, s, N, K, G, n, k);
        for (int64_t i = 0; i < nrows; ++i) {
            const double* xa = ad + i * K;
            double total = 0.0;
            for (int64_t k = 0; k < K; ++k) total += wv[k] * xa[k];
            out[i * ncols + j] = total;
        }
        free(wv);
    }
    free(ad);
}

/* ---------------------------------------------------------------- FP8 */

/* Dequantized FP8 weight (without the per-tensor scale), w_f32[n][k]. */
ORACLE_API void oracle_dequant_fp8(const uint8_t* w, int64_t N, int64_t K, float* out) {
    for (int64_t i = 0; i < N * K; ++i)
        out[i] = (float)oracle_e4m3_to_double(w[i]);
}

/* out[i][j] = alpha * sum_k A[m, k] * e4m3(W[n, k]) + bias[n].
 * bias (same 16-bit type as A) may be NULL. */
ORACLE_API void oracle_gemm_w8a16_fp8(const uint16_t* A, int a_is_bf16, const uint8_t* w,
                                      double alpha, const uint16_t* bias, int64_t M, int64_t N,
                                      int64_t K, const int64_t* rows, int64_t nrows,
                                      const int64_t* cols, int64_t ncols, double* out) {
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    double* ad = act_rows(A, a_is_bf16, M, K, rows, nrows);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < ncols; ++j) {
        int64_t n = cols ? cols[j] : j;
        double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
        for (int64_t k = 0; k < K; ++k)
            wrow[k] = oracle_e4m3_to_double(w[n * K + k]);
        double b = bias ? act_value(bias, a_is_bf16, n) : 0.0;
        for (int64_t i = 0; i < nrows; ++i) {
            const double* a8 = ad + i * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += a8[k] * wrow[k];
            out[i * ncols + j] = alpha * acc + b;
        }
        free(wrow);
    }
    free(ad);
}

/* ---------------------------------------------------------------- FP4 */

/* One FP4 weight: e2m1(code) * e4m3(SF[n, k/16]); code k even in the low nibble. */
static double fp4_weight(const uint8_t* w, const uint8_t* sf, int64_t K, int64_t n, int64_t k) {
    uint8_t byte = w[n * (K / 2) + k / 2];
    uint8_t code = (k % 2 == 0) ? (byte & 0xF) : ((byte >> 4) & 0xF);
    double sfv = oracle_e4m3_to_double(sf[n * (K / 16) + k / 16]);
    return oracle_e2m1_to_double(code) * sfv;
}

/* Dequantized FP4 weight with its block scale (without alpha), w_f32[n][k]. */
ORACLE_API void oracle_dequant_fp4(const uint8_t* w, const uint8_t* sf, int64_t N, int64_t K,
                                   float* out) {
    for (int64_t n = 0; n < N; ++n)
        for (int64_t k = 0; k < K; ++k)
            out[n * K + k] = (float)fp4_weight(w, sf, K, n, k);
}

/* out[i][j] = alpha * sum_k A[m, k] * e2m1(W[n, k]) * e4m3(SF[n, k/16]); A is bf16. */
ORACLE_API void oracle_gemm_bf16_fp4(const uint16_t* A, const uint8_t* w, const uint8_t* sf,
                                     double alpha, int64_t M, int64_t N, int64_t K,
                                     const int64_t* rows, int64_t nrows, const int64_t* cols,
                                     int64_t ncols, double* out) {
    if (!rows) nrows = M;
    if (!cols) ncols = N;
    double* ad = act_rows(A, 1, M, K, rows, nrows);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t j = 0; j < ncols; ++j) {
        int64_t n = cols ? cols[j] : j;
        double* wrow = (double*)malloc(sizeof(double) * (size_t)K);
        for (int64_t k = 0; k < K; ++k)
            wrow[k] = fp4_weight(w, sf, K, n, k);
        for (int64_t i = 0; i < nrows; ++i) {
            const double* a4 = ad + i * K;
            double acc = 0.0;
            for (int64_t k = 0; k < K; ++k)
                acc += a4[k] * wrow[k];
            out[i * ncols + j] = alpha * acc;
        }
        free(wrow);
    }
    free(ad);
}

/* Number of OpenMP threads the GEMM loops use (1 without OpenMP). */
ORACLE_API int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- arrays */

ORACLE_API void oracle_f16_array_to_double(const uint16_t* h, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_double(h[i]);
}

ORACLE_API void oracle_bf16_array_to_double(const uint16_t* b, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_double(b[i]);
}

ORACLE_API void oracle_round_f16_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_f16(x[i]);
}

ORACLE_API void oracle_round_bf16_array(const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_round_bf16(x[i]);
}
