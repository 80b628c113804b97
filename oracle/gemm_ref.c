/*
 * gemm_ref.c -- CPU oracle for the dense matrix multiply C[m,n] = sum_k A[m,k]*B[k,n].
 *
 * TEST INFRASTRUCTURE.  This is the independent reference the CUDA library is
 * checked against.  Only the tests, the smoke check and the benchmark's CPU
 * baseline leg load it; the library never does.  It shares no code, header,
 * table or helper with the CUDA path: the number formats are decoded and
 * encoded here from their IEEE 754 / bfloat16 bit layouts, not with any CUDA
 * conversion.
 *
 * Definition followed.  "Matrix multiplication: reuse the inputs"
 * (buicongnguyen.github.io/triton-cuda-lab, lesson 6), section "The three
 * dimensions have different jobs": A is [M,K], B is [K,N], C is [M,N] and
 * C[row,col] is the sum over `inner` of A[row,inner]*B[inner,col], computed
 * first as a plain three-loop CPU version.  Here the sum is carried in IEEE
 * double, term by term in increasing `inner` (k) order, starting from zero.
 * Every product of two f16, bf16, f32 or FP8 (E4M3 / E5M2) values is exact in
 * double (at most 24+24 significand bits), so the only rounding is the double
 * addition.
 *
 * Alongside C the oracle returns S[m,n] = sum_k |A[m,k]*B[k,n]|, the scale that
 * the floating-point tolerance is stated against.
 *
 * The row loop is split across OpenMP threads (each output row is independent;
 * the per-element summation order is unchanged).
 */
#include <math.h>
#include <stdint.h>
#include <stddef.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* Operand / result format tags (the oracle's own numbering). */
enum { ORC_F16 = 0, ORC_BF16 = 1, ORC_F32 = 2, ORC_E4M3 = 3, ORC_E5M2 = 4 };

static int fmt_bytes(int fmt)
{
    switch (fmt) {
    case ORC_F16: case ORC_BF16: return 2;
    case ORC_F32: return 4;
    case ORC_E4M3: case ORC_E5M2: return 1;
    default: return 0;
    }
}

int orc_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* ---------------------------------------------------------------- decode --
 * binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits.
 * binary32: 1 sign bit, 8 exponent bits (bias 127), 23 fraction bits.
 * A field of all ones is Inf (fraction 0) or NaN; a zero exponent field is a
 * subnormal with value fraction * 2^(1 - bias - fraction_bits).
 */
static double decode_bits(uint32_t w, int exp_bits, int frac_bits)
{
    const uint32_t frac_mask = (1u << frac_bits) - 1u;
    const uint32_t exp_mask = (1u << exp_bits) - 1u;
    const int bias = (1 << (exp_bits - 1)) - 1;
    const int sign = (int)((w >> (exp_bits + frac_bits)) & 1u);
    const uint32_t e = (w >> frac_bits) & exp_mask;
    const uint32_t f = w & frac_mask;
    double v;
    if (e == exp_mask)
        v = f ? NAN : INFINITY;
    else if (e == 0)
        v = ldexp((double)f, 1 - bias - frac_bits);
    else
        v = ldexp((double)(f | (1u << frac_bits)), (int)e - bias - frac_bits);
    return sign ? -v : v;
}

/* 8-bit floating point, the OCP FP8 formats (OCP 8-bit Floating Point
 * Specification, 2023):
 *   E5M2: 1 sign, 5 exponent bits (bias 15), 2 fraction bits, IEEE-like (an
 *         all-ones exponent is Inf or NaN) -- decode_bits applies as is.
 *   E4M3: 1 sign, 4 exponent bits (bias 7), 3 fraction bits, NO infinities:
 *         the all-ones exponent is an ordinary binade except for fraction 111,
 *         the only NaN (S.1111.111), so the largest finite value is
 *         1.75 * 2^8 = 448.
 */
static double decode_e4m3(uint32_t w)
{
    const int sign = (int)((w >> 7) & 1u);
    const uint32_t e = (w >> 3) & 0xFu;
    const uint32_t f = w & 7u;
    double v;
    if (e == 0xFu && f == 7u)
        v = NAN;
    else if (e == 0)
        v = ldexp((double)f, 1 - 7 - 3);
    else
        v = ldexp((double)(f | 8u), (int)e - 7 - 3);
    return sign ? -v : v;
}

double orc_decode_one(int fmt, uint32_t bits)
{
    switch (fmt) {
    case ORC_F16: return decode_bits(bits & 0xFFFFu, 5, 10);
    case ORC_BF16: return decode_bits(bits & 0xFFFFu, 8, 7);
    case ORC_F32: return decode_bits(bits, 8, 23);
    case ORC_E4M3: return decode_e4m3(bits & 0xFFu);
    case ORC_E5M2: return decode_bits(bits & 0xFFu, 5, 2);
    default: return NAN;
    }
}

static uint32_t load_bits(int fmt, const void *src, int64_t i)
{
    switch (fmt_bytes(fmt)) {
    case 1: return ((const uint8_t *)src)[i];
    case 2: return ((const uint16_t *)src)[i];
    default: return ((const uint32_t *)src)[i];
    }
}

/* Decode a rows x cols block with leading dimension `ld` (elements) into a
 * dense rows x cols double array.  Returns 0, or -1 on an unknown format. */
int orc_decode(int fmt, const void *src, int64_t rows, int64_t cols, int64_t ld, double *dst)
{
    if (fmt_bytes(fmt) == 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r) {
        for (int64_t c = 0; c < cols; ++c)
            dst[r * cols + c] = orc_decode_one(fmt, load_bits(fmt, src, r * ld + c));
    }
    return 0;
}

/* ---------------------------------------------------------------- encode --
 * Round a double to the nearest value of the target format, ties to even
 * (IEEE 754 roundTiesToEven), and return its bit pattern.  A magnitude that
 * rounds to 2^(emax+1) or beyond becomes Inf.  NaN becomes the canonical quiet
 * NaN with the input's sign.
 */
static uint32_t encode_bits(double x, int exp_bits, int frac_bits)
{
    const int bias = (1 << (exp_bits - 1)) - 1;
    const int emin = 1 - bias, emax = bias;
    const uint32_t exp_all = ((1u << exp_bits) - 1u) << frac_bits;
    const uint32_t sign = signbit(x) ? (1u << (exp_bits + frac_bits)) : 0u;
    if (isnan(x))
        return sign | exp_all | (1u << (frac_bits - 1));
    double ax = fabs(x);
    if (isinf(ax))
        return sign | exp_all;
    if (ax == 0.0)
        return sign;
    int E;
    (void)frexp(ax, &E);                 /* ax = m * 2^E, 0.5 <= m < 1 */
    int e = E - 1;                       /* exponent of the leading bit */
    if (e < emin)
        e = emin;                        /* subnormal range: fixed quantum */
    const double quantum = ldexp(1.0, e - frac_bits);
    const double v = rint(ax / quantum) * quantum; /* ax/quantum is exact; rint = ties-to-even */
    if (v >= ldexp(1.0, emax + 1))
        return sign | exp_all;
    if (v < ldexp(1.0, emin))            /* subnormal or zero */
        return sign | (uint32_t)(v / ldexp(1.0, emin - frac_bits));
    (void)frexp(v, &E);
    e = E - 1;
    const uint32_t frac = (uint32_t)(v / ldexp(1.0, e - frac_bits)) - (1u << frac_bits);
    return sign | ((uint32_t)(e + bias) << frac_bits) | frac;
}

/* E4M3 round to nearest, ties to even.  Rounding works as in encode_bits
 * with the top binade (2^8) ordinary; a magnitude that rounds to 480 or more
 * (the would-be code S.1111.111) has no finite encoding and becomes the NaN
 * S.1111.111 (there is no Inf). */
static uint32_t encode_e4m3(double x)
{
    const uint32_t sign = signbit(x) ? 0x80u : 0u;
    if (isnan(x))
        return sign | 0x7Fu;
    const double ax = fabs(x);
    if (isinf(ax))
        return sign | 0x7Fu;
    if (ax == 0.0)
        return sign;
    int E;
    (void)frexp(ax, &E);
    int e = E - 1;
    if (e < -6)
        e = -6;                            /* subnormal range: quantum 2^-9 */
    const double quantum = ldexp(1.0, e - 3);
    const double v = rint(ax / quantum) * quantum;
    if (v >= 480.0)
        return sign | 0x7Fu;
    if (v < ldexp(1.0, -6))
        return sign | (uint32_t)(v / ldexp(1.0, -9));
    (void)frexp(v, &E);
    e = E - 1;
    const uint32_t frac = (uint32_t)(v / ldexp(1.0, e - 3)) - 8u;
    return sign | ((uint32_t)(e + 7) << 3) | frac;
}

uint32_t orc_encode_one(int fmt, double x)
{
    switch (fmt) {
    case ORC_F16: return encode_bits(x, 5, 10);
    case ORC_BF16: return encode_bits(x, 8, 7);
    case ORC_F32: return encode_bits(x, 8, 23);
    case ORC_E4M3: return encode_e4m3(x);
    case ORC_E5M2: return encode_bits(x, 5, 2);
    default: return 0;
    }
}

/* Encode n doubles into the bit patterns of `fmt` (uint16 or uint32 elements). */
int orc_encode(int fmt, const double *src, int64_t n, void *dst)
{
    const int nb = fmt_bytes(fmt);
    if (nb == 0)
        return -1;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < n; ++i) {
        uint32_t w = orc_encode_one(fmt, src[i]);
        if (nb == 4)
            ((uint32_t *)dst)[i] = w;
        else if (nb == 2)
            ((uint16_t *)dst)[i] = (uint16_t)w;
        else
            ((uint8_t *)dst)[i] = (uint8_t)w;
    }
    return 0;
}

/* ------------------------------------------------------------------ gemm --
 * For each selected row i of A (all M rows when `rows` is NULL, otherwise the
 * `nrows` indices in `rows`), output row r of C and S is
 *     C[r, j] = sum_{k=0}^{K-1} A[i,k] * B[k,j]
 *     S[r, j] = sum_{k=0}^{K-1} |A[i,k] * B[k,j]|
 * summed in double in increasing k.  A is dense [M,lda], B dense [K,ldb],
 * C and S dense [nrows, ldc]; S may be NULL.  The loops run i, k, j: for every
 * (i, j) the terms are still added in k order, so this is the three-loop
 * definition with the two inner loops swapped for cache locality only.
 * K == 0 gives the empty sum, 0.  Returns 0, or -1 on bad arguments.
 */
int orc_gemm(int64_t M, int64_t N, int64_t K,
             const double *A, int64_t lda, const double *B, int64_t ldb,
             const int64_t *rows, int64_t nrows,
             double *C, double *S, int64_t ldc)
{
    if (M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N)
        return -1;
    const int64_t nr = rows ? nrows : M;
    for (int64_t r = 0; rows && r < nr; ++r)
        if (rows[r] < 0 || rows[r] >= M)
            return -1;
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t r = 0; r < nr; ++r) {
        const int64_t i = rows ? rows[r] : r;
        double *c = C + r * ldc;
        double *s = S ? S + r * ldc : NULL;
        for (int64_t j = 0; j < N; ++j) {
            c[j] = 0.0;
            if (s)
                s[j] = 0.0;
        }
        for (int64_t k = 0; k < K; ++k) {
            const double a = A[i * lda + k];
            const double *b = B + k * ldb;
            if (s) {
                for (int64_t j = 0; j < N; ++j) {
                    const double p = a * b[j];
                    c[j] += p;
                    s[j] += fabs(p);
                }
            } else {
                for (int64_t j = 0; j < N; ++j)
                    c[j] += a * b[j];
            }
        }
    }
    return 0;
}
