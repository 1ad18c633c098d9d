/*
 * oracle/mx_ref.c -- the CPU oracle for the block-scaled FP8 GEMM.  TEST INFRASTRUCTURE ONLY:
 * the product path never links, loads or calls this file.  Only the tests, the package's smoke
 * check and the benchmark's CPU-baseline leg use it.
 *
 * What it computes.  The page "TIRx Layout API" (sections "示例：Blackwell Tensor Memory" and
 * "Scale Factor 布局") describes a block-scaled FP8 GEMM: the MMA reads, besides the FP8
 * operands, 8-bit scale factors, one per row of an operand and per block along K, which the
 * kernel keeps in tensor memory next to two accumulator stages.  The pages fix neither the
 * element formats nor the block length.  This oracle takes the plainest reading, the OCP
 * Microscaling (MX) formats that the tensor cores' mxf8f6f4 kind implements:
 *
 *   - elements: FP8 E4M3 (1 sign, 4 exponent bits with bias 7, 3 fraction bits; subnormals at
 *     exponent field 0; no infinities; S.1111.111 is NaN; largest finite value 448) or FP8 E5M2
 *     (1 sign, 5 exponent bits with bias 15, 2 fraction bits; subnormals at exponent field 0;
 *     exponent field 31 holds infinities and NaNs, as in IEEE 754);
 *   - scales: E8M0, an 8-bit biased exponent e standing for 2^(e - 127); e = 255 is NaN;
 *   - one scale per row and per block of 32 consecutive K elements.
 *
 * With A of shape M x K and B of shape N x K (row-major codes), SA of shape M x K/32 and SB of
 * shape N x K/32 (row-major scale codes):
 *
 *     D[i][j] = sum_{k < K} (a(A[i][k]) * s(SA[i][k/32])) * (b(B[j][k]) * s(SB[j][k/32]))
 *
 * Each factor a * s is exact in binary64 (at most 4 significant bits times a power of two
 * between 2^-127 and 2^127), and so is each product (at most 8 significant bits); the terms are
 * summed in binary64 in increasing k, with no blocking or reordering.  Alongside D the oracle
 * can return Dabs[i][j] = sum_k |term|, the scale of the rounding error any summation order can
 * make, which the parity bound uses.
 *
 * Nothing here is shared with the GPU path: no header, helper or table.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>

/* FP8 code -> binary64 value (exact).  fmt 0: E4M3, fmt 1: E5M2. */
double oracle_fp8_to_f64(uint8_t c, int fmt)
{
    const int sign = (c >> 7) & 1;
    double v;
    if (fmt == 0) {
        const int e = (c >> 3) & 0xF, f = c & 7;
        if (e == 0xF && f == 7) return NAN;
        if (e == 0) v = ldexp((double)f, -9);            /* f/8 * 2^(1-7) */
        else v = ldexp((double)(8 + f), e - 10);         /* (1 + f/8) * 2^(e-7) */
    } else {
        const int e = (c >> 2) & 0x1F, f = c & 3;
        if (e == 0x1F) {
            if (f != 0) return NAN;
            v = INFINITY;
        } else if (e == 0) {
            v = ldexp((double)f, -16);                   /* f/4 * 2^(1-15) */
        } else {
            v = ldexp((double)(4 + f), e - 17);          /* (1 + f/4) * 2^(e-15) */
        }
    }
    return sign ? -v : v;
}

/* E8M0 scale code -> 2^(e - 127); 255 is NaN. */
double oracle_e8m0_to_f64(uint8_t e)
{
    if (e == 0xFF) return NAN;
    return ldexp(1.0, (int)e - 127);
}

void oracle_decode_fp8(const uint8_t* c, double* out, int64_t n, int fmt)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_fp8_to_f64(c[i], fmt);
}

void oracle_decode_e8m0(const uint8_t* c, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_e8m0_to_f64(c[i]);
}

/* Rows of X (rows x K codes) with scales S (rows x K/32) -> scaled binary64 values. */
static void widen_scaled(const uint8_t* X, const uint8_t* S, double* out, int64_t rows,
                         int64_t K, int fmt)
{
    const int64_t KB = K / 32;
#pragma omp parallel for schedule(static)
    for (int64_t r = 0; r < rows; ++r)
        for (int64_t k = 0; k < K; ++k)
            out[r * K + k] = oracle_fp8_to_f64(X[r * K + k], fmt) *
                             oracle_e8m0_to_f64(S[r * KB + k / 32]);
}

static void dot2(const double* a, const double* b, int64_t K, double* sum, double* abs_sum)
{
    double s = 0.0, t = 0.0;
    for (int64_t k = 0; k < K; ++k) {
        const double p = a[k] * b[k];
        s += p;
        t += fabs(p);
    }
    *sum = s;
    *abs_sum = t;
}

/* D (M x N) and, if Dabs is not NULL, Dabs (M x N).  Returns -1 if K is not a multiple of 32,
 * -2 if the binary64 copies cannot be allocated, 0 otherwise. */
int oracle_gemm_mx_f64(const uint8_t* A, const uint8_t* B, const uint8_t* SA, const uint8_t* SB,
                       double* D, double* Dabs, int64_t M, int64_t N, int64_t K, int fmt_a,
                       int fmt_b)
{
    if (K % 32 != 0) return -1;
    double* a = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double* b = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!a || !b) {
        free(a);
        free(b);
        return -2;
    }
    widen_scaled(A, SA, a, M, K, fmt_a);
    widen_scaled(B, SB, b, N, K, fmt_b);
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double s, t;
            dot2(a + i * K, b + j * K, K, &s, &t);
            D[i * N + j] = s;
            if (Dabs) Dabs[i * N + j] = t;
        }
    free(a);
    free(b);
    return 0;
}

/* The same sums for `count` output elements (rows[t], cols[t]); out_abs may be NULL. */
int oracle_gemm_mx_f64_sampled(const uint8_t* A, const uint8_t* B, const uint8_t* SA,
                               const uint8_t* SB, int64_t M, int64_t N, int64_t K, int fmt_a,
                               int fmt_b, const int64_t* rows, const int64_t* cols,
                               int64_t count, double* out, double* out_abs)
{
    if (K % 32 != 0) return -1;
    const int64_t KB = K / 32;
    (void)M;
    (void)N;
#pragma omp parallel for schedule(static)
    for (int64_t t = 0; t < count; ++t) {
        const int64_t i = rows[t], j = cols[t];
        double s = 0.0, u = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            const double x = oracle_fp8_to_f64(A[i * K + k], fmt_a) *
                             oracle_e8m0_to_f64(SA[i * KB + k / 32]);
            const double y = oracle_fp8_to_f64(B[j * K + k], fmt_b) *
                             oracle_e8m0_to_f64(SB[j * KB + k / 32]);
            s += x * y;
            u += fabs(x * y);
        }
        out[t] = s;
        if (out_abs) out_abs[t] = u;
    }
    return 0;
}
