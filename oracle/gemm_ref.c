/*
 * oracle/gemm_ref.c -- the CPU oracle for D = A * B^T.  TEST INFRASTRUCTURE
 * ONLY: the product path never links, loads or calls this file.  Only the
 * tests, the package's smoke check and the benchmark's CPU-baseline leg use it.
 *
 * What it computes (page "TIRx 与高性能GEMM (上)", section "从 GEMM 公式到数据路径",
 * the formula D = A B^T with A of shape M x K and B of shape N x K, D of shape
 * M x N; and Step 3's index reading: a CTA's row band of D comes from a row band
 * of A, its column band from a row band of B):
 *
 *     D[i][j] = sum_{k < K} A[i][k] * B[j][k]
 *
 * A is M x K row-major, B is N x K row-major, both IEEE binary16.  Every input
 * is widened exactly to binary64 (every binary16 value is a binary64 value, and
 * a product of two binary16 values has at most 22 significant bits, so each
 * product is exact in binary64) and summed in binary64 in increasing k.  The
 * only rounding is the final binary64 sum; there is no blocking, tiling or
 * reordering.
 *
 * The same file holds the bfloat16 variants (inputs widened with a bfloat16 decoder, outputs
 * rounded with a bfloat16 round-to-nearest-even encoder) and the epilogue of a linear layer,
 * act(sum + bias), evaluated in binary64 before the single final rounding.
 *
 * The binary16 output value is round-to-nearest-even of that binary64 sum
 * (page "TIRx Compiler Foundation", section "Example: A GEMM Kernel": the
 * result is converted to FP16 with cvt.rn, i.e. round to nearest, ties to
 * even).  The encoder and decoder below are written from the IEEE 754 binary16
 * definition (1 sign bit, 5 exponent bits with bias 15, 10 fraction bits,
 * subnormals at exponent field 0, infinities and NaNs at exponent field 31).
 *
 * Nothing here is shared with the GPU path: no header, helper or table.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* binary16 bit pattern -> binary64 value (exact). */
double oracle_f16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int efield = (h >> 10) & 0x1f;
    const int frac = h & 0x3ff;
    double v;
    if (efield == 0) {
        /* subnormal or zero: frac * 2^-24 */
        v = ldexp((double)frac, -24);
    } else if (efield == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        /* normal: (1024 + frac) * 2^(efield - 15 - 10) */
        v = ldexp((double)(1024 + frac), efield - 25);
    }
    return sign ? -v : v;
}

/* binary64 value -> binary16 bit pattern, round to nearest, ties to even. */
uint16_t oracle_f64_to_f16(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7e00u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7c00u);
    if (a == 0.0) return sign;

    /* e = floor(log2(a)), clamped to the smallest normal exponent -14 so that
     * the subnormal range shares the spacing 2^-24. */
    int E;
    (void)frexp(a, &E);          /* a = f * 2^E with f in [0.5, 1) */
    int e = E - 1;
    if (e < -14) e = -14;
    if (e > 15) return (uint16_t)(sign | 0x7c00u);   /* a >= 65536 */

    /* Spacing of binary16 values in [2^e, 2^(e+1)) is q = 2^(e-10).
     * n = a / q is exact (power-of-two scaling) and below 2048. */
    const double n = ldexp(a, 10 - e);
    double r = floor(n);
    const double rem = n - r;    /* exact: n < 2^11 has few integer bits */
    if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;

    long ri = (long)r;           /* integer significand in units of q */
    if (ri == 0) return sign;    /* rounded down to zero */
    if (ri >= 2048) {            /* carried into the next binade */
        ri = 1024;
        e += 1;
    }
    if (ri < 1024) {
        /* only possible for e == -14: a subnormal */
        return (uint16_t)(sign | (uint16_t)ri);
    }
    const int efield = e + 15;
    if (efield >= 31) return (uint16_t)(sign | 0x7c00u);   /* overflow */
    return (uint16_t)(sign | (uint16_t)(efield << 10) | (uint16_t)(ri - 1024));
}

/* bfloat16 bit pattern -> binary64 value (exact): a bfloat16 value is the binary32 value whose
 * upper 16 bits are the pattern (1 sign bit, 8 exponent bits with bias 127, 7 fraction bits).
 * Written from that definition, field by field. */
double oracle_bf16_to_f64(uint16_t h)
{
    const int sign = (h >> 15) & 1;
    const int efield = (h >> 7) & 0xff;
    const int frac = h & 0x7f;
    double v;
    if (efield == 0) {
        v = ldexp((double)frac, -133);              /* subnormal: frac * 2^(-126-7) */
    } else if (efield == 255) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + frac), efield - 134);  /* (128 + frac) * 2^(e-127-7) */
    }
    return sign ? -v : v;
}

/* binary64 value -> bfloat16 bit pattern, round to nearest, ties to even (same method as the
 * binary16 encoder: scale by the spacing of the target binade, round the integer significand). */
uint16_t oracle_f64_to_bf16(double x)
{
    const uint16_t sign = signbit(x) ? 0x8000u : 0u;
    if (isnan(x)) return (uint16_t)(sign | 0x7fc0u);
    double a = fabs(x);
    if (isinf(a)) return (uint16_t)(sign | 0x7f80u);
    if (a == 0.0) return sign;
    int E;
    (void)frexp(a, &E);
    int e = E - 1;                       /* floor(log2 a) */
    if (e < -126) e = -126;              /* subnormals share the spacing 2^-133 */
    if (e > 127) return (uint16_t)(sign | 0x7f80u);
    const double n = ldexp(a, 7 - e);    /* in units of the spacing 2^(e-7); below 256 */
    double r = floor(n);
    const double rem = n - r;
    if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    long ri = (long)r;
    if (ri == 0) return sign;
    if (ri >= 256) {
        ri = 128;
        e += 1;
    }
    if (ri < 128) return (uint16_t)(sign | (uint16_t)ri);   /* subnormal (e == -126) */
    const int efield = e + 127;
    if (efield >= 255) return (uint16_t)(sign | 0x7f80u);
    return (uint16_t)(sign | (uint16_t)(efield << 7) | (uint16_t)(ri - 128));
}

/* Element decoders by type: 0 = binary16, 1 = bfloat16. */
static double decode_dt(uint16_t h, int dtype)
{
    return dtype == 1 ? oracle_bf16_to_f64(h) : oracle_f16_to_f64(h);
}

void oracle_decode_bf16(const uint16_t* h, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_bf16_to_f64(h[i]);
}

void oracle_round_bf16(const double* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_bf16(x[i]);
}

void oracle_decode_f16(const uint16_t* h, double* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f16_to_f64(h[i]);
}

void oracle_round_f16(const double* x, uint16_t* out, int64_t n)
{
    for (int64_t i = 0; i < n; ++i) out[i] = oracle_f64_to_f16(x[i]);
}

/* The dot product of two binary64 rows of length K, k increasing. */
static double dot(const double* a, const double* b, int64_t K)
{
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];
    return s;
}

/* Full product: D64[i*N + j] = sum_k A[i][k] * B[j][k] in binary64.
 * Step 1 widens A and B to binary64 (exact); step 2 takes one dot product per
 * output element.  Rows of D are independent and are spread over OpenMP
 * threads.  Returns 0, or -1 if the widened copies cannot be allocated. */
int oracle_gemm_f64(const uint16_t* A, const uint16_t* B, double* D,
                    int64_t M, int64_t N, int64_t K)
{
    double* a64 = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double* b64 = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!a64 || !b64) {
        free(a64);
        free(b64);
        return -1;
    }
    oracle_decode_f16(A, a64, M * K);
    oracle_decode_f16(B, b64, N * K);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            D[i * N + j] = dot(a64 + i * K, b64 + j * K, K);
    free(a64);
    free(b64);
    return 0;
}

/* Selected elements only: out[t] = D[rows[t]][cols[t]], each one the same
 * binary64 dot product as above with the two rows widened on the fly.  Used
 * where M*N*K is too large to compute every element on the host. */
void oracle_gemm_f64_sampled(const uint16_t* A, const uint16_t* B,
                             int64_t M, int64_t N, int64_t K,
                             const int64_t* rows, const int64_t* cols,
                             int64_t count, double* out)
{
    (void)M;
    (void)N;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < count; ++t) {
        const uint16_t* a = A + rows[t] * K;
        const uint16_t* b = B + cols[t] * K;
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k)
            s += oracle_f16_to_f64(a[k]) * oracle_f16_to_f64(b[k]);
        out[t] = s;
    }
}

/* The GEMM for either element type (0 = binary16, 1 = bfloat16): the same binary64 sum as
 * oracle_gemm_f64, inputs widened with the type's own decoder. */
int oracle_gemm_f64_dt(const uint16_t* A, const uint16_t* B, double* D, int64_t M, int64_t N,
                       int64_t K, int dtype)
{
    double* a64 = (double*)malloc(sizeof(double) * (size_t)(M * K > 0 ? M * K : 1));
    double* b64 = (double*)malloc(sizeof(double) * (size_t)(N * K > 0 ? N * K : 1));
    if (!a64 || !b64) {
        free(a64);
        free(b64);
        return -1;
    }
    for (int64_t i = 0; i < M * K; ++i) a64[i] = decode_dt(A[i], dtype);
    for (int64_t i = 0; i < N * K; ++i) b64[i] = decode_dt(B[i], dtype);
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j)
            D[i * N + j] = dot(a64 + i * K, b64 + j * K, K);
    free(a64);
    free(b64);
    return 0;
}

void oracle_gemm_f64_sampled_dt(const uint16_t* A, const uint16_t* B, int64_t M, int64_t N,
                                int64_t K, const int64_t* rows, const int64_t* cols,
                                int64_t count, double* out, int dtype)
{
    (void)M;
    (void)N;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < count; ++t) {
        const uint16_t* a = A + rows[t] * K;
        const uint16_t* b = B + cols[t] * K;
        double s = 0.0;
        for (int64_t k = 0; k < K; ++k) s += decode_dt(a[k], dtype) * decode_dt(b[k], dtype);
        out[t] = s;
    }
}

/* The fused epilogue of a linear layer, applied to binary64 sums in place:
 *     y = act(x + bias[j])          for element (i, j) of an M x N row-major array
 * bias: N elements of the given type, or null for none.  act: 0 none, 1 ReLU (max(y, 0)),
 * 2 GELU in its exact form y * Phi(y) = y/2 * (1 + erf(y / sqrt(2))), with erf from libm. */
void oracle_epilogue_f64(double* X, int64_t M, int64_t N, const uint16_t* bias, int dtype,
                         int act)
{
    const double inv_sqrt2 = 0.70710678118654752440084436210485;
#pragma omp parallel for schedule(static)
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double y = X[i * N + j];
            if (bias) y += decode_dt(bias[j], dtype);
            if (act == 1) y = y > 0.0 ? y : 0.0;
            else if (act == 2) y = 0.5 * y * (1.0 + erf(y * inv_sqrt2));
            X[i * N + j] = y;
        }
    }
}

/* Number of OpenMP threads a parallel region of this library uses. */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
