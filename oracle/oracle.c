/*
 * oracle.c -- plain, slow, obviously correct CPU reference for dense GEMM.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing on the product path may link, load or
 * call this file.  Only the test suite, the smoke check and the benchmark's
 * CPU-baseline leg use it.  It shares no code, header, table or constant with
 * the CUDA library.
 *
 * What it computes is the plain definition of the product, accumulated in
 * binary64 in plain k order:
 *
 *     C[m][n] = sum_{k < K} a(m, k) * b(k, n)
 *
 * ("Optimizing GEMM in HIP", section "GEMM fundamentals": an M x K matrix A
 * times a K x N matrix B gives the M x N matrix C; the CPU form is three
 * nested loops, one multiply-add per iteration, 2MNK operations.)
 *
 * Storage layouts follow the pages:
 *   - "TN" ("FP16 GEMM Optimization on AMD RDNA 3 and RDNA 4", section
 *     "What We Are Computing"): A row-major, a(m,k) = A[m*lda + k];
 *     B column-major, b(k,n) = B[n*ldb + k]; C column-major, C[n*ldc + m].
 *   - FP32 ("Optimizing GEMM in HIP", Step 1, the naive kernel's indexing):
 *     everything row-major, a(m,k) = A[m*lda + k], b(k,n) = B[k*ldb + n],
 *     C[m*ldc + n].
 *
 * Element decoding is exact: every fp16, bf16 and e4m3 value is a dyadic
 * rational that binary64 holds exactly.  The decoders are written from the
 * format definitions (IEEE 754 binary16; bfloat16 = the upper 16 bits of
 * binary32; OCP 8-bit "E4M3" with bias 7, no infinities, NaN = S.1111.111).
 * For the FP8 path the per-tensor scales are applied to the decoded inputs
 * ("oracle runs on the dequantised values"): a = dec(qa)*sa, b = dec(qb)*sb.
 * ("FP8 GEMM Optimization on AMD RDNA 4", section "What Changes at FP8":
 * E4M3 x E4M3 with a wider accumulator.)
 *
 * Round-to-nearest-even encoders for fp16 and bf16 are provided so that tests
 * can form the correctly rounded output code of an exact result.
 *
 * Pins (tests/test_oracle.py): hand-worked 2x2, 3x3 and non-square cases;
 * torch float64 matmul on random shapes; every fp16/bf16/e4m3 code against
 * torch's casts; encoders against torch's float32 casts including exact ties;
 * identity, all-ones and row-sum closed forms.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_F16 0
#define ORACLE_BF16 1
#define ORACLE_E4M3 2

/* ---------------------------------------------------------------- decoders */

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_dec_f16(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/2^10) * 2^(e-15) */
    }
    return s ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_dec_bf16(uint16_t h) {
    int s = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133); /* f * 2^-7 * 2^-126 */
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/2^7) * 2^(e-127) */
    }
    return s ? -v : v;
}

/* OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits.
 * No infinities; exponent 15 with fraction 7 is NaN; largest finite 448. */
double oracle_dec_e4m3(uint8_t q) {
    int s = (q >> 7) & 1;
    int e = (q >> 3) & 0xf;
    int f = q & 0x7;
    double v;
    if (e == 15 && f == 7) {
        v = NAN;
    } else if (e == 0) {
        v = ldexp((double)f, -9); /* f * 2^-3 * 2^-6 */
    } else {
        v = ldexp((double)(8 + f), e - 10); /* (1 + f/8) * 2^(e-7) */
    }
    return s ? -v : v;
}

/* ------------------------------------------------- round-to-nearest-even */

/* Round |x| (finite, > 0) to an integer multiple of 2^q with ties to even.
 * Returns the integer multiple as a double. */
static double rne_multiple(double ax, int q) {
    double n = ldexp(ax, -q);
    double fl = floor(n);
    double d = n - fl;
    if (d > 0.5) return fl + 1.0;
    if (d < 0.5) return fl;
    return (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
}

/* Encode a binary64 value as binary16 with round-to-nearest-even;
 * overflow goes to infinity as IEEE rounding prescribes. */
uint16_t oracle_enc_f16_rne(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7e00);
    if (isinf(x)) return (uint16_t)(sign | 0x7c00);
    if (ax == 0.0) return sign;
    int e2;
    frexp(ax, &e2);       /* ax = m * 2^e2, m in [0.5, 1) */
    int E = e2 - 1;       /* ax in [2^E, 2^(E+1)) */
    if (E < -14) E = -14; /* subnormal range shares the quantum 2^-24 */
    double r = rne_multiple(ax, E - 10);
    if (r >= 2048.0) { /* rounding carried into the next binade */
        r = r / 2.0;
        E += 1;
    }
    if (E > 15) return (uint16_t)(sign | 0x7c00);
    if (r < 1024.0) return (uint16_t)(sign | (uint16_t)r); /* subnormal */
    return (uint16_t)(sign | ((E + 15) << 10) | ((uint16_t)r - 1024));
}

/* Encode a binary64 value as bfloat16 with round-to-nearest-even. */
uint16_t oracle_enc_bf16_rne(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double ax = fabs(x);
    if (isnan(x)) return (uint16_t)(sign | 0x7fc0);
    if (isinf(x)) return (uint16_t)(sign | 0x7f80);
    if (ax == 0.0) return sign;
    int e2;
    frexp(ax, &e2);
    int E = e2 - 1;
    if (E < -126) E = -126;
    double r = rne_multiple(ax, E - 7);
    if (r >= 256.0) {
        r = r / 2.0;
        E += 1;
    }
    if (E > 127) return (uint16_t)(sign | 0x7f80);
    if (r < 128.0) return (uint16_t)(sign | (uint16_t)r);
    return (uint16_t)(sign | ((E + 127) << 7) | ((uint16_t)r - 128));
}

/* Vector helpers so that the Python side does not loop per element. */
void oracle_dec_array(int dtype, const void* codes, int64_t n, double* out) {
    for (int64_t i = 0; i < n; ++i) {
        if (dtype == ORACLE_F16)
            out[i] = oracle_dec_f16(((const uint16_t*)codes)[i]);
        else if (dtype == ORACLE_BF16)
            out[i] = oracle_dec_bf16(((const uint16_t*)codes)[i]);
        else
            out[i] = oracle_dec_e4m3(((const uint8_t*)codes)[i]);
    }
}

void oracle_enc_array(int dtype, const double* x, int64_t n, uint16_t* out) {
    for (int64_t i = 0; i < n; ++i)
        out[i] = (dtype == ORACLE_F16) ? oracle_enc_f16_rne(x[i]) : oracle_enc_bf16_rne(x[i]);
}

/* ------------------------------------------------------------ TN operands */

static double tn_elem(int dtype, const void* base, int64_t idx) {
    if (dtype == ORACLE_F16) return oracle_dec_f16(((const uint16_t*)base)[idx]);
    if (dtype == ORACLE_BF16) return oracle_dec_bf16(((const uint16_t*)base)[idx]);
    return oracle_dec_e4m3(((const uint8_t*)base)[idx]);
}

/* Row m of A, decoded and scaled: a(m, k) = dec(A[m*lda + k]) * sa. */
static void tn_row_a(int dtype, const void* A, int64_t lda, int64_t m, int64_t K, double sa,
                     double* out) {
    for (int64_t k = 0; k < K; ++k) out[k] = tn_elem(dtype, A, m * lda + k) * sa;
}

/* Column n of B (column-major), decoded and scaled: b(k, n) = dec(B[n*ldb + k]) * sb. */
static void tn_col_b(int dtype, const void* B, int64_t ldb, int64_t n, int64_t K, double sb,
                     double* out) {
    for (int64_t k = 0; k < K; ++k) out[k] = tn_elem(dtype, B, n * ldb + k) * sb;
}

static double dot_in_k_order(const double* a, const double* b, int64_t K) {
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) s += a[k] * b[k];
    return s;
}

/* Full TN product.  C[n*ldc + m] = sum_k a(m,k) b(k,n), binary64. */
int oracle_gemm_tn(int dtype, int64_t M, int64_t N, int64_t K, const void* A, int64_t lda,
                   const void* B, int64_t ldb, double sa, double sb, double* C, int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return 1;
    if (M == 0 || N == 0) return 0;
    double* a = (double*)malloc(sizeof(double) * (size_t)(M * (K > 0 ? K : 1)));
    double* b = (double*)malloc(sizeof(double) * (size_t)(N * (K > 0 ? K : 1)));
    if (!a || !b) {
        free(a);
        free(b);
        return 2;
    }
    for (int64_t m = 0; m < M; ++m) tn_row_a(dtype, A, lda, m, K, sa, a + m * K);
    for (int64_t n = 0; n < N; ++n) tn_col_b(dtype, B, ldb, n, K, sb, b + n * K);
#pragma omp parallel for schedule(static)
    for (int64_t n = 0; n < N; ++n)
        for (int64_t m = 0; m < M; ++m) C[n * ldc + m] = dot_in_k_order(a + m * K, b + n * K, K);
    free(a);
    free(b);
    return 0;
}

/* Sampled TN product: out[s] = C(ms[s], ns[s]), each a K-long dot product. */
int oracle_gemm_tn_sampled(int dtype, int64_t K, const void* A, int64_t lda, const void* B,
                           int64_t ldb, double sa, double sb, int64_t S, const int64_t* ms,
                           const int64_t* ns, double* out) {
    if (K < 0 || S < 0) return 1;
    int failed = 0;
#pragma omp parallel
    {
        double* a = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        double* b = (double*)malloc(sizeof(double) * (size_t)(K > 0 ? K : 1));
        if (!a || !b) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t s = 0; s < S; ++s) {
                tn_row_a(dtype, A, lda, ms[s], K, sa, a);
                tn_col_b(dtype, B, ldb, ns[s], K, sb, b);
                out[s] = dot_in_k_order(a, b, K);
            }
        }
        free(a);
        free(b);
    }
    return failed ? 2 : 0;
}

/* ---------------------------------------------------------------- FP32 */

/* Full row-major FP32 product, accumulated in binary64:
 * C[m*ldc + n] = sum_k A[m*lda + k] * B[k*ldb + n]. */
int oracle_gemm_f32(int64_t M, int64_t N, int64_t K, const float* A, int64_t lda, const float* B,
                    int64_t ldb, double* C, int64_t ldc) {
    if (M < 0 || N < 0 || K < 0) return 1;
#pragma omp parallel for schedule(static)
    for (int64_t m = 0; m < M; ++m) {
        for (int64_t n = 0; n < N; ++n) {
            double s = 0.0;
            for (int64_t k = 0; k < K; ++k) s += (double)A[m * lda + k] * (double)B[k * ldb + n];
            C[m * ldc + n] = s;
        }
    }
    return 0;
}

/* Sampled row-major FP32 product: out[s] = C(ms[s], ns[s]). */
int oracle_gemm_f32_sampled(int64_t K, const float* A, int64_t lda, const float* B, int64_t ldb,
                            int64_t S, const int64_t* ms, const int64_t* ns, double* out) {
    if (K < 0 || S < 0) return 1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t s = 0; s < S; ++s) {
        double acc = 0.0;
        for (int64_t k = 0; k < K; ++k)
            acc += (double)A[ms[s] * lda + k] * (double)B[k * ldb + ns[s]];
        out[s] = acc;
    }
    return 0;
}

/* Number of threads an OpenMP region here would use (reported by the
 * benchmark next to the CPU baseline). */
int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Sets the number of threads later OpenMP regions here use (n >= 1), so that
 * the benchmark can also time the oracle on one core.  Returns the count now
 * in effect. */
int oracle_set_num_threads(int n) {
#ifdef _OPENMP
    if (n >= 1) omp_set_num_threads(n);
#else
    (void)n;
#endif
    return oracle_num_threads();
}
