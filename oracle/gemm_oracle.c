/*
 * gemm_oracle.c -- the CPU oracle for C = A * B^T.  TEST INFRASTRUCTURE ONLY.
 *
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference
 * leg may load or call this library.  The product path (the CUDA library under
 * dense_gemm_blackwell_sm_gb300/) never links, imports or executes it, and this
 * file shares no code, header, table or constant with that path.
 *
 * What it computes (plain definition, fp64):
 *
 *     C[i][j] = sum_{k=0}^{K-1} a[i][k] * b[j][k]      0 <= i < M, 0 <= j < N
 *     S[i][j] = sum_{k=0}^{K-1} |a[i][k] * b[j][k]|
 *
 * A is M x K row-major and B is N x K row-major (both K-major), so the result
 * is A times B-transposed, C being M x N row-major.  This is the tiled GEMM that
 * "Modern GPU Programming for MLSys" (reading notes, section "9 步优化",
 * steps 1-3) builds tile by tile: the Tensor Core computes D = A x B + C with
 * fp32 accumulation in TMEM (section "计算单元", "存储层次: TMEM"), the K loop
 * adds every K-block's partial product into one accumulator (step 2), and the
 * split of the output into a tile grid (step 3) cannot change the value of any
 * element.  So the oracle is the definition itself: a triple loop, i then j
 * then k innermost, summed sequentially in k order, with no blocking, no
 * reassociation and no BLAS.  Rows are spread over OpenMP threads, which leaves
 * the summation order of every element unchanged.
 *
 * Inputs arrive as raw 16-bit patterns (IEEE binary16 or bfloat16) and are
 * widened exactly to double by this file's own decoders.  Every product of two
 * such values is exact in double (11+11 resp. 8+8 significand bits < 53), so
 * the only rounding is in the k-sum, bounded by (K-1) * 2^-53 * S.
 */
#define _USE_MATH_DEFINES
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#ifndef M_PI
#define M_PI 3.14159265358979323846
#endif

#define ORACLE_IN_F16 0
#define ORACLE_IN_BF16 1

/* IEEE 754 binary16: sign bit 15, 5-bit exponent (bias 15), 10-bit fraction. */
static double widen_binary16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);                 /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);     /* (1 + f/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: the upper half of an IEEE binary32 -- sign bit 15, 8-bit exponent
 * (bias 127), 7-bit fraction. */
static double widen_bfloat16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int f = h & 0x7F;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);                /* subnormal: f * 2^-126 * 2^-7 */
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + f), e - 134);     /* (1 + f/2^7) * 2^(e-127) */
    }
    return sign ? -v : v;
}

double oracle_widen(uint16_t bits, int in_kind) {
    return in_kind == ORACLE_IN_BF16 ? widen_bfloat16(bits) : widen_binary16(bits);
}

/* A 65536-entry table of the decoded values, so the inner loop reads doubles. */
static double* make_table(int in_kind) {
    double* t = (double*)malloc(sizeof(double) * 65536);
    if (!t) return NULL;
    for (uint32_t b = 0; b < 65536; ++b) t[b] = oracle_widen((uint16_t)b, in_kind);
    return t;
}

static void set_threads(int nthreads) {
#ifdef _OPENMP
    if (nthreads > 0) omp_set_num_threads(nthreads);
#else
    (void)nthreads;
#endif
}

int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/*
 * Rows `rows[0..nrows)` of C and S (each nrows x N, row-major).  rows == NULL
 * means every row 0..M-1 (then nrows must equal M).  S may be NULL.
 * Returns 0 on success, -1 on a bad argument or allocation failure.
 */
int oracle_gemm_rows_f64(int64_t M, int64_t N, int64_t K,
                         const uint16_t* A, const uint16_t* B, int in_kind,
                         const int64_t* rows, int64_t nrows,
                         double* C, double* S, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (in_kind != ORACLE_IN_F16 && in_kind != ORACLE_IN_BF16) return -1;
    if (rows == NULL && nrows != M) return -1;
    if (rows != NULL) {
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= M) return -1;
    }
    double* tab = make_table(in_kind);
    if (!tab) return -1;
    set_threads(nthreads);

    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        const uint16_t* a = A + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const uint16_t* b = B + j * K;
            double acc = 0.0;
            double sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = tab[a[k]] * tab[b[k]];   /* exact */
                acc += p;
                sabs += fabs(p);
            }
            C[r * N + j] = acc;
            if (S) S[r * N + j] = sabs;
        }
    }
    free(tab);
    return 0;
}

/* The whole M x N result. */
int oracle_gemm_f64(int64_t M, int64_t N, int64_t K,
                    const uint16_t* A, const uint16_t* B, int in_kind,
                    double* C, double* S, int nthreads) {
    return oracle_gemm_rows_f64(M, N, K, A, B, in_kind, NULL, M, C, S, nthreads);
}

/*
 * Fused epilogue of a linear layer, applied in place to an fp64 result C
 * (M x N, row-major):
 *
 *     C[i][j] = act(C[i][j] + bias[j]) + residual[i][j]
 *
 * The reading notes (section "LLM 推理本质上是一张有向无环图") describe an LLM's
 * forward pass as a DAG whose linear nodes (the GEMMs) feed nonlinear ones such
 * as GeLU and SiLU; the activation formulas below are their standard
 * definitions, evaluated in fp64 with the C library's exp, tanh and erf.
 *
 * bias: N fp32 values or NULL.  residual: M x N values or NULL, of kind
 * 1 = fp32, 2 = bfloat16 bit patterns, 3 = binary16 bit patterns.
 * act: 0 none, 1 relu, 2 silu, 3 gelu (tanh form), 4 gelu (erf form).
 */
static double oracle_act(double x, int act) {
    switch (act) {
        case 1: return x > 0.0 ? x : 0.0;
        case 2: return x / (1.0 + exp(-x));
        case 3: return 0.5 * x * (1.0 + tanh(sqrt(2.0 / M_PI) * (x + 0.044715 * x * x * x)));
        case 4: return 0.5 * x * (1.0 + erf(x / sqrt(2.0)));
        default: return x;
    }
}

double oracle_activation(double x, int act) { return oracle_act(x, act); }

/*
 * Dequantisation scales of the fused epilogue: C[i][j] *= scale_a[i] * scale_b[j]
 * (either may be NULL).  The product of an fp64 value and two fp32 values.
 */
int oracle_scale_f64(int64_t M, int64_t N, double* C, const float* scale_a, const float* scale_b) {
    if (M < 0 || N < 0) return -1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) {
            double x = C[i * N + j];
            if (scale_a) x *= (double)scale_a[i];
            if (scale_b) x *= (double)scale_b[j];
            C[i * N + j] = x;
        }
    return 0;
}

int oracle_epilogue_f64(int64_t M, int64_t N, double* C, const float* bias, const void* residual,
                        int residual_kind, int act) {
    if (M < 0 || N < 0 || act < 0 || act > 4) return -1;
    if (residual != NULL && (residual_kind < 1 || residual_kind > 3)) return -1;
    for (int64_t i = 0; i < M; ++i) {
        for (int64_t j = 0; j < N; ++j) {
            double x = C[i * N + j];
            if (bias) x += (double)bias[j];
            x = oracle_act(x, act);
            if (residual) {
                const int64_t e = i * N + j;
                if (residual_kind == 1) {
                    x += (double)((const float*)residual)[e];
                } else {
                    const uint16_t bits = ((const uint16_t*)residual)[e];
                    x += oracle_widen(bits, residual_kind == 2 ? ORACLE_IN_BF16 : ORACLE_IN_F16);
                }
            }
            C[i * N + j] = x;
        }
    }
    return 0;
}

/*
 * 8-bit floating point inputs (the low-precision GEMM).  OCP FP8 formats:
 *   E4M3: sign bit 7, 4-bit exponent (bias 7), 3-bit fraction; exponent 0 is
 *         subnormal (f * 2^-9); S.1111.111 is NaN; there is no infinity.
 *   E5M2: sign bit 7, 5-bit exponent (bias 15), 2-bit fraction; exponent 0 is
 *         subnormal (f * 2^-16); exponent 31 is infinity (f = 0) or NaN.
 * Products of two such values carry at most 8 significant bits: exact in fp64.
 */
#define ORACLE_IN_E4M3 2
#define ORACLE_IN_E5M2 3

static double widen_e4m3(uint8_t h) {
    int sign = (h >> 7) & 1, e = (h >> 3) & 0xF, f = h & 0x7;
    double v;
    if (e == 0) v = ldexp((double)f, -9);
    else if (e == 15 && f == 7) v = NAN;
    else v = ldexp((double)(8 + f), e - 10);
    return sign ? -v : v;
}

static double widen_e5m2(uint8_t h) {
    int sign = (h >> 7) & 1, e = (h >> 2) & 0x1F, f = h & 0x3;
    double v;
    if (e == 0) v = ldexp((double)f, -16);
    else if (e == 31) v = (f == 0) ? INFINITY : NAN;
    else v = ldexp((double)(4 + f), e - 17);
    return sign ? -v : v;
}

double oracle_widen8(uint8_t bits, int in_kind) {
    return in_kind == ORACLE_IN_E5M2 ? widen_e5m2(bits) : widen_e4m3(bits);
}

int oracle_gemm8_rows_f64(int64_t M, int64_t N, int64_t K,
                          const uint8_t* A, const uint8_t* B, int in_kind,
                          const int64_t* rows, int64_t nrows,
                          double* C, double* S, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0) return -1;
    if (in_kind != ORACLE_IN_E4M3 && in_kind != ORACLE_IN_E5M2) return -1;
    if (rows == NULL && nrows != M) return -1;
    if (rows != NULL) {
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= M) return -1;
    }
    double tab[256];
    for (int b = 0; b < 256; ++b) tab[b] = oracle_widen8((uint8_t)b, in_kind);
    set_threads(nthreads);
    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        const uint8_t* a = A + i * K;
        for (int64_t j = 0; j < N; ++j) {
            const uint8_t* b = B + j * K;
            double acc = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = tab[a[k]] * tab[b[k]];   /* exact */
                acc += p;
                sabs += fabs(p);
            }
            C[r * N + j] = acc;
            if (S) S[r * N + j] = sabs;
        }
    }
    return 0;
}

/*
 * MX block scaling (OCP Microscaling Formats (MX) Specification v1.0, section
 * 5: an MX block is k = 32 consecutive elements sharing one scale X in the
 * UE8M0 format, X = 2^(e - 127), e = 255 encoding NaN).  The block-scaled
 * GEMM multiplies each element by its block's scale before the dot product:
 *
 *   C[i][j] = sum_k (X_A[i][k / 32] * a_ik) * (X_B[j][k / 32] * b_jk)
 *
 * SA is M x ceil(K/32) and SB is N x ceil(K/32), row-major, one byte per
 * scale.  Every term is exact in fp64 (8-bit float products times a power of
 * two between 2^-254 and 2^254).
 */
static double ue8m0(uint8_t e) { return e == 255 ? NAN : ldexp(1.0, (int)e - 127); }

double oracle_ue8m0(uint8_t e) { return ue8m0(e); }

int oracle_gemm_mx_rows_f64(int64_t M, int64_t N, int64_t K, const uint8_t* A, const uint8_t* B,
                            int in_kind, const uint8_t* SA, const uint8_t* SB,
                            const int64_t* rows, int64_t nrows, double* C, double* S, int nthreads) {
    if (M < 0 || N < 0 || K < 0 || nrows < 0 || !SA || !SB) return -1;
    if (in_kind != ORACLE_IN_E4M3 && in_kind != ORACLE_IN_E5M2) return -1;
    if (rows == NULL && nrows != M) return -1;
    if (rows != NULL) {
        for (int64_t r = 0; r < nrows; ++r)
            if (rows[r] < 0 || rows[r] >= M) return -1;
    }
    const int64_t KS = (K + 31) / 32;
    double tab[256], x8[256];
    for (int b = 0; b < 256; ++b) {
        tab[b] = oracle_widen8((uint8_t)b, in_kind);
        x8[b] = ue8m0((uint8_t)b);
    }
    set_threads(nthreads);
    int64_t r;
#pragma omp parallel for schedule(dynamic, 1)
    for (r = 0; r < nrows; ++r) {
        int64_t i = rows ? rows[r] : r;
        const uint8_t* a = A + i * K;
        const uint8_t* sa = SA + i * KS;
        for (int64_t j = 0; j < N; ++j) {
            const uint8_t* b = B + j * K;
            const uint8_t* sb = SB + j * KS;
            double acc = 0.0, sabs = 0.0;
            for (int64_t k = 0; k < K; ++k) {
                double p = (x8[sa[k / 32]] * tab[a[k]]) * (x8[sb[k / 32]] * tab[b[k]]);
                acc += p;
                sabs += fabs(p);
            }
            C[r * N + j] = acc;
            if (S) S[r * N + j] = sabs;
        }
    }
    return 0;
}
