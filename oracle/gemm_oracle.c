/*
 * CPU oracle for the half-precision GEMM  D = A x B  (test infrastructure).
 *
 * This file is TEST INFRASTRUCTURE.  Only the test suite, the smoke check and
 * the CPU-baseline leg of the benchmark may load it.  It shares no code with
 * the CUDA library (no headers, helpers, tables or constants) and must never
 * be reached from the product path.
 *
 * What it computes, and where that is defined:
 *   - "B200 的 2CTA 怎样调优", section 七 (TMEM 与 epilogue), the per-element
 *     logic: acc = sum over k of A[i,k]*B[k,j]; the epilogue then converts acc
 *     to the output type.  The bias term printed there is not part of the
 *     library's operation and is not computed.
 *   - The acceptance bound also needs S[i,j] = sum_k |A[i,k]*B[k,j]|, the
 *     absolute-value sum over the same products.
 *
 * Precision: inputs are BF16 or FP16 bit patterns, each converted exactly to
 * double; every product of two such values is exact in double, and the sum
 * runs in double in ascending k.  No blocking, fusion or reordering: the loop
 * nest is i, then k, then j, which keeps the k order of every (i,j) sum
 * ascending while walking B by rows.  Rows are shared out over OpenMP threads
 * (each row is independent; within a row nothing changes).
 *
 * Layouts: A is row-major [M][lda] (element (i,k) at A[i*lda+k]); B is
 * row-major [K][ldb] (element (k,j) at B[k*ldb+j]); D and S are dense
 * row-major [rows][N] doubles owned by the caller.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

#define ORACLE_IN_BF16 0
#define ORACLE_IN_FP16 1

/* BF16 is the upper half of an IEEE binary32: widen and reinterpret. */
double oracle_bf16_to_double(uint16_t h) {
    uint32_t w = ((uint32_t)h) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

/* IEEE binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits.
 * Decoded from the definition of the format, value by value. */
double oracle_fp16_to_double(uint16_t h) {
    int sign = (h >> 15) & 1;
    int exp = (h >> 10) & 0x1f;
    int frac = h & 0x3ff;
    double v;
    if (exp == 0) {
        v = ldexp((double)frac, -24); /* subnormal: frac * 2^-14 * 2^-10 */
    } else if (exp == 31) {
        v = frac ? NAN : INFINITY;
    } else {
        v = ldexp((double)(frac + 1024), exp - 25); /* (1 + frac/1024) * 2^(exp-15) */
    }
    return sign ? -v : v;
}

static double decode(uint16_t h, int dtype) {
    return dtype == ORACLE_IN_FP16 ? oracle_fp16_to_double(h) : oracle_bf16_to_double(h);
}

/* Rows [row_begin, row_end) of D and S.  D/S point at row row_begin. */
void oracle_gemm_rows(const uint16_t *A, const uint16_t *B, int dtype, int M, int N, int K,
                      long lda, long ldb, int row_begin, int row_end, double *D, double *S) {
    (void)M;
    int i;
#pragma omp parallel for schedule(dynamic, 1)
    for (i = row_begin; i < row_end; ++i) {
        double *d = D + (long)(i - row_begin) * N;
        double *s = S + (long)(i - row_begin) * N;
        for (int j = 0; j < N; ++j) {
            d[j] = 0.0;
            s[j] = 0.0;
        }
        for (int k = 0; k < K; ++k) {
            double a = decode(A[(long)i * lda + k], dtype);
            const uint16_t *brow = B + (long)k * ldb;
            for (int j = 0; j < N; ++j) {
                double p = a * decode(brow[j], dtype);
                d[j] += p;
                s[j] += fabs(p);
            }
        }
    }
}

/* The whole product: D = A x B, S = |A| x |B| (element by element sums). */
void oracle_gemm(const uint16_t *A, const uint16_t *B, int dtype, int M, int N, int K, long lda,
                 long ldb, double *D, double *S) {
    oracle_gemm_rows(A, B, dtype, M, N, K, lda, ldb, 0, M, D, S);
}

/* Single outputs, one dot product each: D[t] = sum_k A[I[t],k]*B[k,J[t]]. */
void oracle_gemm_elements(const uint16_t *A, const uint16_t *B, int dtype, int K, long lda,
                          long ldb, const long *I, const long *J, long count, double *D,
                          double *S) {
    long t;
#pragma omp parallel for schedule(static)
    for (t = 0; t < count; ++t) {
        double acc = 0.0, sabs = 0.0;
        for (int k = 0; k < K; ++k) {
            double p = decode(A[I[t] * lda + k], dtype) * decode(B[(long)k * ldb + J[t]], dtype);
            acc += p;
            sabs += fabs(p);
        }
        D[t] = acc;
        S[t] = sabs;
    }
}

/*
 * Grouped product ("MegaMoE … 融合算子解读", the expert-GEMM stage): rows
 * offsets[g] .. offsets[g+1]-1 of A are multiplied by the g-th weight matrix
 * Bs[g] ([K][N], row-major, leading dimension N).  A is [offsets[G]][K] dense,
 * D and S are [offsets[G]][N] dense.
 */
void oracle_grouped_gemm(const uint16_t *A, const uint16_t *const *Bs, const int *offsets, int G,
                         int N, int K, int dtype, double *D, double *S) {
    for (int g = 0; g < G; ++g) {
        int r0 = offsets[g], r1 = offsets[g + 1];
        if (r1 <= r0) continue;
        oracle_gemm_rows(A, Bs[g], dtype, offsets[G], N, K, K, N, r0, r1, D + (long)r0 * N,
                         S + (long)r0 * N);
    }
}

/*
 * SwiGLU of a gate/up projection computed as one GEMM.
 *   "B200 的 2CTA 怎样调优", section 七, "Gate／SwiGLU": the output at each
 *   position is up x SiLU(gate), where the gate and up projections are column
 *   blocks of the same GEMM; no reduction over a row is involved.
 *   "MegaMoE … 融合算子解读", section 09: FC1's accumulators become
 *   gate/up pairs, then SwiGLU, then the next layer's input.
 * Layout (the library's reading of "column blocks"): D is [rows][2*I], the
 * gate projection in columns 0 .. I-1 and the up projection in columns
 * I .. 2I-1 (the weight matrix is [gate | up] along N).  H is [rows][I]:
 *   H[r][j] = silu(g) * u,   g = D[r][j],  u = D[r][I + j],
 *   silu(x) = x * sigmoid(x) = x / (1 + exp(-x)).
 * For x far below zero exp(-x) overflows to +inf and silu(x) is -0, the
 * limit of x / (1 + e^-x); the true value there is below 1e-300 in size.
 * SILU, if not NULL, receives silu(g) ([rows][I]) for the error bound.
 */
void oracle_swiglu(const double *D, long rows, int I, double *H, double *SILU) {
    long r;
#pragma omp parallel for schedule(static)
    for (r = 0; r < rows; ++r) {
        const double *gate = D + r * 2L * I;
        const double *up = gate + I;
        double *h = H + r * (long)I;
        for (int j = 0; j < I; ++j) {
            double g = gate[j];
            double silu = g / (1.0 + exp(-g));
            h[j] = silu * up[j];
            if (SILU) SILU[r * (long)I + j] = silu;
        }
    }
}

/*
 * Round-to-nearest-even from double to the 16-bit output formats, written
 * from the format definitions.  Used only where the exact result is known to
 * be representable in binary32 (integer-valued inputs), so the double ->
 * binary32 step is exact and only the final rounding matters.
 */
uint16_t oracle_round_bf16(double x) {
    float f = (float)x;
    uint32_t w;
    memcpy(&w, &f, sizeof w);
    if ((w & 0x7fffffffu) > 0x7f800000u) return (uint16_t)((w >> 16) | 0x40); /* quiet NaN */
    uint32_t lsb = (w >> 16) & 1u;
    w += 0x7fffu + lsb; /* ties go to the even neighbour */
    return (uint16_t)(w >> 16);
}

uint16_t oracle_round_fp16(double x) {
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isnan(x)) return 0x7e00;
    if (a >= 65520.0) return sign | 0x7c00; /* at or past the midpoint above 65504 */
    if (a < ldexp(1.0, -14)) {
        /* subnormal range: units of 2^-24 */
        double q = a * ldexp(1.0, 24);
        double r = nearbyint(q); /* default rounding mode: ties to even */
        return sign | (uint16_t)r;
    }
    int e;
    double m = frexp(a, &e); /* a = m * 2^e, m in [0.5, 1) */
    /* 11 significant bits: scale so that the significand is an integer in [1024, 2048) */
    double q = ldexp(m, 11);
    double r = nearbyint(q);
    if (r == 2048.0) {
        r = 1024.0;
        e += 1;
    }
    int biased = e - 1 + 15;
    if (biased >= 31) return sign | 0x7c00;
    return sign | (uint16_t)(biased << 10) | (uint16_t)((int)r - 1024);
}

int oracle_num_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}

/* Number of threads later calls run on (at least 1).  Timing aid: the
 * arithmetic is the same on any number of threads. */
void oracle_set_num_threads(int n) {
#ifdef _OPENMP
    omp_set_num_threads(n > 0 ? n : 1);
#else
    (void)n;
#endif
}
