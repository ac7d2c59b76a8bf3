/*
 * gemm_oracle.c -- test infrastructure, not product code.
 *
 * The CPU oracle for the tiled GEMM: the plain definition of what the tiled
 * kernel approximates, evaluated in fp64 with no blocking, fusion or
 * reordering.  Only the test suite, the smoke check and the bench's CPU
 * baseline load it; the CUDA library never does, and the two share no code.
 *
 * What it computes (ninetoothed.org "Named layouts", the GEMM application and
 * the bias/ReLU/residual postprocessing it supports; pbelevich.github.io
 * "My Triton From Scratch Part 16: Register Tiles", the runtime K loop):
 *
 *     acc(m,n) = sum_{k=0}^{K-1} A(m,k) * B(k,n)                   (fp64)
 *     y        = acc
 *     y        = y * scale_m[m]          if a row scale is given   (axes "m")
 *     y        = y + bias_n[n]           if a column bias is given (axes "n")
 *     y        = max(y, 0)               if relu
 *     y        = y + R(m,n)              if a residual is given
 *
 * The fixed order scale -> bias -> ReLU -> residual is the reading of
 * C = relu(scale_m * (A.B) + bias_n) + R.  y is returned unrounded.
 *
 * Operand addressing (explicit permute for a transposed operand, positive
 * leading dimensions, unit inner stride):
 *     permA = 0: A(m,k) = A[m*lda + k]      permA = 1: A(m,k) = A[k*lda + m]
 *     permB = 0: B(k,n) = B[k*ldb + n]      permB = 1: B(k,n) = B[n*ldb + k]
 *     R(m,n) = R[m*ldr + n]
 *
 * The 16-bit inputs are decoded by this file's own routines, written from the
 * IEEE 754 binary16 and the bfloat16 definitions (sign, exponent, fraction,
 * subnormals); no compiler half type is used.
 */
#include <math.h>
#include <stdint.h>

#ifdef _OPENMP
#include <omp.h>
#endif

/* binary16: 1 sign, 5 exponent (bias 15), 10 fraction bits. */
static double decode_f16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1F;
    int f = h & 0x3FF;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24); /* subnormal: f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(1024 + f), e - 25); /* (1 + f/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign, 8 exponent (bias 127), 7 fraction bits. */
static double decode_bf16(uint16_t h) {
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xFF;
    int f = h & 0x7F;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133); /* f * 2^-7 * 2^-126 */
    } else if (e == 255) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(128 + f), e - 134); /* (1 + f/2^7) * 2^(e-127) */
    }
    return sign ? -v : v;
}

static double decode(uint16_t h, int dtype) {
    return dtype == 0 ? decode_f16(h) : decode_bf16(h);
}

/* Decodes n 16-bit patterns (exported so the decoders can be pinned alone). */
void oracle_decode(const uint16_t* src, int64_t n, int dtype, double* dst) {
    for (int64_t i = 0; i < n; ++i) dst[i] = decode(src[i], dtype);
}

/*
 * Y[(m - row_begin)*N + n] = y(m, n) for row_begin <= m < row_end.
 * bias, scale and R may be NULL.  threads <= 0 means "OpenMP default".
 * Returns 0, or -1 on a bad argument.
 */
int oracle_gemm(int64_t M, int64_t N, int64_t K,
                const uint16_t* A, int64_t lda, int permA,
                const uint16_t* B, int64_t ldb, int permB,
                int dtype,
                const uint16_t* bias, const uint16_t* scale, int relu,
                const uint16_t* R, int64_t ldr,
                int64_t row_begin, int64_t row_end,
                double* Y, int threads) {
    if (M < 0 || N < 0 || K < 0 || row_begin < 0 || row_end > M || row_begin > row_end)
        return -1;
    if ((dtype != 0 && dtype != 1) || (permA != 0 && permA != 1) || (permB != 0 && permB != 1))
        return -1;
#ifdef _OPENMP
    if (threads > 0) omp_set_num_threads(threads);
#else
    (void)threads;
#endif

    /* Every 16-bit pattern decoded once; the sums below index this table. */
    static double table[2][65536];
    static int table_ready[2];
    if (!table_ready[dtype]) {
        for (int h = 0; h < 65536; ++h) table[dtype][h] = decode((uint16_t)h, dtype);
        table_ready[dtype] = 1;
    }
    const double* dec = table[dtype];

    int64_t m;
#pragma omp parallel for schedule(dynamic, 1)
    for (m = row_begin; m < row_end; ++m) {
        double* y = Y + (m - row_begin) * N;
        for (int64_t n = 0; n < N; ++n) y[n] = 0.0;
        /* i-k-j order: the sum over k for each (m, n) is still the plain sum */
        for (int64_t k = 0; k < K; ++k) {
            double a = dec[permA == 0 ? A[m * lda + k] : A[k * lda + m]];
            if (permB == 0) {
                const uint16_t* brow = B + k * ldb;
                for (int64_t n = 0; n < N; ++n) y[n] += a * dec[brow[n]];
            } else {
                for (int64_t n = 0; n < N; ++n) y[n] += a * dec[B[n * ldb + k]];
            }
        }
        double s = scale ? dec[scale[m]] : 1.0;
        for (int64_t n = 0; n < N; ++n) {
            double v = y[n];
            if (scale) v = v * s;
            if (bias) v = v + dec[bias[n]];
            if (relu) v = v > 0.0 ? v : 0.0;
            if (R) v = v + dec[R[m * ldr + n]];
            y[n] = v;
        }
    }
    return 0;
}

/* Threads an OpenMP parallel region gets by default (for reporting). */
int oracle_max_threads(void) {
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
