/*
 * gemm_oracle.c -- TEST INFRASTRUCTURE ONLY.
 *
 * A plain, slow, obviously correct CPU definition of the dense matrix product
 * C[M,N] = A[M,K] @ B[K,N] that the GPU path computes.  Only the test suite,
 * the smoke check and the benchmark's CPU-baseline leg may load this file's
 * library; the product path never does, and this file shares no code, header,
 * table or helper with the CUDA library.
 *
 * Sources (the four web pages this project follows):
 *   - "I Wrote a GPU Matmul Kernel From Scratch in Triton" (cnblogs translation),
 *     Step 1 (naive three-loop matmul) and Step 2 (blockwise six-loop matmul).
 *   - "Writing GPU kernels in Triton: Vector Add, Softmax, MatMul"
 *     (blog.ulna520.top), section 3.1 (C[i,j] = sum_k A[i,k] B[k,j]) and
 *     section 4.1 (row-major offset(i, j) = i * ld + j, in elements).
 *
 * Numerics: every 16-bit input is widened EXACTLY to double (both fp16 and
 * bf16 values are exactly representable in binary64), every product of two
 * such values is exact in binary64, and the sum runs in binary64 with k
 * ascending for each (i, j) -- the order of the naive loop of Step 1.
 * The file must be compiled with -ffp-contract=off so that no FMA changes the
 * rounding on one host and not on another.
 *
 * Threads split the rows i only, so no result depends on the thread count.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

enum { ORACLE_F16 = 0, ORACLE_BF16 = 1 };

/* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits. */
double oracle_f16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);               /* subnormal: f * 2^-10 * 2^-14 */
    } else if (e == 31) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(1024 + f), e - 25);   /* (1 + f/2^10) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* bfloat16: 1 sign bit, 8 exponent bits (bias 127), 7 fraction bits. */
double oracle_bf16_to_f64(uint16_t h)
{
    int sign = (h >> 15) & 1;
    int e = (h >> 7) & 0xff;
    int f = h & 0x7f;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -133);              /* subnormal: f * 2^-7 * 2^-126 */
    } else if (e == 255) {
        v = (f == 0) ? INFINITY : NAN;
    } else {
        v = ldexp((double)(128 + f), e - 134);   /* (1 + f/2^7) * 2^(e-127) */
    }
    return sign ? -v : v;
}

/* Decode tables: table[bits] is the exact value of the 16-bit pattern. */
static double g_table[2][65536];
static int g_table_ready[2];

static const double *table_for(int dtype)
{
    if (dtype != ORACLE_F16 && dtype != ORACLE_BF16) return 0;
    if (!g_table_ready[dtype]) {
        for (uint32_t b = 0; b < 65536u; ++b)
            g_table[dtype][b] = (dtype == ORACLE_F16) ? oracle_f16_to_f64((uint16_t)b)
                                                      : oracle_bf16_to_f64((uint16_t)b);
        g_table_ready[dtype] = 1;
    }
    return g_table[dtype];
}

static int set_threads(int nthreads)
{
#ifdef _OPENMP
    if (nthreads <= 0) nthreads = omp_get_max_threads();
    return nthreads;
#else
    (void)nthreads;
    return 1;
#endif
}

/*
 * C[i, j] = sum_{k=0}^{K-1} A[i, k] * B[k, j]   (i < M, j < N), in binary64.
 * A[i, k] is at A[i*lda + k]; B[k, j] at B[k*ldb + j]; C[i, j] at C[i*ldc + j].
 * The loop nest is i-k-j with a per-row accumulator: for a fixed (i, j) the
 * terms are added with k ascending, exactly as in the naive loop of Step 1.
 * K == 0 gives the empty sum (zeros).  Returns 0, or -1 on a bad argument.
 */
int oracle_gemm(int dtype, const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                double *C, int64_t ldc, int64_t M, int64_t N, int64_t K, int nthreads)
{
    const double *t = table_for(dtype);
    if (!t || M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N) return -1;
    int nt = set_threads(nthreads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
    for (int64_t i = 0; i < M; ++i) {
        double *c = C + i * ldc;
        for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = t[A[i * lda + k]];
            const uint16_t *b = B + k * ldb;
            for (int64_t j = 0; j < N; ++j) c[j] += a * t[b[j]];
        }
    }
    return 0;
}

/*
 * bound[i, j] = sum_k |A[i, k]| * |B[k, j]| in binary64, same loop order.
 * This is the scale of the parity tolerance: |C_gpu - C| <= 1e-3 * bound + 1e-5.
 */
int oracle_absbound(int dtype, const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                    double *Bd, int64_t ldbd, int64_t M, int64_t N, int64_t K, int nthreads)
{
    const double *t = table_for(dtype);
    if (!t || M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldbd < N) return -1;
    int nt = set_threads(nthreads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
    for (int64_t i = 0; i < M; ++i) {
        double *c = Bd + i * ldbd;
        for (int64_t j = 0; j < N; ++j) c[j] = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double a = fabs(t[A[i * lda + k]]);
            const uint16_t *b = B + k * ldb;
            for (int64_t j = 0; j < N; ++j) c[j] += a * fabs(t[b[j]]);
        }
    }
    return 0;
}

/*
 * The same definition evaluated only at the listed entries (rows[e], cols[e]):
 * value[e] = sum_k A[r, k] B[k, c] and bound[e] = sum_k |A[r, k]| |B[k, c]|,
 * k ascending.  Used where the full product would take the CPU too long.
 */
int oracle_gemm_entries(int dtype, const uint16_t *A, int64_t lda, const uint16_t *B, int64_t ldb,
                        int64_t M, int64_t N, int64_t K, const int64_t *rows, const int64_t *cols,
                        int64_t count, double *value, double *bound, int nthreads)
{
    const double *t = table_for(dtype);
    if (!t || M < 0 || N < 0 || K < 0 || lda < K || ldb < N || count < 0) return -1;
    for (int64_t e = 0; e < count; ++e)
        if (rows[e] < 0 || rows[e] >= M || cols[e] < 0 || cols[e] >= N) return -1;
    int nt = set_threads(nthreads);
    (void)nt;
#ifdef _OPENMP
#pragma omp parallel for schedule(static) num_threads(nt)
#endif
    for (int64_t e = 0; e < count; ++e) {
        int64_t r = rows[e], c = cols[e];
        double s = 0.0, sb = 0.0;
        for (int64_t k = 0; k < K; ++k) {
            double p = t[A[r * lda + k]] * t[B[k * ldb + c]];
            s += p;
            sb += fabs(p);
        }
        value[e] = s;
        bound[e] = sb;
    }
    return 0;
}

/*
 * Blockwise six-loop product from Step 2 of "I Wrote a GPU Matmul Kernel From
 * Scratch in Triton": loop over (i, j, k) tiles of size bs (edges clamped with
 * min), and for each (ii, jj) in the tile add the partial sum over the k tile
 * to C[ii, jj].  The multiplications are the same M*N*K as the naive loop;
 * only the grouping of the additions differs, so on inputs whose partial sums
 * are exact (small integers) it equals oracle_gemm bit for bit.
 */
int oracle_gemm_blockwise(int dtype, const uint16_t *A, int64_t lda, const uint16_t *B,
                          int64_t ldb, double *C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                          int64_t bs)
{
    const double *t = table_for(dtype);
    if (!t || bs <= 0 || M < 0 || N < 0 || K < 0 || lda < K || ldb < N || ldc < N) return -1;
    for (int64_t i = 0; i < M; ++i)
        for (int64_t j = 0; j < N; ++j) C[i * ldc + j] = 0.0;
    for (int64_t i = 0; i < M; i += bs)
        for (int64_t j = 0; j < N; j += bs)
            for (int64_t k = 0; k < K; k += bs) {
                int64_t ie = (i + bs < M) ? i + bs : M;
                int64_t je = (j + bs < N) ? j + bs : N;
                int64_t ke = (k + bs < K) ? k + bs : K;
                for (int64_t ii = i; ii < ie; ++ii)
                    for (int64_t jj = j; jj < je; ++jj) {
                        double s = 0.0;
                        for (int64_t kk = k; kk < ke; ++kk)
                            s += t[A[ii * lda + kk]] * t[B[kk * ldb + jj]];
                        C[ii * ldc + jj] += s;
                    }
            }
    return 0;
}

/* Number of threads an OpenMP region with nthreads <= 0 would use. */
int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
