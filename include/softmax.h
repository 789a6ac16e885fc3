/*
 * softmax.h -- C ABI of the row-wise softmax of the GB300 (sm_103a) library
 * (libgemm.so; status codes shared with gemm.h).
 *
 * Operation (chapter 2 of "Writing GPU kernels in Triton: Vector Add, Softmax,
 * MatMul": section 2.4 for the row-wise form, section 2.3 for the five steps):
 *
 *     Y[i, j] = exp(X[i, j] - m_i) / sum_{k<N} exp(X[i, k] - m_i),
 *     m_i = max_{k<N} X[i, k]                       0 <= i < M, 0 <= j < N
 *
 * in fp32 (the chapter's kernel reads and writes fp32), every row on its own.
 * Subtracting the row maximum leaves the result unchanged and keeps every
 * exponent <= 0 (section 2.3).  Fused: each row is read from memory once and
 * written once while it fits on chip (N <= 32768); longer rows are read twice
 * (a pass that keeps a running maximum and a rescaled running sum, then the
 * normalising pass).  When the rows of X start on 16-byte boundaries and
 * 8192 < N <= 24576, a producer warp per CTA streams the CTA's rows into a
 * ring of shared-memory slots with bulk asynchronous copies while the other
 * warps reduce earlier rows.
 *
 * Layout: row-major with unit inner stride and explicit leading dimensions in
 * ELEMENTS: X[i, j] at X + i*ldx + j (ldx >= N), Y[i, j] at Y + i*ldy + j
 * (ldy >= N).  Columns j >= N are never read or written.  Y may be X itself
 * (in place, with ldy == ldx); any other overlap is rejected.
 *
 * Special values follow the formula: an entry of -inf weighs 0 (the padding
 * argument of section 2.6); a row of -inf only, or a row holding +inf or a
 * NaN, comes out NaN.
 *
 * Ownership: the caller owns X, Y (device memory, 4-byte aligned) and the
 * stream; nothing is allocated and the call does not synchronise (unless
 * GEMM_DEBUG_SYNC=1: then it waits and reports a bounded device-side wait that
 * gave up as GEMM_ERR_TIMEOUT, and in the checked build a load or store outside
 * the M x N matrices as GEMM_ERR_BOUNDS).  Work runs on the current CUDA
 * device, which must be compute capability 10.3.
 *
 * Errors: GEMM_ERR_INVALID_ARG for a null pointer when M*N > 0, negative M or
 * N, ldx < N or ldy < N, a misaligned pointer, or X and Y overlapping other
 * than exactly; GEMM_ERR_UNSUPPORTED for N or M beyond 2^31 - 1 or a device
 * that is not sm_103; GEMM_ERR_CUDA when the launch fails.  M == 0 or N == 0
 * is a no-op returning GEMM_OK.
 */
#ifndef DENSE_GEMM_05_GB300_SOFTMAX_H
#define DENSE_GEMM_05_GB300_SOFTMAX_H

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

/* How a call is executed (reported by softmax_rows_query). */
typedef enum {
    SOFTMAX_PATH_NONE = 0,     /* M == 0 or N == 0: nothing to do */
    SOFTMAX_PATH_WARP = 1,     /* one warp per row, the row in registers (N <= 2048) */
    SOFTMAX_PATH_CTA = 2,      /* 512 threads per row, the row in registers (N <= 32768) */
    SOFTMAX_PATH_STREAM = 3    /* one 1024-thread CTA per row, two passes over the row */
} softmax_path_t;

typedef struct {
    int32_t path;              /* softmax_path_t */
    int32_t threads_per_row;   /* threads that share one row */
    int32_t elems_per_thread;  /* row elements each thread holds (register paths) or streams */
    int32_t vec;               /* 4: 16-byte loads and stores; 1: 4-byte (unaligned rows) */
    int32_t rows_per_cta;
    int32_t block;             /* threads per CTA */
    int32_t grid;              /* CTAs launched (a persistent grid over the rows) */
    int32_t staged;            /* 1: rows staged in a shared-memory ring by bulk async copies */
    int32_t slots;             /* staged: row slots in the ring */
} softmax_config_t;

/* Y = row-wise softmax of X (see above).  Asynchronous on `stream`. */
GEMM_API gemm_status_t softmax_rows(const float* X, int64_t ldx, float* Y, int64_t ldy,
                                    int64_t M, int64_t N, struct CUstream_st* stream);

/* The configuration softmax_rows would use for these arguments, without
 * launching anything.  Same argument checks and errors as softmax_rows. */
GEMM_API gemm_status_t softmax_rows_query(const float* X, int64_t ldx, const float* Y,
                                          int64_t ldy, int64_t M, int64_t N,
                                          softmax_config_t* out);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_05_GB300_SOFTMAX_H */
