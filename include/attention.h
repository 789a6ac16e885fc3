/*
 * attention.h -- C ABI of the attention forward pass of the GB300 (sm_103a)
 * library (libgemm.so; status codes and element types shared with gemm.h).
 *
 * Operation (section "Flash Attention in Triton and online softmax" of "How to
 * hand-write Triton kernels for matmul and Flash Attention"): for each of BH
 * independent heads with Q, K, V of shape [seq, d],
 *
 *     O = softmax_rows(Q K^T / sqrt(d)) V,
 *
 * where, with `causal` set, score (i, j) takes part only for j <= i (the
 * section's causal mask keeps query >= key).  Computed as the section does:
 * one program per block of 128 queries walks the key/value blocks with a
 * running row maximum, a rescaled running sum and a rescaled accumulator (the
 * online softmax), so the seq x seq score matrix is never written to memory.
 * Q K^T and P V run on the tensor cores (fp16/bf16 operands, fp32
 * accumulation); the probabilities P are rounded to the input type before the
 * second product; the row sum is kept in fp32.  The launch is persistent: at
 * most one CTA per SM, each walking a fixed share of the work items (one
 * block of 128 queries of one head for d = 128, two for d = 64); a query
 * block's result does not depend on which CTA computes it.
 *
 * Layout: Q, K and V share one layout: element (h, i, c) at
 *     ptr + h*head_stride + i*ld + c          (c < d, i < seq, h < BH)
 * in elements (ld >= d; row-major heads [BH, seq, d] have ld = d and
 * head_stride = seq*d; interleaved layouts such as [seq, BH, d] are other
 * strides).  O: element (h, i, c) at O + h*head_stride_o + i*ldo + c, of type
 * out_type.  Keys i >= seq do not exist (they take no part; the section's
 * kernel leaves that boundary handling out).
 *
 * Limits: d == 64 or 128; ld and head_stride multiples of 8 elements and Q, K, V
 * 16-byte aligned (tensor-memory-access boxes); BH <= 65535; seq <= 2^31 - 256.
 *
 * Ownership: the caller owns all buffers and the stream; nothing is allocated
 * and nothing synchronises (unless GEMM_DEBUG_SYNC=1: then the call waits and
 * reports a device-side wait that gave up as GEMM_ERR_TIMEOUT, and in the
 * checked build an O store outside its rows as GEMM_ERR_BOUNDS).
 *
 * Errors: GEMM_ERR_INVALID_ARG for null pointers (when BH*seq > 0), negative
 * sizes, ld < d, ldo < d, misaligned pointers, or O overlapping Q, K or V;
 * GEMM_ERR_UNSUPPORTED for d other than 64 or 128, strides that are not multiples of 8,
 * BH > 65535, seq > 2^31 - 256, an unknown dtype/out_type, or a device that is not sm_103;
 * GEMM_ERR_CUDA when the launch fails.  BH == 0 or seq == 0 is a no-op.
 */
#ifndef DENSE_GEMM_05_GB300_ATTENTION_H
#define DENSE_GEMM_05_GB300_ATTENTION_H

#include "gemm.h"

#ifdef __cplusplus
extern "C" {
#endif

typedef struct {
    int32_t block_q;      /* queries per block (TMEM lanes) */
    int32_t block_kv;     /* keys per step of the online softmax */
    int32_t head_dim;
    int32_t stages;       /* K/V shared-memory ring depth */
    int32_t grid_x;       /* work items per head (two query blocks each for d = 64, one for 128) */
    int32_t grid_y;       /* heads; the persistent launch has min(grid_x * grid_y, SMs) CTAs */
    int32_t causal;
} attention_config_t;

GEMM_API gemm_status_t attention_fwd(const void* Q, const void* K, const void* V, void* O,
                                     int64_t BH, int64_t seq, int64_t d, int64_t ld,
                                     int64_t head_stride, int64_t ldo, int64_t head_stride_o,
                                     int32_t causal, gemm_dtype_t dtype, int32_t out_type,
                                     struct CUstream_st* stream);

/* The configuration attention_fwd would use, without launching.  Same checks. */
GEMM_API gemm_status_t attention_fwd_query(const void* Q, const void* K, const void* V,
                                           const void* O, int64_t BH, int64_t seq, int64_t d,
                                           int64_t ld, int64_t head_stride, int64_t ldo,
                                           int64_t head_stride_o, int32_t causal,
                                           gemm_dtype_t dtype, int32_t out_type,
                                           attention_config_t* out);

/*
 * Debug settings of every later attention_fwd call in the process (not tied to
 * a stream or thread; for tests).  sync = 1: the call waits for its kernel and
 * returns GEMM_ERR_TIMEOUT when a bounded device-side wait gave up; sync = 0:
 * no waiting, whatever GEMM_DEBUG_SYNC says; sync = -1: as GEMM_DEBUG_SYNC says
 * (the initial setting).  timeout_ns: the limit of every
 * bounded wait in the kernel, 0 = the default of 2 s.  A wait that gives up
 * stops its CTA after its MMAs have completed; O is then incomplete, and the
 * context stays usable.  A limit far below a launch's run time makes real
 * launches give up (a few to a few tens of microseconds after the limit).
 * Errors: INVALID_ARG (sync not -1, 0 or 1).
 */
GEMM_API gemm_status_t attention_set_debug(int32_t sync, uint64_t timeout_ns);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_05_GB300_ATTENTION_H */
