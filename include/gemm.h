/*
 * gemm.h -- C ABI of the GB300 (sm_103a) dense matrix multiply library.
 *
 * Operation (the tiled matmul of "I Wrote a GPU Matmul Kernel From Scratch in
 * Triton", Steps 1-5, and of "Triton 04: Matmul, Autotune and PyTorch
 * integration", section "A teaching matmul kernel"):
 *
 *     C[i, j] = sum_{k=0}^{K-1} A[i, k] * B[k, j]      0 <= i < M, 0 <= j < N
 *
 * with A and B in fp16 or bf16 (both the same type), products accumulated in
 * fp32, and C written in fp32 (the output type of the teaching kernel's
 * wrapper on the "Triton 04" page).  All three matrices are row-major with
 * unit inner stride and an explicit leading dimension, in ELEMENTS, as in
 * section 4.1 of "Writing GPU kernels in Triton: Vector Add, Softmax, MatMul":
 *
 *     A[i, k] at A + i*lda + k     (lda >= K)
 *     B[k, j] at B + k*ldb + j     (ldb >= N)
 *     C[i, j] at C + i*ldc + j     (ldc >= N)
 *
 * Ragged edges are masked: elements outside the M x K, K x N and M x N
 * rectangles are never read (they act as zeros, the masked loads with
 * other=0 of Step 3) and never written (the masked store).  C is overwritten;
 * its previous contents never matter.
 *
 * Threading / ownership: the caller owns A, B, C (device memory) and the
 * stream.  A plan owns a small device workspace (split-K partial sums and
 * tile counters) and must not be used by two gemm_run calls that can be in
 * flight at the same time on different streams; use one plan per stream.
 * Nothing here synchronises the stream unless GEMM_DEBUG_SYNC=1 is set in the
 * environment (then gemm_run waits for the kernel and reports device-side
 * timeouts as GEMM_ERR_TIMEOUT).
 */
#ifndef DENSE_GEMM_05_GB300_GEMM_H
#define DENSE_GEMM_05_GB300_GEMM_H

#include <stdint.h>

#if defined(__GNUC__)
#define GEMM_API __attribute__((visibility("default")))
#else
#define GEMM_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

struct CUstream_st;                         /* == cudaStream_t / CUstream */
typedef struct gemm_plan_s *gemm_plan_t;    /* opaque */

typedef enum {
    GEMM_F16 = 0,   /* IEEE binary16 inputs */
    GEMM_BF16 = 1   /* bfloat16 inputs */
} gemm_dtype_t;

typedef enum {
    GEMM_OK = 0,
    GEMM_ERR_INVALID_ARG = 1,   /* null pointer / plan, negative size, ld too small, overlap,
                                   misaligned element pointer */
    GEMM_ERR_UNSUPPORTED = 2,   /* unknown dtype, not an sm_103 device, size beyond 2^31-1 */
    GEMM_ERR_CUDA = 3,          /* a CUDA runtime/driver call failed (launch error etc.) */
    GEMM_ERR_OOM = 4,           /* workspace allocation failed */
    GEMM_ERR_TIMEOUT = 5,       /* a bounded device-side wait gave up (debug-sync mode) */
    GEMM_ERR_BOUNDS = 6         /* checked build, debug-sync mode: a kernel skipped an access
                                   outside its matrix or buffer (gemm_build_checked) */
} gemm_status_t;

/* Storage of an operand for gemm_run_ex (the operation is always C = A @ B):
 *   A: GEMM_OP_N  A[i, k] at A + i*lda + k   (stored M x K, lda >= K)
 *      GEMM_OP_T  A[i, k] at A + k*lda + i   (stored K x M, lda >= M)
 *   B: GEMM_OP_N  B[k, j] at B + k*ldb + j   (stored K x N, ldb >= N)
 *      GEMM_OP_T  B[k, j] at B + j*ldb + k   (stored N x K, ldb >= K: the
 *                 [out_features, in_features] layout of a linear layer's weight)
 * The pages allow any strides (the stride_ak / stride_bk arguments of the
 * autotuned kernel of Step 5 and of the "Triton 04" teaching kernel); these
 * are the two unit-stride cases of each operand. */
typedef enum { GEMM_OP_N = 0, GEMM_OP_T = 1 } gemm_op_t;

/* Element type of C for gemm_run_ex.  16-bit outputs are the fp32 accumulator
 * rounded to nearest-even once, as the fp16 store of section 4.5 of "Writing
 * GPU kernels in Triton: Vector Add, Softmax, MatMul" (acc.to(float16)). */
typedef enum { GEMM_OUT_F32 = 0, GEMM_OUT_F16 = 1, GEMM_OUT_BF16 = 2 } gemm_out_t;

/* Which kernel gemm_run selects for a problem (see gemm_query). */
typedef enum {
    GEMM_KERNEL_NONE = 0,       /* M == 0 or N == 0: nothing is launched */
    GEMM_KERNEL_ZERO_FILL = 1,  /* K == 0: C is set to zero (the empty sum) */
    GEMM_KERNEL_TMA = 2,        /* persistent warp-specialised tcgen05 kernel fed by TMA;
                                   tiles of 128 x 64/128/256, or 64 x 64 (M = 64 MMAs) for
                                   problems whose 128 x 64 tiles fill at most half the SMs */
    GEMM_KERNEL_GENERIC = 3,    /* same pipeline, operands staged by ordinary loads
                                   (leading dimensions or pointers not 16-byte aligned) */
    GEMM_KERNEL_SKINNY = 4,     /* small M: swap-AB + split-K, deterministic reduction */
    GEMM_KERNEL_PAIR = 5,       /* 2-SM (cta_group::2) pair tiles for large problems */
    GEMM_KERNEL_SPLIT_PAIR = 6  /* a 2-CTA cluster per output tile (M <= 64: a strip of all
                                   rows x block_n columns; else 128 x 128) splits K in
                                   halves; the halves' fp32 partials meet in distributed
                                   shared memory (no workspace, deterministic).  Chosen for
                                   M <= 64 when the first wave of strips keeps >= 3/5 of the
                                   SMs busy and K >= 1024, and for M > 64 when the 128 x 128
                                   tiles fit one wave of clusters and K >= 768 */
} gemm_kernel_t;

typedef struct {
    int32_t kernel;       /* gemm_kernel_t */
    int32_t block_m;      /* rows of C per tile (per CTA pair for GEMM_KERNEL_PAIR; 128 or 64
                             for TMA; the padded M, 16, 32 or 64, for SKINNY and SPLIT_PAIR) */
    int32_t block_n;      /* columns of C per tile (SPLIT_PAIR: 128, 192 or 256 per strip) */
    int32_t block_k;      /* K depth of one pipeline stage */
    int32_t stages;       /* shared-memory ring depth */
    int32_t split_k;      /* most K slices any output tile is split into (1 = none) */
    int32_t grid;         /* CTAs launched (persistent kernels: one per SM or fewer) */
    int32_t cluster;      /* CTAs per cluster */
    int32_t group;        /* group-major strip height in tiles (0 = row-major order) */
    int32_t tiles;        /* work units: output tiles, or stream-K shares for SKINNY */
    int32_t shares;       /* SKINNY: equal contiguous shares of the (tile, K block) iterations;
                             PAIR: shares (one per cluster) of the stream-K phase, 0 = none */
    int32_t staged;       /* bit 1: A copied to 16-byte-aligned rows first; bit 2: B copied;
                             bit 4: B (stored K x N, not 16-byte aligned) read in place by the
                             SPLIT_PAIR kernel's own copies, no staging pass */
} gemm_config_t;

/*
 * Create a plan on CUDA device `device` (that device becomes current for the
 * call).  Checks that the device is compute capability 10.3, queries the SM
 * count, sets kernel attributes and allocates the plan's workspace (64 MiB of
 * split-K / stream-K partials, tile counters, a status word) and its 32 MiB
 * staging buffer.
 * Errors: INVALID_ARG (out == NULL), UNSUPPORTED (not sm_103), CUDA, OOM (an
 * allocation failed; whatever was allocated is freed again).  On error *out is
 * set to NULL.  For tests, GEMM_TEST_FAIL_ALLOC=k in the environment makes the
 * k-th of the four allocations fail as if the device were out of memory.
 */
GEMM_API gemm_status_t gemm_plan_create(gemm_plan_t *out, int device);

/*
 * C = A @ B (see the top of this file).  Asynchronous on `stream` (NULL = the
 * legacy default stream); A, B, C are device pointers; dtype is the type of
 * both A and B.  A and B must be 2-byte aligned, C 4-byte aligned.
 * The region written, rows [0, M) x columns [0, N) of C, must not overlap the
 * regions read from A or B.
 * M == 0 or N == 0: no-op.  K == 0: C[0:M, 0:N] = 0.
 * An operand whose base or row pitch is not a multiple of 16 bytes (e.g. an
 * odd ld) is first copied by a kernel into the plan's 32 MiB staging buffer
 * with rows padded to 16 bytes, when it fits (both together when both are),
 * and the tensor-memory-access kernels read the copy; larger ones are read in
 * place by the generic kernel.  Consecutive calls on one plan reuse the buffer
 * in stream order.  A misaligned B too large for the buffer, with an aligned A,
 * in a problem that goes to the SPLIT_PAIR kernel with 128 x 128 tiles (M >
 * 64), is read in place by that kernel instead of the generic kernel
 * (gemm_config_t.staged bit 4; see also gemm_plan_set_staging).
 * Errors: INVALID_ARG, UNSUPPORTED, CUDA (launch failure), TIMEOUT (only in
 * debug-sync mode).  Nothing is launched when an error is returned, except
 * for CUDA/TIMEOUT, which report a failure of the launched work itself.
 */
GEMM_API gemm_status_t gemm_run(gemm_plan_t plan,
                       const void *A, int64_t lda,
                       const void *B, int64_t ldb,
                       float *C, int64_t ldc,
                       int64_t M, int64_t N, int64_t K,
                       gemm_dtype_t dtype, struct CUstream_st *stream);

/*
 * gemm_run with operand storage and output type chosen by the caller:
 * C = A @ B with A and B stored as op_a / op_b describe (gemm_op_t), fp32
 * accumulation, and C[i, j] at C + i*ldc + j of type c_type (gemm_out_t).
 * gemm_run(...) is gemm_run_ex(GEMM_OP_N, GEMM_OP_N, ..., GEMM_OUT_F32, ...).
 * C must be aligned to its element size.  Same asynchrony, ownership, size
 * rules and errors as gemm_run; INVALID_ARG also for an unknown op, and
 * UNSUPPORTED for an unknown c_type.
 */
GEMM_API gemm_status_t gemm_run_ex(gemm_plan_t plan, gemm_op_t op_a, gemm_op_t op_b,
                                   const void *A, int64_t lda,
                                   const void *B, int64_t ldb,
                                   void *C, int64_t ldc, gemm_out_t c_type,
                                   int64_t M, int64_t N, int64_t K,
                                   gemm_dtype_t dtype, struct CUstream_st *stream);

/* gemm_query for the arguments of gemm_run_ex. */
GEMM_API gemm_status_t gemm_query_ex(gemm_plan_t plan, gemm_op_t op_a, gemm_op_t op_b,
                                     const void *A, int64_t lda,
                                     const void *B, int64_t ldb,
                                     const void *C, int64_t ldc, gemm_out_t c_type,
                                     int64_t M, int64_t N, int64_t K,
                                     gemm_dtype_t dtype, gemm_config_t *out);

/*
 * A plan for a modelled device, for gemm_query / gemm_query_ex only: the kernel
 * and configuration choice of a device with `num_sms` SMs and the given numbers
 * of co-resident 2-CTA clusters for the pair kernel (128- and 256-column tiles)
 * and the split-pair kernel (a GB300 reports 152, 76, 76, 76), with the
 * workspace, staging and counter capacities of a device plan.  Touches no
 * device and allocates no device memory, so the planner can be examined on a
 * host without a GPU; the query's pointer arguments are only checked for
 * alignment and overlap.  gemm_run / gemm_run_ex on it return INVALID_ARG;
 * gemm_plan_force and gemm_plan_set_group apply as to a device plan.
 * Errors: INVALID_ARG (null out, num_sms outside 1..4096, a cluster count
 * negative or above num_sms / 2), OOM.
 */
GEMM_API gemm_status_t gemm_plan_create_model(gemm_plan_t *out, int32_t num_sms,
                                              int32_t pair_clusters_128,
                                              int32_t pair_clusters_256,
                                              int32_t splitpair_clusters);

/* Release the plan and its workspace.  NULL-safe.  Waits for nothing: the
 * caller must make sure no gemm_run using the plan is still in flight. */
GEMM_API gemm_status_t gemm_plan_destroy(gemm_plan_t plan);

/* Static, human-readable name of a status code. */
GEMM_API const char *gemm_status_string(gemm_status_t s);

/*
 * Report the kernel and configuration gemm_run would use for these
 * arguments, without launching anything (the offline-tuned replacement of the
 * autotune step of Step 5 / the "What autotune selects" section).
 * Same argument checks and errors as gemm_run.
 */
GEMM_API gemm_status_t gemm_query(gemm_plan_t plan,
                         const void *A, int64_t lda,
                         const void *B, int64_t ldb,
                         const float *C, int64_t ldc,
                         int64_t M, int64_t N, int64_t K,
                         gemm_dtype_t dtype, gemm_config_t *out);

/*
 * Override the plan's tile order for the persistent kernels: group > 0 is the
 * group-major order of Step 4 with strips `group` tiles tall; group == 0 is
 * the row-major order of the "Triton 04" teaching kernel.  Default 8.
 * Errors: INVALID_ARG (null plan, group < 0 or > 64).
 */
GEMM_API gemm_status_t gemm_plan_set_group(gemm_plan_t plan, int32_t group);

/*
 * Force the next gemm_run calls on this plan to use `kernel` (a
 * gemm_kernel_t of TMA, GENERIC, SKINNY, PAIR or SPLIT_PAIR; 0 = automatic choice),
 * `split_k` stream-K shares for SKINNY -- the (tile, K block) iterations of
 * all tiles are cut into that many equal contiguous runs, one CTA each
 * (0 = automatic); for PAIR, `split_k` = 1 turns off the stream-K phase that
 * otherwise splits the last, partial wave of pair tiles (plus one full wave)
 * by K across all clusters, `split_k` = 2 splits every tile's K loop over all
 * clusters (whole-problem stream-K), `split_k` = 3 runs the stream-K phase for any
 * partial last wave, any other value = automatic -- and `block_n`
 * tile columns for TMA/PAIR (128 or 256) or strip columns for SPLIT_PAIR (128,
 * 192 or 256; 0 = automatic).  For tests and tuning.
 * gemm_run returns UNSUPPORTED when the forced kernel cannot run the given
 * arguments (e.g. SKINNY with M > 64, SPLIT_PAIR with K < 128, with A transposed,
 * or with block_n other than 128 for M > 64, block_n 192 with another kernel, or
 * TMA with an operand that is neither
 * 16-byte aligned nor small enough for the staging buffer).  Forcing GENERIC
 * also turns staging off (misaligned operands are read in place).
 * Errors: INVALID_ARG (null plan, unknown kernel, negative split, bad block_n).
 */
GEMM_API gemm_status_t gemm_plan_force(gemm_plan_t plan, int32_t kernel, int32_t split_k,
                                       int32_t block_n);

/*
 * Debug settings of the plan's next gemm_run calls.  sync = 1: gemm_run waits
 * for its kernels and returns GEMM_ERR_TIMEOUT when a bounded device-side wait
 * gave up (the device status word is then cleared, and so are the plan's tile
 * counters, which a kernel that stopped early may leave non-zero); sync = 0:
 * no waiting (the default, unless GEMM_DEBUG_SYNC=1 was set when the plan was
 * created).  timeout_ns: the limit of every bounded wait in the kernels, 0 =
 * the default of 2 s (GEMM_WAIT_TIMEOUT_MS at plan creation also sets it).  A
 * wait that gives up stops its CTA and the others it works with after their
 * copies and MMAs in flight have landed; C is then incomplete.  A wait gives
 * up a few to a few tens of microseconds after its limit (its polls suspend
 * the thread for up to about a microsecond each, on the hardware's schedule).
 * A limit far below a kernel's run time makes real launches give up: the
 * tests use that to exercise the path, and the context stays usable afterwards.
 * Errors: INVALID_ARG (null plan, sync not 0 or 1).
 */
GEMM_API gemm_status_t gemm_plan_set_debug(gemm_plan_t plan, int32_t sync, uint64_t timeout_ns);

/*
 * Checked builds.  The same sources compiled with DG_CHECKED=1 give a second
 * library, libgemm_checked.so, with this same ABI.  In it every ordinary
 * (non-TMA) global load and store of the kernels (the GEMM kernels, and those of
 * softmax.h and attention.h) first tests the range it
 * touches against the matrix or buffer it belongs to: A, B and C against the
 * rows x columns rectangles the caller passed (so a row's padding between N and
 * ldc counts as outside), the staging copy against its source and destination,
 * split-K partials and tile counters against the plan's workspace.  An access
 * that fails the test is skipped -- it never reaches memory -- and sets a bit
 * of the plan's device status word: 2 (out of range) plus one bit per kind of
 * access, 1<<8 C store, 1<<9 A load, 1<<10 B load, 1<<11 workspace,
 * 1<<12 tile counter, 1<<13 staging copy.  A debug-sync gemm_run (see
 * gemm_plan_set_debug) then returns GEMM_ERR_BOUNDS (softmax_rows and
 * attention_fwd likewise under GEMM_DEBUG_SYNC=1); without debug-sync the
 * word is cleared unread by the next debug-sync call.  A partial tile whose
 * workspace range fails stops its kernel as a wait that gave up does.  TMA copies
 * are not tested: their tensor maps bound them in hardware (elements outside
 * read as zeros, stores are clipped).  There is no counterpart in the pages;
 * the checked build stands in for a memory checker, and runs slower.
 *
 * gemm_build_checked: 1 in the checked library, 0 in the normal one.
 * gemm_plan_device_status: the status word the plan's last debug-sync gemm_run
 * read (0: none; 1 = a wait gave up; 2 and the bits above = out of range).
 * Errors: INVALID_ARG (null plan or word).
 */
GEMM_API int32_t gemm_build_checked(void);
GEMM_API gemm_status_t gemm_plan_device_status(gemm_plan_t plan, int32_t* word);

/*
 * Turn the staging of misaligned operands on (1, the default) or off (0) for
 * the next gemm_run calls on this plan.  With staging off, an operand whose
 * base or row pitch is not a multiple of 16 bytes is never copied: a K x N B
 * with an aligned A in a SPLIT_PAIR-sized problem (M > 64) is read in place by
 * that kernel, anything else by the generic kernel.  For tests, tuning, and
 * callers that want no extra pass over their operands.
 * Errors: INVALID_ARG (null plan, enabled not 0 or 1).
 */
GEMM_API gemm_status_t gemm_plan_set_staging(gemm_plan_t plan, int32_t enabled);

/*
 * The scheduler's tile order, evaluated on the host by the same function the
 * kernels use: linear work index t -> (tile_m, tile_n) for a grid of
 * tiles_m x tiles_n tiles and strip height `group` (0 = row-major).
 * Errors: INVALID_ARG (null outputs, t outside [0, tiles_m*tiles_n), bad sizes).
 */
GEMM_API gemm_status_t gemm_tile_coord(int64_t t, int64_t tiles_m, int64_t tiles_n, int32_t group,
                              int64_t *tile_m, int64_t *tile_n);

/*
 * Device-side wait self-test: launches one block that waits on a shared-memory
 * barrier nobody arrives on, with a limit of `timeout_us` microseconds, then
 * synchronises `stream`.  Returns GEMM_ERR_TIMEOUT when the bounded wait gave
 * up as designed (the expected result), GEMM_OK if it did not time out, or
 * GEMM_ERR_CUDA.  Used by tests to check that every spin-wait in the kernels
 * ends; the CUDA context stays usable afterwards.
 */
GEMM_API gemm_status_t gemm_wait_selftest(uint32_t timeout_us, struct CUstream_st *stream);

/*
 * Launch floor probe (the pages have no counterpart): enqueue on `stream` one
 * kernel that does no work, launched the way the GEMM kernels are -- `grid`
 * CTAs of 192 threads in clusters of `cluster` (1 or 2) CTAs, as a
 * programmatic dependent of the previous work in the stream (it waits for
 * that work, then lets the next kernel start).  Timing a graph of these
 * launches gives the fixed cost that every launch of a short GEMM pays, the
 * bound against which the small problems are measured.  Asynchronous; reads
 * and writes no memory.
 * Errors: INVALID_ARG (grid outside 1..65535, cluster not 1 or 2, grid not a
 * multiple of cluster), CUDA (launch failure).
 */
GEMM_API gemm_status_t gemm_noop_launch(int32_t grid, int32_t cluster, struct CUstream_st *stream);

/*
 * ---------------------------------------------------------------- partitioned GEMM
 * C = A @ B split over `world` devices by output rows or columns, the "rank
 * offset" of "How to hand-write Triton kernels for matmul and Flash Attention"
 * (engineering advice: each device takes different output blocks).  The
 * slices need no exchange of data to compute: by rows, rank r multiplies its
 * rows of A by all of B into its rows of C; by columns, all of A by its
 * columns of B into its columns of C.  (Gathering C onto every device, where
 * that is wanted, is the caller's collective; the Python binding has one.)
 */
typedef enum {
    GEMM_SPLIT_AUTO = -1,   /* rows, or columns when M <= 64 (B is then the large operand) */
    GEMM_SPLIT_M = 0,       /* rows of A and C */
    GEMM_SPLIT_N = 1        /* columns of B and C */
} gemm_split_t;

typedef struct {
    int32_t axis;           /* GEMM_SPLIT_M or GEMM_SPLIT_N */
    int32_t rank, world;
    int64_t row0, rows;     /* rows [row0, row0 + rows) of A and C */
    int64_t col0, cols;     /* columns [col0, col0 + cols) of B and C */
} gemm_slice_t;

/*
 * The slice of the M x N output that rank `rank` of `world` computes: the
 * split axis is cut into units of 128 (the kernels' tile edge), U units in
 * all, and rank r takes units [floor(r U / world), floor((r + 1) U / world)),
 * clipped to the matrix -- contiguous, disjoint, in rank order, covering the
 * axis, their sizes differing by at most one unit, every boundary but the
 * matrix's end a multiple of 128 (so operand offsets keep their alignment).
 * A rank may get an empty slice (rows or cols 0) when U < world.  The other
 * axis is whole.  Pure host arithmetic; no device is touched.
 * Errors: INVALID_ARG (null out, negative sizes, world < 1, rank outside
 * [0, world), unknown axis).
 */
GEMM_API gemm_status_t gemm_partition(int64_t M, int64_t N, int64_t K, int32_t world,
                                      int32_t rank, int32_t axis, gemm_slice_t *out);

/*
 * Compute one slice of C = A @ B: C[row0 : row0 + rows, col0 : col0 + cols] =
 * A[row0 : row0 + rows, :] @ B[:, col0 : col0 + cols], with A, B and C given
 * as the whole matrices' layouts (the pointers and leading dimensions of
 * gemm_run; the slice must lie inside M x N).  It is gemm_run on the offset
 * pointers, with the same asynchrony, ownership and errors; an empty slice is
 * a no-op.  Running every rank's slice (on one device one after another, or on
 * each rank's own device with its own copies) writes all of C, bit for bit as
 * one gemm_run would where the kernel choice is the same.
 * Errors: INVALID_ARG (null plan or slice, a slice outside M x N or with an
 * unknown axis) and those of gemm_run.
 */
GEMM_API gemm_status_t gemm_run_slice(gemm_plan_t plan, const gemm_slice_t *slice,
                                      const void *A, int64_t lda,
                                      const void *B, int64_t ldb,
                                      float *C, int64_t ldc,
                                      int64_t M, int64_t N, int64_t K,
                                      gemm_dtype_t dtype, struct CUstream_st *stream);

/*
 * gemm_run_noalloc -- C = A @ B for small M without a plan and without any
 * allocation.  The pages have no counterpart to this entry point; it exists
 * for callers that cannot allocate device memory.  A serving process that
 * gives all free device memory to its own pool at start-up has none left for
 * a library's workspace, and a latency-sensitive loop that shares the GPU
 * with other streams cannot take the device-wide synchronisation that
 * cudaMalloc/cudaFree may cause.  Such callers pass A, B and C as usual; the
 * scratch the split-K kernel needs (fp32 partial tiles, a status word and
 * per-tile counters) lives in one static device array of
 * GEMM_NOALLOC_SCRATCH_BYTES, which a device holds from this entry point's
 * first call on it until the process exits.
 *
 * Same operation, layout and argument rules as gemm_run, on the CURRENT device
 * and `stream`.  Limits: M <= GEMM_NOALLOC_MAX_M, N <= GEMM_NOALLOC_MAX_N,
 * A and B 16-byte aligned with lda and ldb multiples of 8 elements; anything
 * beyond them returns GEMM_ERR_UNSUPPORTED and launches nothing.  The K split
 * is chosen to fit the scratch.  This call never calls cudaMalloc, cudaFree or
 * any allocating routine.
 *
 * Set-up: the first call on a device (any call that passes the size checks,
 * including one with M == 0 or N == 0, which launches nothing) checks the
 * architecture, sets kernel attributes and looks up the scratch array's device
 * address.  With CUDA's default lazy module loading, that is the moment the
 * array and this entry point's kernels are placed in device memory, so a
 * caller that will later give all free memory to its own pool makes its first
 * call -- e.g. gemm_run_noalloc(NULL, 0, NULL, 0, NULL, 0, 0, 0, 0, GEMM_BF16,
 * NULL) -- before it does, and before any stream capture.  A set-up that
 * fails is retried by the next call.  With CUDA_MODULE_LOADING=EAGER the array
 * is placed when the library is loaded.
 *
 * Every call on a device shares the one scratch array, which keeps the last
 * call's contents (each call clears the status word and the counters it
 * uses): calls that can overlap on the GPU -- on different streams, or from
 * different threads -- race and give wrong results.  Serialise them.
 *
 * Errors: INVALID_ARG and UNSUPPORTED as above, CUDA for a failed set-up or
 * launch.  A bounded device-side wait that gives up (the kernel then stops
 * and C is left incomplete) is recorded in the status word but NOT reported
 * by the call, which does not wait for the kernel -- unless GEMM_DEBUG_SYNC=1
 * was set when the device was set up: then every call waits for its kernel
 * and returns GEMM_ERR_TIMEOUT for a wait that gave up.
 */
#define GEMM_NOALLOC_MAX_M 64
#define GEMM_NOALLOC_MAX_N 131072
#define GEMM_NOALLOC_SCRATCH_BYTES 8392960   /* 8 MiB of partial tiles, 16 B of status, 4 KiB of
                                                counters, rounded up to 256 B */
GEMM_API gemm_status_t gemm_run_noalloc(const void *A, int64_t lda,
                                        const void *B, int64_t ldb,
                                        float *C, int64_t ldc,
                                        int64_t M, int64_t N, int64_t K,
                                        gemm_dtype_t dtype, struct CUstream_st *stream);

#ifdef __cplusplus
}
#endif

#endif /* DENSE_GEMM_05_GB300_GEMM_H */
