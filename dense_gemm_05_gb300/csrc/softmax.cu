// softmax.cu -- row-wise softmax on GB300 (sm_103a), fp32 in and out: the C ABI
// declared in include/softmax.h.
//
// What is computed: chapter 2 of "Writing GPU kernels in Triton: Vector Add,
// Softmax, MatMul" -- every row on its own (section 2.4), by the five steps of
// section 2.3 (max, subtract, exp, sum, divide).  The chapter's kernel holds a
// whole row in one program and reads it once (section 2.7, "kernel fusion");
// the same holds here while a row fits in the registers of one warp
// (N <= 2048) or of one 512-thread CTA (N <= 32768).  Longer rows stream
// through a 1024-thread CTA twice: a first pass keeps a running maximum and a
// running sum rescaled whenever the maximum grows, a second pass writes
// exp(x - m) / s.  Out-of-range columns simply take no part (the effect of the
// chapter's -inf padding of section 2.6).
//
// Memory: softmax moves 8 bytes per element (one fp32 read, one fp32 write)
// for a handful of flops, so it is bound by HBM bandwidth.  Rows are read with
// 16-byte streaming loads (ld.global.cs) when the row starts are 16-byte
// aligned, all of a thread's loads issued before the first use, and written
// with 16-byte streaming stores; the grid is persistent (a multiple of the SM
// count, from the occupancy of each instantiation) and walks the rows.
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/softmax.h"
#include "common.cuh"
#include "ptx.cuh"

namespace {

// Set by a staged kernel whose bounded wait gave up (checked in debug-sync mode).
__device__ int g_softmax_status;

constexpr int kWarpRowsBlock = 256;   // warp path: 8 rows per CTA
constexpr int kCtaThreads = 512;      // CTA path: one row per 512-thread CTA
constexpr int kStreamThreads = 1024;  // streaming path: one row per 1024-thread CTA
constexpr int kStreamSlab = 16;       // floats a thread loads per step of the streaming path
constexpr int kMaxWarpN = 2048;
// exp(t) is evaluated as exp2f(t * log2(e)) (measured faster than expf here):
// the extra rounding of the product adds a relative error of at most
// u * |t| to the result, the same size as the rounding of t = x - m itself.
constexpr float kLog2e = 1.4426950408889634f;
constexpr int kMaxCtaN = 32768;

// NaN-propagating maximum: a NaN in either operand wins (fmaxf would drop it).
// The one-pass paths use fmaxf: there a NaN entry still reaches the row sum
// (exp(NaN - m) = NaN) and so every output of its row, and entries beyond N
// hold -inf, which adds exp(-inf - m) = 0 whenever the row is finite (and a
// row that is not finite is NaN anyway).  The two-pass path skips slabs whose
// maximum is -inf, so it needs the NaN-propagating form.
__device__ __forceinline__ float max_nan(float a, float b) { return (b > a || b != b) ? b : a; }

// Butterfly reductions: every lane ends with the same bits (each step adds a
// value to its partner's, and a + b == b + a).
__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v = max_nan(v, __shfl_xor_sync(0xffffffffu, v, o));
    return v;
}

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
    return v;
}

// Reductions over a whole CTA of NT threads (NT a multiple of 32, <= 1024).
template <int NT>
__device__ __forceinline__ float cta_max(float v, float* red) {
    v = warp_max(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = (l < NT / 32) ? red[l] : -INFINITY;
    r = warp_max(r);
    __syncthreads();   // red is reused by the next reduction
    return r;
}

template <int NT>
__device__ __forceinline__ float cta_sum(float v, float* red) {
    v = warp_sum(v);
    const int w = threadIdx.x >> 5, l = threadIdx.x & 31;
    if (l == 0) red[w] = v;
    __syncthreads();
    float r = (l < NT / 32) ? red[l] : 0.0f;
    r = warp_sum(r);
    __syncthreads();
    return r;
}

// Load the W floats of one chunk that starts at column col (-inf beyond N).
// NC: through the read-only data path (ld.global.nc), which measured faster
// for the 512-thread rows; otherwise a streaming load (ld.global.cs).
// row = X + r * ldx; a checked build tests each load against the M x N matrix.
template <int W, bool NC = false>
__device__ __forceinline__ void load_chunk(const float* row, int64_t r, int64_t M, int64_t col,
                                           int64_t N, float* v) {
    if (W == 4 && col + 3 < N) {
        if (!DG_CHECK(&g_softmax_status, dg::kChkA, dg::span_inside(r, col, 4, M, N))) {
            v[0] = v[1] = v[2] = v[3] = -INFINITY;
            return;
        }
        const float4* p = reinterpret_cast<const float4*>(row + col);
        const float4 q = NC ? __ldg(p) : __ldcs(p);
        v[0] = q.x;
        v[1] = q.y;
        v[2] = q.z;
        v[3] = q.w;
    } else {
#pragma unroll
        for (int e = 0; e < W; ++e)
            v[e] = (col + e < N &&
                    DG_CHECK(&g_softmax_status, dg::kChkA, dg::span_inside(r, col + e, 1, M, N)))
                       ? (NC ? __ldg(row + col + e) : __ldcs(row + col + e))
                       : -INFINITY;
    }
}

// row = Y + r * ldy; a checked build tests each store against the M x N matrix.
template <int W>
__device__ __forceinline__ void store_chunk(float* row, int64_t r, int64_t M, int64_t col, int64_t N,
                                            const float* v) {
    if (W == 4 && col + 3 < N) {
        if (DG_CHECK(&g_softmax_status, dg::kChkC, dg::span_inside(r, col, 4, M, N)))
            __stcs(reinterpret_cast<float4*>(row + col), make_float4(v[0], v[1], v[2], v[3]));
    } else {
#pragma unroll
        for (int e = 0; e < W; ++e)
            if (col + e < N &&
                DG_CHECK(&g_softmax_status, dg::kChkC, dg::span_inside(r, col + e, 1, M, N)))
                __stcs(row + col + e, v[e]);
    }
}

// Register paths: TPR threads share a row (32: a warp, several rows per CTA;
// kCtaThreads: the whole CTA).  Thread t holds chunks j = 0..C-1 of W floats
// at columns (j*TPR + t)*W, so a warp's loads of one chunk are contiguous.
template <int TPR, int C, int W>
__global__ void __launch_bounds__(TPR == 32 ? kWarpRowsBlock : TPR)
    softmax_rows_reg_kernel(const float* X, int64_t ldx, float* Y, int64_t ldy, int64_t M,
                            int64_t N) {
    constexpr int kBlock = TPR == 32 ? kWarpRowsBlock : TPR;
    constexpr int kRows = kBlock / TPR;
    constexpr int kE = C * W;
    __shared__ float red[32];
    const int t = threadIdx.x % TPR;
    const int g = threadIdx.x / TPR;
    dg::griddep_wait();              // X may be written, Y still read, by the previous grid
    dg::griddep_launch_dependents();
    for (int64_t r = int64_t(blockIdx.x) * kRows + g; r < M; r += int64_t(gridDim.x) * kRows) {
        const float* xr = X + r * ldx;
        float* yr = Y + r * ldy;
        float v[kE];
#pragma unroll
        for (int j = 0; j < C; ++j)
            load_chunk<W, (TPR > 32)>(xr, r, M, int64_t(j * TPR + t) * W, N, v + j * W);

        // Max
        float m = -INFINITY;
#pragma unroll
        for (int i = 0; i < kE; ++i) m = fmaxf(m, v[i]);
        m = (TPR == 32) ? warp_max(m) : cta_max<TPR>(m, red);

        // Subtract, Exp, Sum
        float s = 0.0f;
#pragma unroll
        for (int i = 0; i < kE; ++i) {
            v[i] = exp2f((v[i] - m) * kLog2e);
            s += v[i];
        }
        s = (TPR == 32) ? warp_sum(s) : cta_sum<TPR>(s, red);

        // Divide (scale by 1/s), store
        const float inv = 1.0f / s;
#pragma unroll
        for (int i = 0; i < kE; ++i) v[i] *= inv;
#pragma unroll
        for (int j = 0; j < C; ++j) store_chunk<W>(yr, r, M, int64_t(j * TPR + t) * W, N, v + j * W);
    }
}

// Staged paths (row starts 16-byte aligned): one producer warp streams this
// CTA's rows -- a contiguous block of rows -- into a ring of shared-memory
// slots with bulk asynchronous copies (cp.async.bulk, completion counted on
// the slot's `full` mbarrier), so that many rows are in flight from HBM while
// the consumer warps reduce earlier ones.  A consumer group (one warp per row,
// or all NW consumer warps on one row when GROUPED) copies its row from the
// slot into registers, hands the slot back (`empty` mbarrier), and finishes
// exactly as the register path: max, exp(x - m), sum, scale by 1/sum,
// 16-byte streaming stores.  The copy covers the first 4*floor(N/4) floats; the last
// N mod 4 are read directly.  Every wait is bounded.
template <bool GROUPED, int NW, int CPL>
__global__ void __launch_bounds__(32 * (NW + 1), 1)
    softmax_rows_staged_kernel(const float* X, int64_t ldx, float* Y, int64_t ldy, int64_t M,
                               int64_t N, int slots, int slot_bytes, int y_vec,
                               uint64_t timeout_ns) {
    constexpr int kTpr = GROUPED ? NW * 32 : 32;     // threads per row
    constexpr int kGroups = GROUPED ? 1 : NW;
    extern __shared__ __align__(128) uint8_t smem[];
    uint64_t* full = reinterpret_cast<uint64_t*>(smem + size_t(slots) * slot_bytes);
    uint64_t* empty = full + slots;
    __shared__ float red[2][32];
    __shared__ volatile int abort_flag;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int64_t r0 = M * blockIdx.x / gridDim.x;
    const int64_t r1 = M * (blockIdx.x + 1) / gridDim.x;
    const int64_t count = r1 - r0;
    const int64_t n4 = N & ~int64_t(3);               // floats moved by the bulk copy
    const uint32_t bulk_bytes = static_cast<uint32_t>(n4 * 4);

    if (threadIdx.x == 0) {
        for (int i = 0; i < slots; ++i) {
            dg::mbar_init(dg::smem_u32(&full[i]), 1u);
            dg::mbar_init(dg::smem_u32(&empty[i]), 1u);
        }
        abort_flag = 0;
        dg::fence_mbar_init();
    }
    __syncthreads();
    dg::griddep_wait();              // X may be written, Y still read, by the previous grid
    dg::griddep_launch_dependents();

    if (warp == NW) {
        // ------------------------------------------------------------ producer
        if (lane == 0) {
            for (int64_t i = 0; i < count; ++i) {
                const int slot = static_cast<int>(i % slots);
                const uint32_t k = static_cast<uint32_t>(i / slots);
                if (!dg::mbar_wait(dg::smem_u32(&empty[slot]), (k & 1u) ^ 1u, &abort_flag,
                                   timeout_ns)) {
                    abort_flag = 1;
                    atomicOr(&g_softmax_status, dg::kDevTimeout);
                    break;
                }
                const uint32_t fb = dg::smem_u32(&full[slot]);
                if (bulk_bytes == 0u ||
                    !DG_CHECK(&g_softmax_status, dg::kChkA, dg::span_inside(r0 + i, 0, n4, M, N))) {
                    dg::mbar_arrive(fb);
                    continue;
                }
                dg::mbar_arrive_expect_tx(fb, bulk_bytes);
                const char* src = reinterpret_cast<const char*>(X + (r0 + i) * ldx);
                const uint32_t dst = dg::smem_u32(smem + size_t(slot) * slot_bytes);
                for (uint32_t off = 0; off < bulk_bytes; off += 32768u) {
                    const uint32_t n = bulk_bytes - off < 32768u ? bulk_bytes - off : 32768u;
                    dg::bulk_load_g2s(dst + off, src + off, n, fb);
                }
            }
        }
        __syncwarp();
    } else {
        // ------------------------------------------------------------ consumers
        const int g = GROUPED ? 0 : warp;
        const int t = GROUPED ? threadIdx.x : lane;
        int buf = 0;
        for (int64_t i = g; i < count; i += kGroups) {
            const int slot = static_cast<int>(i % slots);
            const uint32_t k = static_cast<uint32_t>(i / slots);
            bool ok = dg::mbar_wait(dg::smem_u32(&full[slot]), k & 1u, &abort_flag, timeout_ns);
            if (GROUPED) ok = dg::named_bar_and(1, kTpr, ok);
            if (!ok) {
                abort_flag = 1;
                atomicOr(&g_softmax_status, dg::kDevTimeout);
                break;
            }
            const float* srow = reinterpret_cast<const float*>(smem + size_t(slot) * slot_bytes);
            const float* xr = X + (r0 + i) * ldx;
            float v[CPL * 4];
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int64_t col = int64_t(j * kTpr + t) * 4;
                if (col + 3 < N) {
                    const float4 q = *reinterpret_cast<const float4*>(srow + col);
                    v[4 * j] = q.x;
                    v[4 * j + 1] = q.y;
                    v[4 * j + 2] = q.z;
                    v[4 * j + 3] = q.w;
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        v[4 * j + e] = (col + e < N && DG_CHECK(&g_softmax_status, dg::kChkA,
                                                                 dg::span_inside(r0 + i, col + e, 1, M, N)))
                                           ? __ldcs(xr + col + e)
                                           : -INFINITY;
                }
            }
            // Max (the group's barrier also orders every thread's slot reads
            // before the slot is handed back)
            float m = -INFINITY;
#pragma unroll
            for (int q = 0; q < CPL * 4; ++q) m = fmaxf(m, v[q]);
            m = warp_max(m);
            if (GROUPED) {
                if (lane == 0) red[buf][warp] = m;
                dg::named_bar_sync(1, kTpr);
                float r = lane < NW ? red[buf][lane] : -INFINITY;
                m = warp_max(r);
                buf ^= 1;
                if (threadIdx.x == 0) dg::mbar_arrive(dg::smem_u32(&empty[slot]));
            } else {
                __syncwarp();
                if (lane == 0) dg::mbar_arrive(dg::smem_u32(&empty[slot]));
            }
            // Subtract, Exp, Sum
            float s = 0.0f;
#pragma unroll
            for (int q = 0; q < CPL * 4; ++q) {
                v[q] = exp2f((v[q] - m) * kLog2e);
                s += v[q];
            }
            s = warp_sum(s);
            if (GROUPED) {
                if (lane == 0) red[buf][warp] = s;
                dg::named_bar_sync(1, kTpr);
                float r = lane < NW ? red[buf][lane] : 0.0f;
                s = warp_sum(r);
                buf ^= 1;
            }
            // Divide (scale by 1/s), store
            float* yr = Y + (r0 + i) * ldy;
            const float inv = 1.0f / s;
#pragma unroll
            for (int q = 0; q < CPL * 4; ++q) v[q] *= inv;
#pragma unroll
            for (int j = 0; j < CPL; ++j) {
                const int64_t col = int64_t(j * kTpr + t) * 4;
                if (y_vec && col + 3 < N) {
                    if (DG_CHECK(&g_softmax_status, dg::kChkC, dg::span_inside(r0 + i, col, 4, M, N)))
                        __stcs(reinterpret_cast<float4*>(yr + col),
                               make_float4(v[4 * j], v[4 * j + 1], v[4 * j + 2], v[4 * j + 3]));
                } else {
#pragma unroll
                    for (int e = 0; e < 4; ++e)
                        if (col + e < N &&
                            DG_CHECK(&g_softmax_status, dg::kChkC, dg::span_inside(r0 + i, col + e, 1, M, N)))
                            __stcs(yr + col + e, v[4 * j + e]);
                }
            }
        }
    }
    if (abort_flag) {
        // Copies already issued still land in this CTA's shared memory: give them
        // a bounded 2 ms before the CTA leaves.
        const uint64_t t0 = dg::global_timer_ns();
        while (dg::global_timer_ns() - t0 < 2000000ull) {
        }
    }
}

// Streaming path for rows longer than a CTA's registers hold.  Pass 1: each
// thread walks its columns kStreamSlab floats at a time and keeps (m, s) with
// s = sum of exp(x - m) over what it has seen; when a slab raises m, s is
// rescaled by exp(m_old - m_new) once.  The CTA then combines the (m, s) pairs
// the same way.  Pass 2 reads the row again and writes exp(x - m) / s.
template <int W>
__global__ void __launch_bounds__(kStreamThreads)
    softmax_rows_stream_kernel(const float* X, int64_t ldx, float* Y, int64_t ldy, int64_t M,
                               int64_t N) {
    constexpr int kChunks = kStreamSlab / W;
    constexpr int64_t kStep = int64_t(kStreamThreads) * kStreamSlab;
    __shared__ float red[32];
    const int t = threadIdx.x;
    dg::griddep_wait();              // X may be written, Y still read, by the previous grid
    dg::griddep_launch_dependents();
    for (int64_t r = blockIdx.x; r < M; r += gridDim.x) {
        const float* xr = X + r * ldx;
        float* yr = Y + r * ldy;
        float m = -INFINITY, s = 0.0f;
        for (int64_t base = 0; base < N; base += kStep) {
            float v[kStreamSlab];
#pragma unroll
            for (int j = 0; j < kChunks; ++j)
                load_chunk<W>(xr, r, M, base + int64_t(j * kStreamThreads + t) * W, N, v + j * W);
            float mm = m;
#pragma unroll
            for (int i = 0; i < kStreamSlab; ++i) mm = max_nan(mm, v[i]);
            if (mm == -INFINITY) continue;   // only -inf (or nothing) so far: s stays 0
            float acc = 0.0f;
#pragma unroll
            for (int i = 0; i < kStreamSlab; ++i) acc += expf(v[i] - mm);   // -inf entries add 0
            s = (m == -INFINITY ? 0.0f : s * expf(m - mm)) + acc;
            m = mm;
        }
        const float mr = cta_max<kStreamThreads>(m, red);
        const float sr = cta_sum<kStreamThreads>(m == -INFINITY ? 0.0f : s * expf(m - mr), red);
        const float inv = 1.0f / sr;
        for (int64_t base = 0; base < N; base += kStep) {
            float v[kStreamSlab];
#pragma unroll
            for (int j = 0; j < kChunks; ++j)
                load_chunk<W>(xr, r, M, base + int64_t(j * kStreamThreads + t) * W, N, v + j * W);
#pragma unroll
            for (int i = 0; i < kStreamSlab; ++i) v[i] = expf(v[i] - mr) * inv;
#pragma unroll
            for (int j = 0; j < kChunks; ++j)
                store_chunk<W>(yr, r, M, base + int64_t(j * kStreamThreads + t) * W, N, v + j * W);
        }
    }
}

// ---------------------------------------------------------------- host side

using KernelFn = void (*)(const float*, int64_t, float*, int64_t, int64_t, int64_t);
using StagedFn = void (*)(const float*, int64_t, float*, int64_t, int64_t, int64_t, int, int, int,
                          uint64_t);

constexpr int kStagedGroupWarps = 16;    // consumer warps of the grouped staged path
constexpr int kMinStagedN = 8192;        // shorter rows: the register paths measured faster
constexpr int kMaxStagedN = 24576;       // two 96 KiB slots
constexpr int kStagedSmem = 200 * 1024;  // ring of row slots
constexpr int kMaxSlots = 32;
constexpr uint64_t kTimeoutNs = 2000000000ull;

struct Choice {
    softmax_config_t cfg;
    KernelFn fn = nullptr;     // register and streaming paths
    StagedFn sfn = nullptr;    // staged paths
    int slot_bytes = 0;
    int smem = 0;
};

template <int TPR, int C, int W>
Choice reg_choice(int path) {
    Choice c{};
    c.fn = softmax_rows_reg_kernel<TPR, C, W>;
    c.cfg.path = path;
    c.cfg.threads_per_row = TPR;
    c.cfg.elems_per_thread = C * W;
    c.cfg.vec = W;
    c.cfg.block = TPR == 32 ? kWarpRowsBlock : TPR;
    c.cfg.rows_per_cta = c.cfg.block / TPR;
    return c;
}

template <bool GROUPED, int NW, int CPL>
Choice staged_choice(int64_t N) {
    Choice c{};
    c.sfn = softmax_rows_staged_kernel<GROUPED, NW, CPL>;
    c.cfg.path = GROUPED ? SOFTMAX_PATH_CTA : SOFTMAX_PATH_WARP;
    c.cfg.threads_per_row = GROUPED ? NW * 32 : 32;
    c.cfg.elems_per_thread = CPL * 4;
    c.cfg.block = 32 * (NW + 1);
    c.cfg.staged = 1;
    const int64_t bytes = (N & ~int64_t(3)) * 4;
    c.slot_bytes = static_cast<int>(bytes < 128 ? 128 : (bytes + 127) / 128 * 128);
    int slots = kStagedSmem / c.slot_bytes;
    c.cfg.slots = slots < kMaxSlots ? slots : kMaxSlots;
    c.smem = c.cfg.slots * c.slot_bytes + c.cfg.slots * 16;
    return c;
}

Choice choose(int64_t N, bool vec, bool staged) {
    if (staged && N > kMinStagedN && N <= kMaxStagedN) {
        if (N <= 16384) return staged_choice<true, kStagedGroupWarps, 8>(N);
        return staged_choice<true, kStagedGroupWarps, 12>(N);
    }
    if (N <= kMaxWarpN) {
        if (vec) {
            if (N <= 128) return reg_choice<32, 1, 4>(SOFTMAX_PATH_WARP);
            if (N <= 256) return reg_choice<32, 2, 4>(SOFTMAX_PATH_WARP);
            if (N <= 512) return reg_choice<32, 4, 4>(SOFTMAX_PATH_WARP);
            if (N <= 1024) return reg_choice<32, 8, 4>(SOFTMAX_PATH_WARP);
            return reg_choice<32, 16, 4>(SOFTMAX_PATH_WARP);
        }
        if (N <= 128) return reg_choice<32, 4, 1>(SOFTMAX_PATH_WARP);
        if (N <= 256) return reg_choice<32, 8, 1>(SOFTMAX_PATH_WARP);
        if (N <= 512) return reg_choice<32, 16, 1>(SOFTMAX_PATH_WARP);
        if (N <= 1024) return reg_choice<32, 32, 1>(SOFTMAX_PATH_WARP);
        return reg_choice<32, 64, 1>(SOFTMAX_PATH_WARP);
    }
    if (N <= kMaxCtaN) {
        if (vec) {
            if (N <= 4096) return reg_choice<kCtaThreads, 2, 4>(SOFTMAX_PATH_CTA);
            if (N <= 8192) return reg_choice<kCtaThreads, 4, 4>(SOFTMAX_PATH_CTA);
            if (N <= 16384) return reg_choice<kCtaThreads, 8, 4>(SOFTMAX_PATH_CTA);
            return reg_choice<kCtaThreads, 16, 4>(SOFTMAX_PATH_CTA);
        }
        if (N <= 4096) return reg_choice<kCtaThreads, 8, 1>(SOFTMAX_PATH_CTA);
        if (N <= 8192) return reg_choice<kCtaThreads, 16, 1>(SOFTMAX_PATH_CTA);
        if (N <= 16384) return reg_choice<kCtaThreads, 32, 1>(SOFTMAX_PATH_CTA);
        return reg_choice<kCtaThreads, 64, 1>(SOFTMAX_PATH_CTA);
    }
    Choice c{};
    c.fn = vec ? softmax_rows_stream_kernel<4> : softmax_rows_stream_kernel<1>;
    c.cfg.path = SOFTMAX_PATH_STREAM;
    c.cfg.threads_per_row = kStreamThreads;
    c.cfg.elems_per_thread = kStreamSlab;
    c.cfg.vec = vec ? 4 : 1;
    c.cfg.block = kStreamThreads;
    c.cfg.rows_per_cta = 1;
    return c;
}

// Per-device facts, looked up once per device.
struct DeviceFacts {
    bool known = false;
    bool sm103 = false;
    int sms = 0;
};

std::mutex g_dev_mu;
DeviceFacts g_dev[64];

bool device_facts(DeviceFacts* out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(g_dev_mu);
    DeviceFacts& f = g_dev[dev];
    if (!f.known) {
        int major = 0, minor = 0, sms = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        f.sm103 = major == 10 && minor == 3;
        f.sms = sms;
        f.known = true;
    }
    *out = f;
    return true;
}

bool overlaps(const float* a, int64_t lda, const float* b, int64_t ldb, int64_t M, int64_t N) {
    const uintptr_t a0 = reinterpret_cast<uintptr_t>(a);
    const uintptr_t b0 = reinterpret_cast<uintptr_t>(b);
    const uintptr_t a1 = a0 + static_cast<uintptr_t>(((M - 1) * lda + N) * 4);
    const uintptr_t b1 = b0 + static_cast<uintptr_t>(((M - 1) * ldb + N) * 4);
    return a0 < b1 && b0 < a1;
}

gemm_status_t check(const float* X, int64_t ldx, const float* Y, int64_t ldy, int64_t M,
                    int64_t N) {
    if (M < 0 || N < 0) return GEMM_ERR_INVALID_ARG;
    if (M == 0 || N == 0) return GEMM_OK;
    if (X == nullptr || Y == nullptr) return GEMM_ERR_INVALID_ARG;
    if (ldx < N || ldy < N) return GEMM_ERR_INVALID_ARG;
    if ((reinterpret_cast<uintptr_t>(X) | reinterpret_cast<uintptr_t>(Y)) % 4u != 0u)
        return GEMM_ERR_INVALID_ARG;
    if (M > INT32_MAX || N > INT32_MAX || ldx > (int64_t(1) << 40) || ldy > (int64_t(1) << 40))
        return GEMM_ERR_UNSUPPORTED;
    const bool same = X == Y && ldx == ldy;
    if (!same && overlaps(X, ldx, Y, ldy, M, N)) return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

gemm_status_t plan(const float* X, int64_t ldx, const float* Y, int64_t ldy, int64_t M,
                   int64_t N, Choice* c) {
    const gemm_status_t st = check(X, ldx, Y, ldy, M, N);
    if (st != GEMM_OK) return st;
    if (M == 0 || N == 0) {
        *c = Choice{};
        c->cfg.path = SOFTMAX_PATH_NONE;
        return GEMM_OK;
    }
    DeviceFacts f;
    if (!device_facts(&f)) return GEMM_ERR_CUDA;
    if (!f.sm103) return GEMM_ERR_UNSUPPORTED;
    const bool x16 = reinterpret_cast<uintptr_t>(X) % 16u == 0u && ldx % 4 == 0;
    const bool y16 = reinterpret_cast<uintptr_t>(Y) % 16u == 0u && ldy % 4 == 0;
    *c = choose(N, x16 && y16, x16);
    int per_sm = 0;
    if (c->sfn != nullptr) {
        c->cfg.vec = y16 ? 4 : 1;
        if (cudaFuncSetAttribute(c->sfn, cudaFuncAttributeMaxDynamicSharedMemorySize, c->smem) !=
                cudaSuccess ||
            cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, c->sfn, c->cfg.block,
                                                          c->smem) != cudaSuccess) {
            (void)cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
    } else if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, c->fn, c->cfg.block, 0) !=
               cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (per_sm < 1) return GEMM_ERR_UNSUPPORTED;
    const int64_t cap = int64_t(f.sms) * per_sm;
    if (c->sfn != nullptr) {
        // Contiguous blocks of rows, one block per CTA.
        c->cfg.grid = static_cast<int>(M < cap ? M : cap);
        c->cfg.rows_per_cta = static_cast<int>((M + c->cfg.grid - 1) / c->cfg.grid);
    } else {
        // One-warp rows longer than 128 floats: one row per warp and no row loop
        // (measured 9 % faster at N = 1000 than a persistent grid, whose warps
        // each wait out one row's load latency after another); other paths: a
        // persistent grid of `cap` CTAs.
        const int64_t need = (M + c->cfg.rows_per_cta - 1) / c->cfg.rows_per_cta;
        const bool one_pass = c->cfg.path == SOFTMAX_PATH_WARP && N > 128;
        c->cfg.grid = static_cast<int>((one_pass || need < cap) ? need : cap);
    }
    return GEMM_OK;
}

bool debug_sync() {
    static const bool on = [] {
        const char* e = std::getenv("GEMM_DEBUG_SYNC");
        return e != nullptr && e[0] == '1';
    }();
    return on;
}

}  // namespace

extern "C" {

gemm_status_t softmax_rows(const float* X, int64_t ldx, float* Y, int64_t ldy, int64_t M,
                           int64_t N, struct CUstream_st* stream) {
    Choice c;
    const gemm_status_t st = plan(X, ldx, Y, ldy, M, N, &c);
    if (st != GEMM_OK || c.cfg.path == SOFTMAX_PATH_NONE) return st;
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Launched as programmatic dependents (the kernels wait before touching memory).
    const cudaError_t e =
        c.sfn != nullptr
            ? dg::launch_pdl(c.sfn, dim3(c.cfg.grid), dim3(c.cfg.block), size_t(c.smem), s, X, ldx,
                             Y, ldy, M, N, int(c.cfg.slots), int(c.slot_bytes),
                             int(c.cfg.vec == 4), kTimeoutNs)
            : dg::launch_pdl(c.fn, dim3(c.cfg.grid), dim3(c.cfg.block), size_t(0), s, X, ldx, Y,
                             ldy, M, N);
    if (e != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (debug_sync() && c.sfn != nullptr) {
        if (cudaStreamSynchronize(s) != cudaSuccess) {
            (void)cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        int status = 0;
        if (cudaMemcpyFromSymbol(&status, g_softmax_status, sizeof(int)) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (status != 0) {
            const int zero = 0;
            (void)cudaMemcpyToSymbol(g_softmax_status, &zero, sizeof(int));
            return (status & dg::kDevBounds) ? GEMM_ERR_BOUNDS : GEMM_ERR_TIMEOUT;
        }
    }
    return GEMM_OK;
}

gemm_status_t softmax_rows_query(const float* X, int64_t ldx, const float* Y, int64_t ldy,
                                 int64_t M, int64_t N, softmax_config_t* out) {
    if (out == nullptr) return GEMM_ERR_INVALID_ARG;
    Choice c;
    const gemm_status_t st = plan(X, ldx, Y, ldy, M, N, &c);
    if (st != GEMM_OK) return st;
    *out = c.cfg;
    return GEMM_OK;
}

}  // extern "C"
