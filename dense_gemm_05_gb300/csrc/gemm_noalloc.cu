// gemm_noalloc.cu -- gemm_run_noalloc: the small-M (swap-AB, split-K) GEMM run
// without a plan and without allocating anything.
//
// gemm_run needs a plan, and a plan allocates its split-K workspace with
// cudaMalloc.  Some callers cannot do that: a serving process that hands all
// free device memory to its own pool at start-up has nothing left to give a
// library later, and latency-sensitive loops that share the GPU with other
// streams cannot afford the device-wide synchronisation that cudaMalloc and
// cudaFree may bring.  For them this entry point keeps the scratch memory the
// kernel needs -- fp32 partial tiles and per-tile arrival counters -- in one
// fixed array of static device memory that every GPU which loads the library
// holds until the process exits.  The caller still passes A, B and C.
#include <atomic>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gemm.h"
#include "common.cuh"
#include "ptx.cuh"

namespace {

// Layout of the scratch array: fp32 partial tiles, then (256 bytes further on)
// the device status word, then the per-tile arrival counters right behind it,
// so that one memset clears the status word and the counters a call uses.
constexpr int64_t kScratchWsBytes = int64_t(8) << 20;
constexpr int64_t kStatusOffset = kScratchWsBytes;
constexpr int64_t kCountersOffset = kStatusOffset + 16;
constexpr int kScratchCounters = 1024;   // one per 128-column tile of C
static_assert(int64_t(kScratchCounters) * 128 == GEMM_NOALLOC_MAX_N, "counter capacity");
static_assert(kCountersOffset + kScratchCounters * 4 <= GEMM_NOALLOC_SCRATCH_BYTES, "layout");

}  // namespace

// The scratch array.  In host code this name is only a stand-in; its device
// address comes from cudaGetSymbolAddress below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[GEMM_NOALLOC_SCRATCH_BYTES];

namespace {

constexpr int kMaxDevices = 64;

// Per-device set-up.  A set-up that failed is not remembered: the next call
// on that device tries again (the failure may have been a transient lack of
// device memory for the array or the kernels' code).
struct DeviceState {
    std::mutex mu;
    std::atomic<bool> ready{false};
    unsigned char* scratch = nullptr;   // device address of g_noalloc_scratch on this device
    int num_sms = 0;
    bool debug_sync = false;
};

DeviceState g_state[kMaxDevices];

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);
EncodeTiledFn g_encode = nullptr;
std::once_flag g_encode_once;

// Set-up for the current device: architecture check, kernel attributes (which
// also loads the kernels onto the device), and the device address of the
// scratch array (which loads the array).  Done under the device's lock until it
// succeeds once; afterwards the fast path only reads `ready`.
gemm_status_t setup_device(DeviceState* s, int dev) {
    if (s->ready.load(std::memory_order_acquire)) return GEMM_OK;
    std::lock_guard<std::mutex> lock(s->mu);
    if (s->ready.load(std::memory_order_relaxed)) return GEMM_OK;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
    if (dg::skinny_prepare() != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    s->scratch = static_cast<unsigned char*>(ptr);
    s->num_sms = sms;
    const char* v = std::getenv("GEMM_DEBUG_SYNC");
    s->debug_sync = v != nullptr && v[0] != '\0' && v[0] != '0';
    s->ready.store(true, std::memory_order_release);
    return GEMM_OK;
}

bool encode_2d(CUtensorMap* map, gemm_dtype_t dt, const void* ptr, int64_t inner, int64_t outer,
               int64_t ld, uint32_t box_inner, uint32_t box_outer) {
    std::call_once(g_encode_once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            g_encode = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    if (g_encode == nullptr) return false;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * 2u};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1u, 1u};
    return g_encode(map,
                    dt == GEMM_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16,
                    2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                    CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

bool aligned16(const void* p, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(p) % 16u) == 0u && (ld * 2) % 16 == 0;
}

bool disjoint(const void* p, uint64_t plen, const void* q, uint64_t qlen) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return !(a < b + qlen && b < a + plen);
}

}  // namespace

extern "C" gemm_status_t gemm_run_noalloc(const void* A, int64_t lda, const void* B, int64_t ldb,
                                          float* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                                          gemm_dtype_t dtype, struct CUstream_st* stream_handle) {
    if (M < 0 || N < 0 || K < 0) return GEMM_ERR_INVALID_ARG;
    if (dtype != GEMM_F16 && dtype != GEMM_BF16) return GEMM_ERR_UNSUPPORTED;
    if (M > GEMM_NOALLOC_MAX_M || N > GEMM_NOALLOC_MAX_N || K > INT32_MAX - 1024)
        return GEMM_ERR_UNSUPPORTED;

    // The device set-up comes first, so that a call with M == 0 or N == 0 (which
    // launches nothing) can be used to do it at a time of the caller's choosing.
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (dev < 0 || dev >= kMaxDevices) return GEMM_ERR_UNSUPPORTED;
    DeviceState* s = &g_state[dev];
    const gemm_status_t ready = setup_device(s, dev);
    if (ready != GEMM_OK) return ready;
    if (M == 0 || N == 0) return GEMM_OK;

    if (C == nullptr || ldc < N || ldc > (int64_t(1) << 40) ||
        reinterpret_cast<uintptr_t>(C) % 4u != 0u)
        return GEMM_ERR_INVALID_ARG;
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    if (K == 0) {
        if (cudaMemset2DAsync(C, static_cast<size_t>(ldc) * 4u, 0, static_cast<size_t>(N) * 4u,
                              static_cast<size_t>(M), stream) != cudaSuccess) {
            (void)cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        return GEMM_OK;
    }
    if (A == nullptr || B == nullptr || lda < K || ldb < N || lda > (int64_t(1) << 40) ||
        ldb > (int64_t(1) << 40))
        return GEMM_ERR_INVALID_ARG;
    if (reinterpret_cast<uintptr_t>(A) % 2u != 0u || reinterpret_cast<uintptr_t>(B) % 2u != 0u)
        return GEMM_ERR_INVALID_ARG;
    const uint64_t a_len = (uint64_t(M - 1) * uint64_t(lda) + uint64_t(K)) * 2u;
    const uint64_t b_len = (uint64_t(K - 1) * uint64_t(ldb) + uint64_t(N)) * 2u;
    const uint64_t c_len = (uint64_t(M - 1) * uint64_t(ldc) + uint64_t(N)) * 4u;
    if (!disjoint(C, c_len, A, a_len) || !disjoint(C, c_len, B, b_len))
        return GEMM_ERR_INVALID_ARG;
    // The kernel stages A and B with TMA: 16-byte aligned bases and pitches.
    if (!aligned16(A, lda) || !aligned16(B, ldb)) return GEMM_ERR_UNSUPPORTED;

    // Stream-K shares as gemm_run chooses them; if their partial tiles would not
    // fit the scratch, one share per tile (no partials).
    const int ms = M <= 16 ? 16 : (M <= 32 ? 32 : 64);
    const int tiles_n = static_cast<int>(cdiv(N, 128));
    const int num_kb = static_cast<int>(cdiv(K, dg::kBK));
    const int64_t T = int64_t(tiles_n) * num_kb;
    int64_t shares = dg::skinny_auto_shares(tiles_n, num_kb, s->num_sms);
    if (shares != tiles_n &&
        int64_t(tiles_n) * dg::shares_per_tile_bound(T, shares, num_kb) * ms * 128 * 4 >
            kScratchWsBytes)
        shares = tiles_n;
    const int max_slots = dg::shares_per_tile_bound(T, shares, num_kb);
    int* status = reinterpret_cast<int*>(s->scratch + kStatusOffset);
    int* counters = reinterpret_cast<int*>(s->scratch + kCountersOffset);
    // The array keeps whatever the previous call left: the status word and the
    // counters this call uses must start at zero.
    if (cudaMemsetAsync(status, 0, static_cast<size_t>(kCountersOffset - kStatusOffset) +
                                       sizeof(int) * static_cast<size_t>(tiles_n),
                        stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }

    CUtensorMap mb, ma;
    if (!encode_2d(&mb, dtype, B, N, K, ldb, dg::kSubN, dg::kBK) ||
        !encode_2d(&ma, dtype, A, K, M, lda, dg::kBK, static_cast<uint32_t>(ms)))
        return GEMM_ERR_CUDA;
    dg::Params p{};
    p.A = static_cast<const uint16_t*>(A);
    p.B = static_cast<const uint16_t*>(B);
    p.C = C;
    p.c_type = 0;   // fp32 C
    p.lda = lda;
    p.ldb = ldb;
    p.ldc = ldc;
    p.M = static_cast<int32_t>(M);
    p.N = static_cast<int32_t>(N);
    p.K = static_cast<int32_t>(K);
    p.tiles_m = 1;
    p.tiles_n = tiles_n;
    p.num_kb = num_kb;
    p.group = 0;
    p.shares = static_cast<int32_t>(shares);
    p.max_slots = max_slots;
    p.a_vec = 1;
    p.b_vec = 1;
    p.c_vec = 0;
    p.ws = reinterpret_cast<float*>(s->scratch);
    p.counters = counters;
    p.ws_len = kScratchWsBytes / static_cast<int64_t>(sizeof(float));
    p.counters_len = kScratchCounters;
    p.status = status;
    p.timeout_ns = 2000000000ull;
    const int grid = shares < s->num_sms ? static_cast<int>(shares) : s->num_sms;
    const bool bf16 = dtype == GEMM_BF16;
    if (dg::launch_skinny(ms, true, mb, ma, p, dg::idesc_f16(bf16, true, false, 128, ms), grid,
                          stream) != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (s->debug_sync) {
        // Debug mode: wait for the kernel and report a bounded wait that gave up.
        int dev_status = 0;
        if (cudaStreamSynchronize(stream) != cudaSuccess ||
            cudaMemcpy(&dev_status, status, sizeof(int), cudaMemcpyDeviceToHost) != cudaSuccess) {
            (void)cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        if (dev_status & dg::kDevBounds) return GEMM_ERR_BOUNDS;
        if (dev_status != 0) return GEMM_ERR_TIMEOUT;
    }
    return GEMM_OK;
}
