// gemm_api.cu -- the C ABI declared in include/gemm.h: argument checks, the
// plan (workspace, device facts, options), kernel selection (the offline
// replacement of the autotune step of "I Wrote a GPU Matmul Kernel From
// Scratch in Triton", Step 5), TMA descriptor encoding and launches.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <algorithm>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/gemm.h"
#include "common.cuh"
#include "ptx.cuh"

// Recently encoded TMA descriptors, keyed by everything they encode (address,
// extents, pitch, type, box): repeated calls on the same operands skip the
// driver's encoder.  The descriptor is passed to the kernel by value, so a
// cached entry never aliases one that a launch in flight still uses.
struct TmapCacheEntry {
    bool valid = false;
    const void* ptr = nullptr;
    int64_t inner = 0, outer = 0, ld = 0;
    int dtype = 0;
    uint32_t box_inner = 0, box_outer = 0;
    CUtensorMap map;
};

struct gemm_plan_s {
    std::mutex cache_mu;
    TmapCacheEntry cache[8];
    int cache_next = 0;
    int device = 0;
    int num_sms = 0;
    float* ws = nullptr;          // split-K partial tiles
    size_t ws_bytes = 0;
    int* counters = nullptr;      // split-K per-tile arrival counters (kept at zero)
    int counters_len = 0;
    int* status = nullptr;        // device error word
    uint16_t* stage = nullptr;    // copies of operands whose rows are not 16-byte aligned
    size_t stage_bytes = 0;
    int group = 8;
    int force_kernel = 0;
    int force_split = 0;
    int force_bn = 0;
    bool staging = true;             // copy misaligned operands to 16-byte rows when they fit
    int pair_clusters[2] = {0, 0};   // co-resident 2-CTA clusters for pair tiles of 128 / 256
    int splitpair_clusters = 0;         // co-resident 2-CTA clusters of the small-M cluster kernel
    bool debug_sync = false;
    int last_device_status = 0;      // status word seen by the last debug-sync gemm_run
    bool model = false;              // a device model for gemm_query only (no device, no memory)
    uint64_t timeout_ns = 2000000000ull;   // limit of every bounded device-side wait
};

namespace {

constexpr size_t kWorkspaceBytes = size_t(64) << 20;   // split-K / stream-K partials
constexpr uint64_t kDefaultTimeoutNs = 2000000000ull;  // 2 s per bounded device-side wait
constexpr int64_t kPairMinShareKb = 16;   // a pair stream-K share streams at least this many K blocks
constexpr size_t kStageBytes = size_t(32) << 20;       // staging copies of misaligned operands
constexpr int kPairMinSkKb = 32;          // K blocks per tile below which no pair stream-K phase
constexpr int kSplitPairMinKb = 12;       // K blocks below which M > 64 keeps one-CTA tiles
constexpr int kL2PrefetchKb = 6;          // split pair, one tile row: K blocks per CTA warmed in L2 early
constexpr int kL2PrefetchKbSkinny = 3;    // the same for the swap-AB stream-K kernel (deeper was slower)

// Kernel choice: flop/s each SM sustains on one tile of each kind, measured on
// GB300 with one wave of tiles (bf16, K = 8192): pair tiles 256 x 256 (two
// SMs), one-CTA tiles 128 x 256 and 128 x 128.  A one-CTA 128 x 128 tile loads
// twice the bytes per flop of a pair tile's half, which is why it is slowest.
constexpr double kRatePairPerSm = 10.6e12;
constexpr double kRateTma256PerSm = 9.1e12;
constexpr double kRateTma128PerSm = 6.6e12;

// Seconds for `tiles` equal tiles of `tile_flops` each on `slots` units that
// each run one tile at `rate` flop/s: whole waves times one tile's time.
double est_seconds(int64_t tiles, int64_t slots, double tile_flops, double rate) {
    const int64_t waves = (tiles + slots - 1) / slots;
    return static_cast<double>(waves) * tile_flops / rate;
}
constexpr int kMaxCounters = 1 << 16;                   // output tiles that may be split
constexpr int64_t kMaxDim = INT32_MAX - 1024;   // headroom for tile-edge arithmetic in int32

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(p);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// Element types of the tensors the library describes to TMA.
enum Elem : int { kElemF16 = 0, kElemBF16 = 1, kElemF32 = 2 };

Elem elem_of(gemm_dtype_t dt) { return dt == GEMM_BF16 ? kElemBF16 : kElemF16; }

Elem elem_of_out(int c_type) {
    return c_type == GEMM_OUT_F32 ? kElemF32 : (c_type == GEMM_OUT_BF16 ? kElemBF16 : kElemF16);
}

// Row-major [outer, inner] matrix with row pitch ld (elements), tiles of
// box_outer x box_inner elements, 128-byte swizzle, zero fill out of bounds.
bool encode_2d(CUtensorMap* map, Elem et, const void* ptr, int64_t inner, int64_t outer,
               int64_t ld, uint32_t box_inner, uint32_t box_outer) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    const uint64_t esize = et == kElemF32 ? 4u : 2u;
    const CUtensorMapDataType t = et == kElemF32    ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32
                                  : et == kElemBF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(outer)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(ld) * esize};
    cuuint32_t box[2] = {box_inner, box_outer};
    cuuint32_t estr[2] = {1u, 1u};
    CUresult r = fn(map, t, 2, const_cast<void*>(ptr), dims, strides, box, estr,
                    CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                    CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS;
}

bool cached_encode_2d(gemm_plan_s* plan, CUtensorMap* map, Elem dt, const void* ptr,
                      int64_t inner, int64_t outer, int64_t ld, uint32_t box_inner,
                      uint32_t box_outer) {
    std::lock_guard<std::mutex> lock(plan->cache_mu);
    for (const TmapCacheEntry& e : plan->cache) {
        if (e.valid && e.ptr == ptr && e.inner == inner && e.outer == outer && e.ld == ld &&
            e.dtype == static_cast<int>(dt) && e.box_inner == box_inner &&
            e.box_outer == box_outer) {
            *map = e.map;
            return true;
        }
    }
    if (!encode_2d(map, dt, ptr, inner, outer, ld, box_inner, box_outer)) return false;
    TmapCacheEntry& e = plan->cache[plan->cache_next];
    plan->cache_next = (plan->cache_next + 1) % 8;
    e.valid = true;
    e.ptr = ptr;
    e.inner = inner;
    e.outer = outer;
    e.ld = ld;
    e.dtype = static_cast<int>(dt);
    e.box_inner = box_inner;
    e.box_outer = box_outer;
    e.map = *map;
    return true;
}

bool tma_ok(const void* ptr, int64_t ld) {
    return (reinterpret_cast<uintptr_t>(ptr) % 16u) == 0u && ((ld * 2) % 16) == 0;
}

int64_t cdiv(int64_t a, int64_t b) { return (a + b - 1) / b; }

struct Args {
    const void* A;
    int64_t lda;
    const void* B;
    int64_t ldb;
    const void* C;
    int64_t ldc;
    int64_t M, N, K;
    gemm_dtype_t dtype;
    int op_a = GEMM_OP_N;       // GEMM_OP_T: A stored K x M
    int op_b = GEMM_OP_N;       // GEMM_OP_T: B stored N x K
    int c_type = GEMM_OUT_F32;

    int64_t c_esize() const { return c_type == GEMM_OUT_F32 ? 4 : 2; }
    // Stored shapes (rows x cols, row pitch = ld) of A and B.
    int64_t a_rows() const { return op_a == GEMM_OP_N ? M : K; }
    int64_t a_cols() const { return op_a == GEMM_OP_N ? K : M; }
    int64_t b_rows() const { return op_b == GEMM_OP_N ? K : N; }
    int64_t b_cols() const { return op_b == GEMM_OP_N ? N : K; }
};

struct Choice {
    int kernel = GEMM_KERNEL_NONE;
    int bn = 0;          // TMA/GENERIC: tile columns
    int bm = 128;        // TMA: tile rows (128, or 64 with bn = 64)
    int ms = 0;          // SKINNY, SPLIT_PAIR: padded M
    int split = 1;       // SKINNY: most stream-K shares that touch one tile
    int shares = 0;      // SKINNY: stream-K shares
    int max_slots = 0;   // SKINNY: workspace slots per tile
    int sk_tiles = 0;    // PAIR: tiles in the stream-K phase
    int tiles_m = 0, tiles_n = 0, num_kb = 0;
    int units = 0;
    int grid = 0;
    int stages = 0;
};

// Last byte (exclusive) touched by a row-major rows x cols region with pitch ld.
bool region_end(int64_t rows, int64_t cols, int64_t ld, int64_t esize, uint64_t* end_bytes) {
    // rows, cols <= 2^31 - 1 and ld <= 2^40 were checked by the caller.
    const unsigned __int128 e =
        (static_cast<unsigned __int128>(rows - 1) * static_cast<uint64_t>(ld) +
         static_cast<uint64_t>(cols)) *
        static_cast<uint64_t>(esize);
    if (e > static_cast<unsigned __int128>(UINT64_MAX / 2)) return false;
    *end_bytes = static_cast<uint64_t>(e);
    return true;
}

bool overlaps(const void* p, uint64_t plen, const void* q, uint64_t qlen) {
    const uintptr_t a = reinterpret_cast<uintptr_t>(p), b = reinterpret_cast<uintptr_t>(q);
    return a < b + qlen && b < a + plen;
}

gemm_status_t check_args(const Args& a) {
    if (a.M < 0 || a.N < 0 || a.K < 0) return GEMM_ERR_INVALID_ARG;
    if ((a.op_a != GEMM_OP_N && a.op_a != GEMM_OP_T) ||
        (a.op_b != GEMM_OP_N && a.op_b != GEMM_OP_T))
        return GEMM_ERR_INVALID_ARG;
    if (a.dtype != GEMM_F16 && a.dtype != GEMM_BF16) return GEMM_ERR_UNSUPPORTED;
    if (a.c_type != GEMM_OUT_F32 && a.c_type != GEMM_OUT_F16 && a.c_type != GEMM_OUT_BF16)
        return GEMM_ERR_UNSUPPORTED;
    if (a.M > kMaxDim || a.N > kMaxDim || a.K > kMaxDim) return GEMM_ERR_UNSUPPORTED;
    if (a.M == 0 || a.N == 0) return GEMM_OK;
    constexpr int64_t kMaxLd = int64_t(1) << 40;
    if (a.C == nullptr || a.ldc < a.N) return GEMM_ERR_INVALID_ARG;
    if (a.ldc > kMaxLd) return GEMM_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(a.C) % static_cast<uintptr_t>(a.c_esize()) != 0u)
        return GEMM_ERR_INVALID_ARG;
    uint64_t c_end = 0;
    if (!region_end(a.M, a.N, a.ldc, a.c_esize(), &c_end)) return GEMM_ERR_UNSUPPORTED;
    if (a.K == 0) return GEMM_OK;
    if (a.A == nullptr || a.B == nullptr || a.lda < a.a_cols() || a.ldb < a.b_cols())
        return GEMM_ERR_INVALID_ARG;
    if (a.lda > kMaxLd || a.ldb > kMaxLd) return GEMM_ERR_UNSUPPORTED;
    if (reinterpret_cast<uintptr_t>(a.A) % 2u != 0u || reinterpret_cast<uintptr_t>(a.B) % 2u != 0u)
        return GEMM_ERR_INVALID_ARG;
    uint64_t a_end = 0, b_end = 0;
    if (!region_end(a.a_rows(), a.a_cols(), a.lda, 2, &a_end) ||
        !region_end(a.b_rows(), a.b_cols(), a.ldb, 2, &b_end))
        return GEMM_ERR_UNSUPPORTED;
    if (overlaps(a.C, c_end, a.A, a_end) || overlaps(a.C, c_end, a.B, b_end))
        return GEMM_ERR_INVALID_ARG;
    return GEMM_OK;
}

constexpr int64_t kMaxShares = dg::kSkinnyMaxShares;

// Skinny stream-K shares.  `shares` <= 0: dg::skinny_auto_shares; otherwise
// exactly that many shares.  Falls back to one share per tile (no partial
// tiles) when the workspace or counters cannot hold the partials; that
// needs neither, so it is open to any number of tiles (the CTAs walk the
// shares persistently).  Returns false for a forced share count that does
// not fit.
bool choose_shares(const gemm_plan_s* plan, Choice* c, int64_t shares) {
    const int64_t T = int64_t(c->tiles_n) * c->num_kb;
    int64_t G = shares > 0 ? shares : dg::skinny_auto_shares(c->tiles_n, c->num_kb, plan->num_sms);
    G = std::max<int64_t>(1, std::min<int64_t>({G, T, kMaxShares}));
    const int slots = dg::shares_per_tile_bound(T, G, c->num_kb);
    const int64_t need = int64_t(c->tiles_n) * slots * c->ms * 128 * 4;
    const bool aligned = (G % c->tiles_n == 0) && (G / c->tiles_n == 1);   // one share per tile
    if (!aligned &&
        (c->tiles_n > plan->counters_len || need > static_cast<int64_t>(plan->ws_bytes))) {
        if (shares > 0) return false;
        G = c->tiles_n;
    }
    c->shares = static_cast<int>(G);
    c->max_slots = dg::shares_per_tile_bound(T, G, c->num_kb);
    // Most shares touching one tile (the "K split" a tile sees), for reporting.
    int most = 1;
    for (int64_t t = 0; t < c->tiles_n && t < 65536; ++t) {
        const int64_t first = dg::share_of(t * c->num_kb, T, G);
        const int64_t last = dg::share_of((t + 1) * c->num_kb - 1, T, G);
        most = std::max<int>(most, static_cast<int>(last - first + 1));
    }
    c->split = most;
    return true;
}

// Operands whose base or row pitch is not a multiple of 16 bytes cannot be read
// by TMA.  When they fit in the plan's staging buffer they are copied there
// first, rows padded to a multiple of 8 elements, and the TMA kernels read the
// copies; otherwise (or with the generic kernel forced) the generic kernel
// reads them in place.  `out` gets the arguments the GEMM kernel will see.
struct Staging {
    bool a = false, b = false;
    int64_t lda = 0, ldb = 0;
    size_t off_b = 0;
};

bool plan_staging(const gemm_plan_s* plan, const Args& a, Staging* st, Args* out) {
    *out = a;
    *st = Staging{};
    if (plan->force_kernel == GEMM_KERNEL_GENERIC || !plan->staging || plan->stage_bytes == 0 ||
        a.M == 0 ||
        a.N == 0 || a.K == 0)
        return false;
    const bool a_bad = !tma_ok(a.A, a.lda);
    const bool b_bad = !tma_ok(a.B, a.ldb);
    if (!a_bad && !b_bad) return false;
    const int64_t lda2 = (a.a_cols() + 7) / 8 * 8;
    const int64_t ldb2 = (a.b_cols() + 7) / 8 * 8;
    const uint64_t bytes_a = a_bad ? static_cast<uint64_t>(a.a_rows()) * lda2 * 2 : 0;
    const uint64_t off_b = (bytes_a + 255) / 256 * 256;
    const uint64_t bytes_b = b_bad ? static_cast<uint64_t>(a.b_rows()) * ldb2 * 2 : 0;
    if (off_b + bytes_b > plan->stage_bytes) return false;
    st->a = a_bad;
    st->b = b_bad;
    st->lda = lda2;
    st->ldb = ldb2;
    st->off_b = static_cast<size_t>(off_b);
    if (a_bad) {
        out->A = plan->stage;
        out->lda = lda2;
    }
    if (b_bad) {
        out->B = reinterpret_cast<const uint8_t*>(plan->stage) + off_b;
        out->ldb = ldb2;
    }
    return true;
}

// Small M on 2-CTA clusters, strip width when not forced: 128 columns while
// the strips of 128 fit on the SMs in one wave, else 256 (wider strips stream
// B faster per SM: 512-byte row pieces), 192 with M > 32 (whose 256-column
// stages leave room for only four in flight), if those fit in one wave.
// Measured at M = 16, K = 4096: N = 8192 128 columns 13.6 us, 256 14.3;
// N = 14336 256 columns 21.1 us, 192 21.9; at M = 64 192 columns 23.1 us, 256 24.4.
int splitpair_auto_width(const gemm_plan_s* plan, const Args& a) {
    if (2 * cdiv(a.N, 128) <= plan->num_sms) return 128;
    if (a.M > 32 && cdiv(a.N, 192) <= plan->splitpair_clusters) return 192;
    return 256;
}

// The cluster kernel is chosen (returning its strip width) when its first wave
// keeps at least 3/5 of the SMs streaming B and there are at least 8 K blocks
// per half; otherwise (0) the stream-K kernel, which balances any shape but
// pays a global fix-up (measured at M = 16, K = 4096: N = 4096, 64 CTAs of the
// cluster kernel 12.3 us against 11.3 for stream-K; N = 8192, 128 CTAs 13.6
// against 16.1; N = 28672, two waves, 42.6 against 49.1).
int splitpair_auto_bn(const gemm_plan_s* plan, const Args& a) {
    if (plan->splitpair_clusters <= 0 || cdiv(a.K, dg::kBK) < 16) return 0;
    const int bn = splitpair_auto_width(plan, a);
    const int64_t strips = cdiv(a.N, bn);
    const int64_t first_wave = std::min<int64_t>(strips, plan->splitpair_clusters);
    if (5 * 2 * first_wave < 3 * int64_t(plan->num_sms)) return 0;
    return bn;
}

// B read in place by the split-pair kernel (no staging copy): A 16-byte aligned
// and not transposed, B stored K x N (N contiguous) with a base or pitch that is
// not a multiple of 16 bytes, and a problem the split-pair kernel takes with
// 128 x 128 tiles -- by the automatic rule of `choose` (M > 64, the tiles fit one
// wave of clusters, at least kSplitPairMinKb K blocks) or forced -- when B does
// not fit the staging buffer (or staging is off).  A staged B is faster where it
// fits: on the ragged 1023 x 1000 x 1029 fp16 workload (graph-replayed) 12.2 us
// staged against 14.0 us read in place, whose loader warps (copies of each
// row's aligned span, then a shift into the swizzled stage) add about 0.55 us
// per K block over TMA; where B does not fit, the alternative is the generic
// kernel, about six times slower.
bool b_in_place(const gemm_plan_s* plan, const Args& a) {
    if (a.M <= 64 || a.N == 0 || a.K == 0 || a.op_a != GEMM_OP_N || a.op_b != GEMM_OP_N)
        return false;
    if (!tma_ok(a.A, a.lda) || tma_ok(a.B, a.ldb) || plan->splitpair_clusters <= 0) return false;
    const uint64_t staged_b = static_cast<uint64_t>(a.K) * static_cast<uint64_t>((a.N + 7) / 8 * 8) * 2;
    if (plan->staging && plan->stage_bytes > 0 && staged_b <= plan->stage_bytes) return false;
    if (plan->force_kernel == GEMM_KERNEL_SPLIT_PAIR)
        return cdiv(a.K, dg::kBK) >= 2 && (plan->force_bn == 0 || plan->force_bn == 128);
    if (plan->force_kernel != 0) return false;
    return cdiv(a.M, dg::kBM) * cdiv(a.N, 128) <= plan->splitpair_clusters &&
           cdiv(a.K, dg::kBK) >= kSplitPairMinKb;
}

// b_gen: B is read in place by the split-pair kernel (b_in_place holds).
gemm_status_t choose(const gemm_plan_s* plan, const Args& a, Choice* c, bool b_gen = false) {
    *c = Choice{};
    if (a.M == 0 || a.N == 0) {
        c->kernel = GEMM_KERNEL_NONE;
        return GEMM_OK;
    }
    if (a.K == 0) {
        c->kernel = GEMM_KERNEL_ZERO_FILL;
        return GEMM_OK;
    }
    const bool tma = tma_ok(a.A, a.lda) && (b_gen || tma_ok(a.B, a.ldb));
    int kernel = plan->force_kernel;
    int auto_bn = 0;
    if (kernel == 0) {
        if (tma && a.M <= 64 && a.op_a == GEMM_OP_N) {
            // A cluster per strip of columns (K split in two) when the strips
            // fill nearly every SM in one wave; otherwise stream-K over tiles.
            const int bn = splitpair_auto_bn(plan, a);
            kernel = bn ? GEMM_KERNEL_SPLIT_PAIR : GEMM_KERNEL_SKINNY;
            auto_bn = bn;
        } else if (tma && a.op_a == GEMM_OP_N && plan->splitpair_clusters > 0 &&
                   cdiv(a.M, dg::kBM) * cdiv(a.N, 128) <= plan->splitpair_clusters &&
                   cdiv(a.K, dg::kBK) >= kSplitPairMinKb) {
            // Few 128 x 128 tiles (one wave of clusters): each tile's K loop split
            // over a 2-CTA cluster puts twice as many SMs on the problem as
            // one-CTA tiles do.  Measured (graph-replayed, M x K x N):
            // 1024 x 8192 x 1024 39.7 -> 23.1 us, 256 x 4096 x 2048 21.6 -> 14.3,
            // 1023 x 1000 x 1029 18.9 -> 15.1; at 16 K blocks and fewer it is
            // about even (1024^3 8.1 vs 8.3 us), below 12 slower (65 x 512 x 512).
            kernel = GEMM_KERNEL_SPLIT_PAIR;
            auto_bn = 128;
        } else if (tma) {
            // The cheapest of pair tiles 256 x 256, one-CTA tiles 128 x 256 and
            // 128 x 128 under est_seconds (waves x time of one tile).
            const double k = static_cast<double>(a.K);
            const int64_t pair_slots = plan->pair_clusters[1];
            const double t_pair =
                pair_slots > 0 ? est_seconds(cdiv(a.M, 256) * cdiv(a.N, 256), pair_slots,
                                             2.0 * 256 * 256 * k, 2.0 * kRatePairPerSm)
                               : 1e30;
            const double t_tma256 = est_seconds(cdiv(a.M, 128) * cdiv(a.N, 256), plan->num_sms,
                                                2.0 * 128 * 256 * k, kRateTma256PerSm);
            const double t_tma128 = est_seconds(cdiv(a.M, 128) * cdiv(a.N, 128), plan->num_sms,
                                                2.0 * 128 * 128 * k, kRateTma128PerSm);
            if (t_pair <= t_tma256 && t_pair <= t_tma128) {
                kernel = GEMM_KERNEL_PAIR;
                auto_bn = 256;
            } else {
                kernel = GEMM_KERNEL_TMA;
                auto_bn = t_tma256 < t_tma128 ? 256 : 128;
                // Few 128 x 128 tiles (a partial wave) whose 128 x 64 halves still fit
                // one wave: twice the CTAs, each with half the loads and stores.
                // Measured (graph-replayed): 256^3 4.71 -> 3.99 us, 512 x 256 x 512
                // 4.71 -> 4.09 us.
                if (auto_bn == 128 && cdiv(a.M, dg::kBM) * cdiv(a.N, 128) < plan->num_sms &&
                    cdiv(a.M, dg::kBM) * cdiv(a.N, 64) <= plan->num_sms)
                    auto_bn = 64;
            }
        } else {
            kernel = GEMM_KERNEL_GENERIC;
        }
    }
    if ((kernel == GEMM_KERNEL_TMA || kernel == GEMM_KERNEL_SKINNY ||
         kernel == GEMM_KERNEL_PAIR || kernel == GEMM_KERNEL_SPLIT_PAIR) && !tma)
        return GEMM_ERR_UNSUPPORTED;
    if (kernel == GEMM_KERNEL_SKINNY && (a.M > 64 || a.op_a != GEMM_OP_N))
        return GEMM_ERR_UNSUPPORTED;
    if (kernel == GEMM_KERNEL_SPLIT_PAIR &&
        (a.op_a != GEMM_OP_N || (a.M > 64 && plan->force_bn != 0 && plan->force_bn != 128)))
        return GEMM_ERR_UNSUPPORTED;
    if (kernel == GEMM_KERNEL_SPLIT_PAIR && (cdiv(a.K, dg::kBK) < 2 || plan->splitpair_clusters <= 0))
        return GEMM_ERR_UNSUPPORTED;
    // 192-column tiles exist only in the small-M cluster kernel, 64-column ones only in
    // the one-CTA kernel.
    if (plan->force_bn == 192 && kernel != GEMM_KERNEL_SPLIT_PAIR) return GEMM_ERR_UNSUPPORTED;
    if (plan->force_bn == 64 && kernel != GEMM_KERNEL_TMA) return GEMM_ERR_UNSUPPORTED;
    if (kernel == GEMM_KERNEL_PAIR && plan->pair_clusters[0] <= 0) return GEMM_ERR_UNSUPPORTED;
    if (kernel != GEMM_KERNEL_TMA && kernel != GEMM_KERNEL_SKINNY &&
        kernel != GEMM_KERNEL_GENERIC && kernel != GEMM_KERNEL_PAIR &&
        kernel != GEMM_KERNEL_SPLIT_PAIR)
        return GEMM_ERR_UNSUPPORTED;
    if (b_gen && kernel != GEMM_KERNEL_SPLIT_PAIR) return GEMM_ERR_UNSUPPORTED;
    c->kernel = kernel;
    c->num_kb = static_cast<int>(cdiv(a.K, dg::kBK));
    if (kernel == GEMM_KERNEL_SKINNY) {
        c->ms = a.M <= 16 ? 16 : (a.M <= 32 ? 32 : 64);
        c->tiles_m = 1;
        c->tiles_n = static_cast<int>(cdiv(a.N, 128));
        // A forced split is the total number of stream-K shares.
        if (!choose_shares(plan, c, plan->force_split)) return GEMM_ERR_UNSUPPORTED;
        c->units = c->shares;
        c->stages = dg::skinny_stages(c->ms);
    } else if (kernel == GEMM_KERNEL_SPLIT_PAIR) {
        c->ms = a.M <= 16 ? 16 : (a.M <= 32 ? 32 : (a.M <= 64 ? 64 : 128));
        if (c->ms == 128)
            c->bn = 128;
        else
            c->bn = plan->force_bn ? plan->force_bn
                                   : (auto_bn ? auto_bn : splitpair_auto_width(plan, a));
        const int64_t tm = c->ms == 128 ? cdiv(a.M, dg::kBM) : 1;
        const int64_t tiles = tm * cdiv(a.N, c->bn);
        if (tiles > INT32_MAX / 2) return GEMM_ERR_UNSUPPORTED;
        c->tiles_m = static_cast<int>(tm);
        c->tiles_n = static_cast<int>(cdiv(a.N, c->bn));
        c->units = static_cast<int>(tiles);
        c->split = 2;
        c->grid = 2 * c->units;
        c->stages = dg::splitpair_stages(c->ms, c->bn, b_gen);
        return GEMM_OK;
    } else if (kernel == GEMM_KERNEL_PAIR) {
        const int64_t tm = cdiv(a.M, 2 * dg::kBM);
        const int64_t t256 = tm * cdiv(a.N, 256);
        c->bn = plan->force_bn ? plan->force_bn
                               : (auto_bn ? auto_bn
                                          : ((t256 >= int64_t(plan->pair_clusters[1])) ? 256 : 128));
        c->stages = dg::pair_stages(c->bn);
        c->tiles_m = static_cast<int>(tm);
        c->tiles_n = static_cast<int>(cdiv(a.N, c->bn));
        const int64_t units = int64_t(c->tiles_m) * c->tiles_n;
        if (units > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
        c->units = static_cast<int>(units);
        const int clusters = plan->pair_clusters[c->bn == 256 ? 1 : 0];
        c->sk_tiles = 0;
        c->shares = 0;
        // Whole-problem stream-K: every tile's K loop is split over all the
        // clusters (split_k = 2 forces it), so that a problem with fewer pair
        // tiles than clusters still occupies every SM.
        if (plan->force_split == 2) {
            const int64_t T = units * c->num_kb;
            const int64_t need = int64_t(clusters) * 2 * 2 * c->bn * 128 * 4;
            if (T / clusters >= kPairMinShareKb && need <= static_cast<int64_t>(plan->ws_bytes) &&
                units * 2 <= plan->counters_len) {
                c->grid = 2 * clusters;
                c->sk_tiles = c->units;
                c->shares = clusters;
                int most = 1;
                for (int64_t t = 0; t < units; ++t)
                    most = std::max<int>(most, static_cast<int>(
                                                   dg::share_of((t + 1) * c->num_kb - 1, T, clusters) -
                                                   dg::share_of(t * c->num_kb, T, clusters) + 1));
                c->split = most;
                return GEMM_OK;
            }
        }
        const int ncl = c->units < clusters ? c->units : clusters;
        c->grid = 2 * ncl;
        // Stream-K phase: when the last wave of tiles leaves at least half of the
        // clusters idle (or at least 30% of them, behind five or more full waves),
        // that partial wave is cut into one equal K share per cluster, taken first;
        // the rest are whole tiles.  A fuller last wave costs less idle time than
        // the split's slower streaming and fix-ups, and with few full waves the
        // fix-ups have too little whole-tile work to hide behind (all measured:
        // 6144^3, 58% full behind 7 waves, gains 1.5%; 3584^3, 58% behind 2,
        // loses 11%; 5376^3, 80% behind 5, loses 0.7%).  If the shares would be
        // shorter than kPairMinShareKb K blocks, one full wave joins the split
        // tiles.  Also skipped when the partial tiles would not fit the workspace,
        // with fewer than kPairMinSkKb K blocks per tile (the fix-ups then cost
        // more than the idle time they save; measured at K = 1024), or when
        // forced off (split_k = 1).
        // split_k = 3 forces the phase for any partial last wave (tuning).
        const bool sk_forced = plan->force_split == 3;
        const int64_t rem = units % ncl, waves = units / ncl;
        const bool sk_pays = (2 * rem <= ncl && waves >= 2) || (10 * rem <= 7 * ncl && waves >= 5);
        if (plan->force_split != 1 && rem != 0 && (sk_forced || sk_pays) &&
            c->num_kb >= kPairMinSkKb) {
            int64_t sk = units % ncl;
            if (sk * c->num_kb / ncl < kPairMinShareKb) sk += ncl;
            const int64_t share_kb = sk * c->num_kb / ncl;
            const int64_t need = int64_t(ncl) * 2 * 2 * c->bn * 128 * 4;   // [share][slot][rank]
            if (share_kb >= kPairMinShareKb && need <= static_cast<int64_t>(plan->ws_bytes) &&
                sk * 2 <= plan->counters_len) {
                c->sk_tiles = static_cast<int>(sk);
                c->shares = ncl;
                const int64_t T = sk * c->num_kb;
                int most = 1;
                for (int64_t t = 0; t < sk; ++t)
                    most = std::max<int>(most, static_cast<int>(
                                                   dg::share_of((t + 1) * c->num_kb - 1, T, ncl) -
                                                   dg::share_of(t * c->num_kb, T, ncl) + 1));
                c->split = most;
            }
        }
        return GEMM_OK;
    } else {
        int64_t tm = cdiv(a.M, dg::kBM);
        if (kernel == GEMM_KERNEL_TMA) {
            const int64_t t256 = tm * cdiv(a.N, 256);
            c->bn = plan->force_bn ? plan->force_bn
                                   : (auto_bn ? auto_bn
                                              : ((t256 >= 2 * int64_t(plan->num_sms)) ? 256 : 128));
            c->stages = dg::tma_stages(c->bn);
            // 128 x 64 tiles that fill less than half the SMs: 64 x 64 tiles (M = 64
            // MMAs) if they still fit one wave -- twice the CTAs, each with half
            // the A loads and half the stores.
            if (c->bn == 64 && 2 * tm * cdiv(a.N, 64) <= plan->num_sms &&
                cdiv(a.M, 64) * cdiv(a.N, 64) <= plan->num_sms) {
                c->bm = 64;
                tm = cdiv(a.M, 64);
            }
        } else {
            c->bn = 128;
            c->stages = dg::generic_stages();
        }
        c->tiles_m = static_cast<int>(tm);
        c->tiles_n = static_cast<int>(cdiv(a.N, c->bn));
        const int64_t units = int64_t(c->tiles_m) * c->tiles_n;
        if (units > INT32_MAX) return GEMM_ERR_UNSUPPORTED;
        c->units = static_cast<int>(units);
    }
    c->grid = c->units < plan->num_sms ? c->units : plan->num_sms;
    return GEMM_OK;
}

struct DeviceGuard {
    int prev = -1;
    bool ok = false;
    explicit DeviceGuard(int dev) {
        if (cudaGetDevice(&prev) != cudaSuccess) {
            (void)cudaGetLastError();
            prev = -1;
        }
        ok = (prev == dev) || cudaSetDevice(dev) == cudaSuccess;
        if (!ok) (void)cudaGetLastError();
    }
    ~DeviceGuard() {
        if (prev >= 0) (void)cudaSetDevice(prev);
    }
};

bool env_flag(const char* name) {
    const char* v = std::getenv(name);
    return v != nullptr && v[0] != '\0' && v[0] != '0';
}

}  // namespace

namespace dg {

__global__ void wait_selftest_kernel(int* out, uint64_t timeout_ns) {
    __shared__ uint64_t bar;
    __shared__ int abort_flag;
    if (threadIdx.x == 0) {
        mbar_init(smem_u32(&bar), 1u);
        abort_flag = 0;
        fence_mbar_init();
    }
    __syncthreads();
    if (threadIdx.x == 0) {
        // Nothing ever arrives on `bar`: the bounded wait must give up.
        const bool ok = mbar_wait(smem_u32(&bar), 0u, &abort_flag, timeout_ns);
        *out = ok ? 1 : 2;
    }
}

cudaError_t launch_wait_selftest(int* out, uint64_t timeout_ns, cudaStream_t stream) {
    wait_selftest_kernel<<<1, 32, 0, stream>>>(out, timeout_ns);
    return cudaGetLastError();
}

// No work: the dependency wait and the early release of the next kernel, as
// every GEMM kernel does them.
__global__ void __launch_bounds__(192) noop_kernel() {
    griddep_wait();
    griddep_launch_dependents();
}

cudaError_t launch_noop(int grid, int cluster, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    attr[1].id = cudaLaunchAttributeClusterDimension;
    attr[1].val.clusterDim.x = static_cast<unsigned>(cluster);
    attr[1].val.clusterDim.y = 1;
    attr[1].val.clusterDim.z = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = cluster > 1 ? 2 : 1;
    return cudaLaunchKernelEx(&cfg, noop_kernel);
}

}  // namespace dg

extern "C" {

const char* gemm_status_string(gemm_status_t s) {
    switch (s) {
        case GEMM_OK: return "GEMM_OK";
        case GEMM_ERR_INVALID_ARG: return "GEMM_ERR_INVALID_ARG";
        case GEMM_ERR_UNSUPPORTED: return "GEMM_ERR_UNSUPPORTED";
        case GEMM_ERR_CUDA: return "GEMM_ERR_CUDA";
        case GEMM_ERR_OOM: return "GEMM_ERR_OOM";
        case GEMM_ERR_TIMEOUT: return "GEMM_ERR_TIMEOUT";
        case GEMM_ERR_BOUNDS: return "GEMM_ERR_BOUNDS";
    }
    return "GEMM_ERR_UNKNOWN";
}

gemm_status_t gemm_plan_create(gemm_plan_t* out, int device) {
    if (out == nullptr) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    int count = 0;
    if (cudaGetDeviceCount(&count) != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (device < 0 || device >= count) return GEMM_ERR_INVALID_ARG;
    DeviceGuard guard(device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    int major = 0, minor = 0, sms = 0;
    if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, device) != cudaSuccess ||
        cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, device) != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (major != 10 || minor != 3) return GEMM_ERR_UNSUPPORTED;
    if (encode_fn() == nullptr) return GEMM_ERR_CUDA;
    if (dg::tma_prepare() != cudaSuccess || dg::generic_prepare() != cudaSuccess ||
        dg::skinny_prepare() != cudaSuccess || dg::pair_prepare() != cudaSuccess ||
        dg::splitpair_prepare() != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    gemm_plan_s* p = new (std::nothrow) gemm_plan_s();
    if (p == nullptr) return GEMM_ERR_OOM;
    p->device = device;
    p->num_sms = sms;
    // Pair tiles need both SMs of a cluster resident at once; size their
    // persistent grids by what the device can co-schedule.
    p->pair_clusters[0] = dg::pair_max_clusters(128);
    p->pair_clusters[1] = dg::pair_max_clusters(256);
    p->splitpair_clusters = dg::splitpair_max_clusters();
    p->debug_sync = env_flag("GEMM_DEBUG_SYNC");
    if (const char* t = std::getenv("GEMM_WAIT_TIMEOUT_MS")) {
        const long long ms = std::atoll(t);
        if (ms > 0) p->timeout_ns = static_cast<uint64_t>(ms) * 1000000ull;
    }
    // Fault injection for tests: GEMM_TEST_FAIL_ALLOC=k makes the k-th of the four
    // device allocations below fail as if the device were out of memory.
    int fail_at = 0;
    if (const char* f = std::getenv("GEMM_TEST_FAIL_ALLOC")) fail_at = std::atoi(f);
    int n_alloc = 0;
    auto alloc = [&](void** ptr, size_t bytes) {
        if (++n_alloc == fail_at) return false;
        return cudaMalloc(ptr, bytes) == cudaSuccess;
    };
    if (!alloc(reinterpret_cast<void**>(&p->ws), kWorkspaceBytes) ||
        !alloc(reinterpret_cast<void**>(&p->counters), sizeof(int) * kMaxCounters) ||
        !alloc(reinterpret_cast<void**>(&p->status), sizeof(int)) ||
        !alloc(reinterpret_cast<void**>(&p->stage), kStageBytes)) {
        (void)cudaGetLastError();
        cudaFree(p->ws);
        cudaFree(p->counters);
        cudaFree(p->status);
        cudaFree(p->stage);
        delete p;
        return GEMM_ERR_OOM;
    }
    p->ws_bytes = kWorkspaceBytes;
    p->stage_bytes = kStageBytes;
    p->counters_len = kMaxCounters;
    if (cudaMemset(p->counters, 0, sizeof(int) * kMaxCounters) != cudaSuccess ||
        cudaMemset(p->status, 0, sizeof(int)) != cudaSuccess) {
        (void)cudaGetLastError();
        cudaFree(p->ws);
        cudaFree(p->counters);
        cudaFree(p->status);
        cudaFree(p->stage);
        delete p;
        return GEMM_ERR_CUDA;
    }
    *out = p;
    return GEMM_OK;
}

gemm_status_t gemm_plan_create_model(gemm_plan_t* out, int32_t num_sms, int32_t pair_clusters_128,
                                     int32_t pair_clusters_256, int32_t splitpair_clusters) {
    if (out == nullptr) return GEMM_ERR_INVALID_ARG;
    *out = nullptr;
    if (num_sms < 1 || num_sms > 4096) return GEMM_ERR_INVALID_ARG;
    for (int c : {pair_clusters_128, pair_clusters_256, splitpair_clusters})
        if (c < 0 || 2 * c > num_sms) return GEMM_ERR_INVALID_ARG;
    gemm_plan_s* p = new (std::nothrow) gemm_plan_s();
    if (p == nullptr) return GEMM_ERR_OOM;
    p->model = true;
    p->device = -1;
    p->num_sms = num_sms;
    p->pair_clusters[0] = pair_clusters_128;
    p->pair_clusters[1] = pair_clusters_256;
    p->splitpair_clusters = splitpair_clusters;
    p->ws_bytes = kWorkspaceBytes;       // what a device plan holds, so the choices match
    p->stage_bytes = kStageBytes;
    p->counters_len = kMaxCounters;
    *out = p;
    return GEMM_OK;
}

gemm_status_t gemm_plan_destroy(gemm_plan_t plan) {
    if (plan == nullptr) return GEMM_OK;
    if (plan->model) {
        delete plan;
        return GEMM_OK;
    }
    DeviceGuard guard(plan->device);
    cudaFree(plan->ws);
    cudaFree(plan->counters);
    cudaFree(plan->status);
    cudaFree(plan->stage);
    delete plan;
    return GEMM_OK;
}

gemm_status_t gemm_plan_set_group(gemm_plan_t plan, int32_t group) {
    if (plan == nullptr || group < 0 || group > 64) return GEMM_ERR_INVALID_ARG;
    plan->group = group;
    return GEMM_OK;
}

gemm_status_t gemm_plan_force(gemm_plan_t plan, int32_t kernel, int32_t split_k,
                              int32_t block_n) {
    if (plan == nullptr || split_k < 0) return GEMM_ERR_INVALID_ARG;
    if (block_n != 0 && block_n != 64 && block_n != 128 && block_n != 192 && block_n != 256)
        return GEMM_ERR_INVALID_ARG;
    if (kernel != 0 && kernel != GEMM_KERNEL_TMA && kernel != GEMM_KERNEL_GENERIC &&
        kernel != GEMM_KERNEL_SKINNY && kernel != GEMM_KERNEL_PAIR &&
        kernel != GEMM_KERNEL_SPLIT_PAIR)
        return GEMM_ERR_INVALID_ARG;
    plan->force_kernel = kernel;
    plan->force_split = split_k;
    plan->force_bn = block_n;
    return GEMM_OK;
}

int32_t gemm_build_checked(void) { return DG_CHECKED ? 1 : 0; }

gemm_status_t gemm_plan_device_status(gemm_plan_t plan, int32_t* word) {
    if (plan == nullptr || word == nullptr) return GEMM_ERR_INVALID_ARG;
    *word = plan->last_device_status;
    return GEMM_OK;
}

gemm_status_t gemm_plan_set_debug(gemm_plan_t plan, int32_t sync, uint64_t timeout_ns) {
    if (plan == nullptr || (sync != 0 && sync != 1)) return GEMM_ERR_INVALID_ARG;
    plan->debug_sync = sync != 0;
    plan->timeout_ns = timeout_ns != 0 ? timeout_ns : kDefaultTimeoutNs;
    return GEMM_OK;
}

gemm_status_t gemm_plan_set_staging(gemm_plan_t plan, int32_t enabled) {
    if (plan == nullptr || (enabled != 0 && enabled != 1)) return GEMM_ERR_INVALID_ARG;
    plan->staging = enabled != 0;
    return GEMM_OK;
}

gemm_status_t gemm_tile_coord(int64_t t, int64_t tiles_m, int64_t tiles_n, int32_t group,
                              int64_t* tile_m, int64_t* tile_n) {
    if (tile_m == nullptr || tile_n == nullptr || tiles_m <= 0 || tiles_n <= 0 || group < 0 ||
        tiles_m > kMaxDim || tiles_n > kMaxDim || t < 0 || t >= tiles_m * tiles_n)
        return GEMM_ERR_INVALID_ARG;
    dg::tile_coord(t, tiles_m, tiles_n, group, *tile_m, *tile_n);
    return GEMM_OK;
}

}  // extern "C"

namespace {

gemm_status_t query_impl(gemm_plan_t plan, const Args& a_in, gemm_config_t* out) {
    if (plan == nullptr || out == nullptr) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = check_args(a_in);
    if (st != GEMM_OK) return st;
    Args a = a_in;
    Staging sg;
    const bool b_gen = b_in_place(plan, a_in);
    if (!b_gen) plan_staging(plan, a_in, &sg, &a);
    Choice c;
    st = choose(plan, a, &c, b_gen);
    if (st != GEMM_OK) return st;
    gemm_config_t cfg{};
    cfg.kernel = c.kernel;
    cfg.block_m = (c.kernel == GEMM_KERNEL_SKINNY || c.kernel == GEMM_KERNEL_SPLIT_PAIR)
                      ? c.ms
                      : (c.kernel == GEMM_KERNEL_PAIR ? 2 * dg::kBM
                                                        : (c.kernel == GEMM_KERNEL_TMA ? c.bm : dg::kBM));
    cfg.block_n = (c.kernel == GEMM_KERNEL_SKINNY) ? 128 : c.bn;
    cfg.block_k = (c.kernel == GEMM_KERNEL_NONE || c.kernel == GEMM_KERNEL_ZERO_FILL) ? 0 : dg::kBK;
    cfg.stages = c.stages;
    cfg.split_k = c.split;
    cfg.grid = c.grid;
    cfg.cluster = (c.kernel == GEMM_KERNEL_NONE || c.kernel == GEMM_KERNEL_ZERO_FILL)
                      ? 0
                      : ((c.kernel == GEMM_KERNEL_PAIR || c.kernel == GEMM_KERNEL_SPLIT_PAIR) ? 2
                                                                                          : 1);
    cfg.group = (c.kernel == GEMM_KERNEL_TMA || c.kernel == GEMM_KERNEL_GENERIC ||
                 c.kernel == GEMM_KERNEL_PAIR)
                    ? plan->group
                    : 0;
    cfg.tiles = c.units;
    cfg.shares = c.shares;
    cfg.staged = (sg.a ? 1 : 0) | (sg.b ? 2 : 0) | (b_gen ? 4 : 0);
    *out = cfg;
    return GEMM_OK;
}

gemm_status_t run_impl(gemm_plan_t plan, const Args& a_in, cudaStream_t stream) {
    if (plan == nullptr || plan->model) return GEMM_ERR_INVALID_ARG;
    gemm_status_t st = check_args(a_in);
    if (st != GEMM_OK) return st;
    Args a = a_in;
    Staging sg;
    const bool b_gen = b_in_place(plan, a_in);
    const bool staged = b_gen ? false : plan_staging(plan, a_in, &sg, &a);
    Choice c;
    st = choose(plan, a, &c, b_gen);
    if (st != GEMM_OK) return st;
    if (c.kernel == GEMM_KERNEL_NONE) return GEMM_OK;

    DeviceGuard guard(plan->device);
    if (!guard.ok) return GEMM_ERR_CUDA;
    cudaError_t err = cudaSuccess;
    if (staged) {
        if (sg.a)
            err = dg::launch_stage_rows(static_cast<const uint16_t*>(a_in.A), a_in.lda,
                                        const_cast<uint16_t*>(static_cast<const uint16_t*>(a.A)),
                                        a.lda, a_in.a_rows(), a_in.a_cols(), plan->status,
                                        plan->num_sms,
                                        stream);
        if (err == cudaSuccess && sg.b)
            err = dg::launch_stage_rows(static_cast<const uint16_t*>(a_in.B), a_in.ldb,
                                        const_cast<uint16_t*>(static_cast<const uint16_t*>(a.B)),
                                        a.ldb, a_in.b_rows(), a_in.b_cols(), plan->status,
                                        plan->num_sms,
                                        stream);
        if (err != cudaSuccess) {
            (void)cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
    }
    const int64_t esize = a.c_esize();

    if (c.kernel == GEMM_KERNEL_ZERO_FILL) {
        err = cudaMemset2DAsync(const_cast<void*>(a.C), static_cast<size_t>(a.ldc * esize), 0,
                                static_cast<size_t>(a.N * esize), static_cast<size_t>(a.M),
                                stream);
    } else {
        const bool a_mn = a.op_a == GEMM_OP_T;     // A stored K x M: M contiguous
        const bool b_mn = a.op_b == GEMM_OP_N;     // B stored K x N: N contiguous
        dg::Params p{};
        p.A = static_cast<const uint16_t*>(a.A);
        p.B = static_cast<const uint16_t*>(a.B);
        p.C = const_cast<void*>(a.C);
        p.c_type = a.c_type;
        p.lda = a.lda;
        p.ldb = a.ldb;
        p.ldc = a.ldc;
        p.M = static_cast<int32_t>(a.M);
        p.N = static_cast<int32_t>(a.N);
        p.K = static_cast<int32_t>(a.K);
        p.tiles_m = c.tiles_m;
        p.tiles_n = c.tiles_n;
        p.num_kb = c.num_kb;
        p.group = plan->group;
        p.shares = c.shares;
        p.max_slots = c.max_slots;
        p.sk_tiles = c.sk_tiles;
        p.a_vec = tma_ok(a.A, a.lda) ? 1 : 0;
        p.b_vec = tma_ok(a.B, a.ldb) ? 1 : 0;
        p.c_vec = ((reinterpret_cast<uintptr_t>(a.C) % 16u) == 0u && (a.ldc * esize) % 16 == 0)
                      ? 1
                      : 0;
        p.ws = plan->ws;
        p.counters = plan->counters;
        p.ws_len = static_cast<int64_t>(plan->ws_bytes / sizeof(float));
        p.counters_len = plan->counters_len;
        p.status = plan->status;
        p.timeout_ns = plan->timeout_ns;
        const bool bf16 = a.dtype == GEMM_BF16;
        const Elem in = elem_of(a.dtype);
        // TMA descriptors: a K-major operand is read as boxes {64 k, rows}; an
        // MN-major one as boxes {64 mn, 64 k}.
        auto map_a = [&](CUtensorMap* m, uint32_t rows) {
            return a_mn ? cached_encode_2d(plan, m, in, a.A, a.M, a.K, a.lda, dg::kSubN, dg::kBK)
                        : cached_encode_2d(plan, m, in, a.A, a.K, a.M, a.lda, dg::kBK, rows);
        };
        auto map_b = [&](CUtensorMap* m, uint32_t rows) {
            return b_mn ? cached_encode_2d(plan, m, in, a.B, a.N, a.K, a.ldb, dg::kSubN, dg::kBK)
                        : cached_encode_2d(plan, m, in, a.B, a.K, a.N, a.ldb, dg::kBK, rows);
        };
        // C written by TMA stores of {128 bytes of columns, 32 rows (16 for 64-row
        // tiles)} boxes when its
        // base, pitch and row length are 16-byte multiples; otherwise by ordinary
        // stores.  (With a row length that is not, the right edge of C was seen
        // to be written in whole 16-byte pieces, past column N: the guard-band
        // tests catch that.)
        CUtensorMap mc;
        memset(&mc, 0, sizeof(mc));
        auto map_c = [&](uint32_t rows = 32u) {
            p.c_tma = 0;
            if (!p.c_vec || (a.N * esize) % 16 != 0) return;
            const uint32_t cols = a.c_type == GEMM_OUT_F32 ? 32u : 64u;
            if (cached_encode_2d(plan, &mc, elem_of_out(a.c_type), a.C, a.N, a.M, a.ldc, cols, rows))
                p.c_tma = 1;
        };
        if (c.kernel == GEMM_KERNEL_TMA) {
            CUtensorMap ma, mb;
            if (!map_a(&ma, static_cast<uint32_t>(c.bm)) || !map_b(&mb, static_cast<uint32_t>(c.bn)))
                return GEMM_ERR_CUDA;
            map_c(static_cast<uint32_t>(c.bm / 4));     // each epilogue warp's rows
            err = dg::launch_tma(c.bm, c.bn, a_mn, b_mn, ma, mb, mc, p,
                                 dg::idesc_f16(bf16, a_mn, b_mn, c.bm, c.bn), c.grid, stream);
        } else if (c.kernel == GEMM_KERNEL_PAIR) {
            // Each CTA of a pair loads 128 rows of A and its half (bn / 2) of the B tile.
            CUtensorMap ma, mb;
            if (!map_a(&ma, dg::kBM) || !map_b(&mb, static_cast<uint32_t>(c.bn / 2)))
                return GEMM_ERR_CUDA;
            map_c();
            err = dg::launch_pair(c.bn, a_mn, b_mn, ma, mb, mc, p,
                                  dg::idesc_f16(bf16, a_mn, b_mn, 2 * dg::kBM, c.bn), c.grid,
                                  stream);
        } else if (c.kernel == GEMM_KERNEL_SPLIT_PAIR) {
            // A tile (M <= 64 rows, K-major) as the MMA's 128-row A operand, the
            // B tile (bn columns) as its B operand.  A B read in place (b_gen) has
            // no tensor map.
            CUtensorMap ma, mb;
            memset(&mb, 0, sizeof(mb));
            if (!map_a(&ma, static_cast<uint32_t>(c.ms)) ||
                (!b_gen && !map_b(&mb, static_cast<uint32_t>(c.bn))))
                return GEMM_ERR_CUDA;
            // With one row of tiles every CTA streams its own B strip once from
            // DRAM: its first K blocks are prefetched into L2 before the wait on
            // the previous grid (not after a staging copy, which is still writing
            // them).  With several tile rows B is shared through L2 and the early
            // reads only compete (measured slower at 1024 x 1024 x 8192).
            p.prefetch_kb = (!staged && c.tiles_m == 1) ? kL2PrefetchKb : 0;
            map_c();
            err = dg::launch_splitpair(c.ms, c.bn, b_mn, b_gen, ma, mb, mc, p,
                                       dg::idesc_f16(bf16, false, b_mn, dg::kBM, c.bn), c.grid,
                                       stream);
        } else if (c.kernel == GEMM_KERNEL_GENERIC) {
            err = dg::launch_generic(a_mn, b_mn, p,
                                     dg::idesc_f16(bf16, a_mn, b_mn, dg::kBM, 128), c.grid,
                                     stream);
        } else {
            // Swap-AB: the B^T tile (128 N rows) is the MMA's A operand, the A tile
            // (K-major, M <= 64 rows) its B operand.
            CUtensorMap mb, ma;
            if (!map_b(&mb, 128) || !map_a(&ma, static_cast<uint32_t>(c.ms)))
                return GEMM_ERR_CUDA;
            p.prefetch_kb = staged ? 0 : kL2PrefetchKbSkinny;    // one tile row, as above
            err = dg::launch_skinny(c.ms, b_mn, mb, ma, p,
                                    dg::idesc_f16(bf16, b_mn, false, 128, c.ms), c.grid, stream);
        }
    }
    if (err != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (plan->debug_sync) {
        if (cudaStreamSynchronize(stream) != cudaSuccess) {
            (void)cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        int dev_status = 0;
        if (cudaMemcpy(&dev_status, plan->status, sizeof(int), cudaMemcpyDeviceToHost) !=
            cudaSuccess)
            return GEMM_ERR_CUDA;
        plan->last_device_status = dev_status;
        if (dev_status != 0) {
            (void)cudaMemset(plan->status, 0, sizeof(int));
            (void)cudaMemset(plan->counters, 0, sizeof(int) * plan->counters_len);
            return (dev_status & dg::kDevBounds) ? GEMM_ERR_BOUNDS : GEMM_ERR_TIMEOUT;
        }
    }
    return GEMM_OK;
}

}  // namespace

extern "C" {

gemm_status_t gemm_query(gemm_plan_t plan, const void* A, int64_t lda, const void* B, int64_t ldb,
                         const float* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                         gemm_dtype_t dtype, gemm_config_t* out) {
    const Args a{A, lda, B, ldb, C, ldc, M, N, K, dtype};
    return query_impl(plan, a, out);
}

gemm_status_t gemm_query_ex(gemm_plan_t plan, gemm_op_t op_a, gemm_op_t op_b, const void* A,
                            int64_t lda, const void* B, int64_t ldb, const void* C, int64_t ldc,
                            gemm_out_t c_type, int64_t M, int64_t N, int64_t K,
                            gemm_dtype_t dtype, gemm_config_t* out) {
    Args a{A, lda, B, ldb, C, ldc, M, N, K, dtype};
    a.op_a = op_a;
    a.op_b = op_b;
    a.c_type = c_type;
    return query_impl(plan, a, out);
}

gemm_status_t gemm_run(gemm_plan_t plan, const void* A, int64_t lda, const void* B, int64_t ldb,
                       float* C, int64_t ldc, int64_t M, int64_t N, int64_t K,
                       gemm_dtype_t dtype, struct CUstream_st* stream_handle) {
    const Args a{A, lda, B, ldb, C, ldc, M, N, K, dtype};
    return run_impl(plan, a, reinterpret_cast<cudaStream_t>(stream_handle));
}

gemm_status_t gemm_run_ex(gemm_plan_t plan, gemm_op_t op_a, gemm_op_t op_b, const void* A,
                          int64_t lda, const void* B, int64_t ldb, void* C, int64_t ldc,
                          gemm_out_t c_type, int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                          struct CUstream_st* stream_handle) {
    Args a{A, lda, B, ldb, C, ldc, M, N, K, dtype};
    a.op_a = op_a;
    a.op_b = op_b;
    a.c_type = c_type;
    return run_impl(plan, a, reinterpret_cast<cudaStream_t>(stream_handle));
}

gemm_status_t gemm_partition(int64_t M, int64_t N, int64_t K, int32_t world, int32_t rank,
                             int32_t axis, gemm_slice_t* out) {
    if (out == nullptr || M < 0 || N < 0 || K < 0 || world < 1 || rank < 0 || rank >= world)
        return GEMM_ERR_INVALID_ARG;
    if (axis != GEMM_SPLIT_AUTO && axis != GEMM_SPLIT_M && axis != GEMM_SPLIT_N)
        return GEMM_ERR_INVALID_ARG;
    if (axis == GEMM_SPLIT_AUTO) axis = M <= 64 ? GEMM_SPLIT_N : GEMM_SPLIT_M;
    constexpr int64_t kUnit = 128;
    const int64_t extent = axis == GEMM_SPLIT_M ? M : N;
    const int64_t units = cdiv(extent, kUnit);
    const int64_t u0 = static_cast<int64_t>(rank) * units / world;
    const int64_t u1 = static_cast<int64_t>(rank + 1) * units / world;
    const int64_t lo = std::min(extent, u0 * kUnit), hi = std::min(extent, u1 * kUnit);
    gemm_slice_t sl{};
    sl.axis = axis;
    sl.rank = rank;
    sl.world = world;
    if (axis == GEMM_SPLIT_M) {
        sl.row0 = lo;
        sl.rows = hi - lo;
        sl.col0 = 0;
        sl.cols = N;
    } else {
        sl.row0 = 0;
        sl.rows = M;
        sl.col0 = lo;
        sl.cols = hi - lo;
    }
    *out = sl;
    return GEMM_OK;
}

gemm_status_t gemm_run_slice(gemm_plan_t plan, const gemm_slice_t* slice, const void* A,
                             int64_t lda, const void* B, int64_t ldb, float* C, int64_t ldc,
                             int64_t M, int64_t N, int64_t K, gemm_dtype_t dtype,
                             struct CUstream_st* stream_handle) {
    if (plan == nullptr || slice == nullptr) return GEMM_ERR_INVALID_ARG;
    const gemm_slice_t& sl = *slice;
    if ((sl.axis != GEMM_SPLIT_M && sl.axis != GEMM_SPLIT_N) || sl.row0 < 0 || sl.rows < 0 ||
        sl.col0 < 0 || sl.cols < 0 || M < 0 || N < 0 || sl.row0 > M || sl.col0 > N ||
        sl.rows > M - sl.row0 || sl.cols > N - sl.col0)
        return GEMM_ERR_INVALID_ARG;
    // The whole problem's arguments must be valid on their own.
    const Args whole{A, lda, B, ldb, C, ldc, M, N, K, dtype};
    gemm_status_t st = check_args(whole);
    if (st != GEMM_OK) return st;
    if (sl.rows == 0 || sl.cols == 0) return GEMM_OK;
    const auto* a16 = static_cast<const uint16_t*>(A);
    const auto* b16 = static_cast<const uint16_t*>(B);
    const Args part{K == 0 ? A : a16 + sl.row0 * lda, lda, K == 0 ? B : b16 + sl.col0, ldb,
                    C + sl.row0 * ldc + sl.col0, ldc, sl.rows, sl.cols, K, dtype};
    return run_impl(plan, part, reinterpret_cast<cudaStream_t>(stream_handle));
}

gemm_status_t gemm_wait_selftest(uint32_t timeout_us, struct CUstream_st* stream_handle) {
    cudaStream_t stream = reinterpret_cast<cudaStream_t>(stream_handle);
    int* d = nullptr;
    if (cudaMalloc(&d, sizeof(int)) != cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    int h = 0;
    gemm_status_t st = GEMM_OK;
    if (cudaMemsetAsync(d, 0, sizeof(int), stream) != cudaSuccess ||
        dg::launch_wait_selftest(d, static_cast<uint64_t>(timeout_us) * 1000ull, stream) !=
            cudaSuccess ||
        cudaMemcpyAsync(&h, d, sizeof(int), cudaMemcpyDeviceToHost, stream) != cudaSuccess ||
        cudaStreamSynchronize(stream) != cudaSuccess) {
        (void)cudaGetLastError();
        st = GEMM_ERR_CUDA;
    } else if (h == 2) {
        st = GEMM_ERR_TIMEOUT;
    } else if (h != 1) {
        st = GEMM_ERR_CUDA;
    }
    cudaFree(d);
    return st;
}

gemm_status_t gemm_noop_launch(int32_t grid, int32_t cluster, struct CUstream_st* stream_handle) {
    if (grid < 1 || grid > 65535 || (cluster != 1 && cluster != 2) || grid % cluster != 0)
        return GEMM_ERR_INVALID_ARG;
    if (dg::launch_noop(grid, cluster, reinterpret_cast<cudaStream_t>(stream_handle)) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    return GEMM_OK;
}

}  // extern "C"
