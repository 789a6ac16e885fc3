// common.cuh -- parameters, tile order and launcher declarations shared by the
// kernel translation units and the C-ABI layer of the GEMM library.
#pragma once

#include <cstdint>
#include <utility>
#include <cuda.h>
#include <cuda_runtime.h>

namespace dg {

constexpr int kBM = 128;                 // rows of C per CTA tile (TMEM lanes)
constexpr int kBK = 64;                  // K depth of one stage: 64 x 2 B = one 128-B swizzle row
constexpr int kAStageBytes = kBM * kBK * 2;
constexpr int kSubN = 64;                // columns of one MN-major swizzle sub-tile (128 B)
constexpr int kSubTileBytes = kSubN * kBK * 2;   // 8 KB: 64 K-rows of 128 B

// Status word bits.  kDevTimeout: a bounded wait gave up.  kDevBounds: a
// checked build (below) skipped an access outside its matrix or buffer; the
// kChk* bits say which kind of access it was.
constexpr int kDevTimeout = 1;
constexpr int kDevBounds = 2;
constexpr int kChkC = 1 << 8;         // a store of C outside rows [0, M) x columns [0, N)
constexpr int kChkA = 1 << 9;         // a load of A outside its stored rectangle
constexpr int kChkB = 1 << 10;        // a load of B outside its stored rectangle
constexpr int kChkWs = 1 << 11;       // a partial-sum access outside the plan's workspace
constexpr int kChkCounter = 1 << 12;  // a tile-counter access outside the counter array
constexpr int kChkStage = 1 << 13;    // the staging copy outside its source or destination

// Checked builds.  Compiled with DG_CHECKED=1 (the library libgemm_checked.so),
// every ordinary global load and store of the kernels first tests the range it
// touches against the matrix or buffer it belongs to -- the rectangle of rows x
// columns the caller passed, or the plan's workspace -- and is skipped when the
// test fails, which sets kDevBounds and the access's bit in the status word (a
// debug-sync gemm_run reports it).  TMA copies are not tested: their tensor
// maps bound them in hardware (elements outside read as zeros, stores are
// clipped).  In the normal build the tests are the constant true.
#ifndef DG_CHECKED
#define DG_CHECKED 0
#endif

// Elements [c, c + n) of row r lie inside a rows x cols rectangle (n >= 1).
__host__ __device__ __forceinline__ bool span_inside(int64_t r, int64_t c, int64_t n, int64_t rows,
                                                     int64_t cols) {
    return r >= 0 && r < rows && c >= 0 && n >= 1 && c <= cols - n;
}

// Bytes [a, a + n) lie inside [lo, hi).
__host__ __device__ __forceinline__ bool bytes_inside(uintptr_t a, uintptr_t n, uintptr_t lo,
                                                      uintptr_t hi) {
    return a >= lo && a <= hi && n <= hi - a;
}

#if DG_CHECKED
__device__ __forceinline__ bool check_record(int* status, int kind, bool ok) {
    if (!ok && status != nullptr) atomicOr(status, kDevBounds | kind);
    return ok;
}
#define DG_CHECK(status, kind, cond) ::dg::check_record((status), (kind), (cond))
#else
#define DG_CHECK(status, kind, cond) true
#endif

struct Params {
    const uint16_t* A;
    const uint16_t* B;
    void* C;                // fp32, fp16 or bf16 elements (c_type)
    int32_t c_type;         // 0 fp32, 1 fp16, 2 bf16
    int64_t lda, ldb, ldc;
    int32_t M, N, K;
    int32_t tiles_m, tiles_n, num_kb;
    int32_t group;          // group-major strip height (0 = row-major)
    int32_t shares;         // skinny / pair: equal stream-K shares of the (tile, K block) iterations
    int32_t max_slots;      // skinny: partial-tile slots per output tile in the workspace
    int32_t sk_tiles;       // pair: tiles [0, sk_tiles) are split into `shares` stream-K shares
    int32_t a_vec, b_vec;   // generic producer: 16-byte vector loads are legal
    int32_t c_vec;          // 16-byte vector stores of C are legal
    int32_t c_tma;          // the epilogue writes C with TMA stores (mapC is valid)
    int32_t prefetch_kb;    // split pair, skinny: K blocks per CTA warmed in L2 before the grid wait
    float* ws;              // skinny, pair: split-K partial sums
    int* counters;          // skinny, pair: per-tile arrival counters (zero between launches)
    int64_t ws_len;         // floats at ws (the range a checked build tests against)
    int64_t counters_len;   // ints at counters
    int* status;            // device error word (kDev* bits)
    uint64_t timeout_ns;    // limit of every device-side wait
};

// Linear work index t -> (tile row, tile column).
// group > 0: group-major order of "I Wrote a GPU Matmul Kernel From Scratch in
// Triton", Step 4 -- strips of `group` tile rows, walked column by column,
// the last strip only as tall as the rows that remain.  group <= 0: row-major
// order of the "Triton 04" teaching kernel.
__host__ __device__ __forceinline__ void tile_coord(int64_t t, int64_t tiles_m, int64_t tiles_n,
                                                    int group, int64_t& tm, int64_t& tn) {
    if (group <= 0) {
        tm = t / tiles_n;
        tn = t - tm * tiles_n;
        return;
    }
    const int64_t per_strip = static_cast<int64_t>(group) * tiles_n;
    const int64_t strip = t / per_strip;
    const int64_t first = strip * group;
    const int64_t rem = tiles_m - first;
    const int64_t height = rem < group ? rem : group;
    const int64_t local = t - strip * per_strip;
    tm = first + local % height;
    tn = local / height;
}

__device__ __forceinline__ void tile_coord32(int t, int tiles_m, int tiles_n, int group, int& tm,
                                             int& tn) {
    if (group <= 0) {
        tm = t / tiles_n;
        tn = t - tm * tiles_n;
        return;
    }
    const int per_strip = group * tiles_n;
    const int strip = t / per_strip;
    const int first = strip * group;
    const int rem = tiles_m - first;
    const int height = rem < group ? rem : group;
    const int local = t - strip * per_strip;
    tm = first + local % height;
    tn = local / height;
}

// Stream-K shares of the skinny kernel.  The T = tiles * num_kb (tile, K block)
// iterations, tile-major, are cut into G contiguous shares; share c covers
// [c*T/G, (c+1)*T/G).  G <= 4096 and T < 2^49 keep the products in int64.
__host__ __device__ __forceinline__ int64_t share_begin(int64_t c, int64_t T, int64_t G) {
    return c * T / G;
}

// The share that contains iteration i (the largest c with share_begin(c) <= i).
__host__ __device__ __forceinline__ int64_t share_of(int64_t i, int64_t T, int64_t G) {
    return ((i + 1) * G - 1) / T;
}

// Upper bound on how many shares can touch one tile's num_kb iterations.
__host__ __device__ __forceinline__ int shares_per_tile_bound(int64_t T, int64_t G, int num_kb) {
    const int64_t shortest = T / G;   // every share has at least this many iterations
    return static_cast<int>((num_kb + shortest - 1) / shortest) + 1;
}

// Cost model of the skinny kernel, in units of one 64-deep K block streamed by
// one SM (measured on GB300 with graph-replayed launches): HBM saturates at
// about 100 SMs streaming at once, and a split tile's fix-up (partial stores,
// arrival counter, last-arriver reduction) costs about 10 K blocks.
constexpr int64_t kSkinnyDramStreams = 100;
constexpr int64_t kSkinnyFixupKb = 10;
constexpr int64_t kSkinnyMinShareKb = 4;   // a split share streams at least this many K blocks
constexpr int64_t kSkinnyMaxShares = 4096;

inline int64_t skinny_cost(int64_t T, int64_t G, int num_sms, int tiles) {
    const int64_t waves = (G + num_sms - 1) / num_sms;
    const int64_t longest = waves * ((T + G - 1) / G);
    const int64_t dram = (T + kSkinnyDramStreams - 1) / kSkinnyDramStreams;
    const bool split = G != tiles;   // one share per tile covers every tile whole
    return (longest > dram ? longest : dram) + (split ? kSkinnyFixupKb : 0);
}

// The cheapest share count under skinny_cost among one share per tile, 2-4
// equal shares per tile, and one share per SM.
inline int64_t skinny_auto_shares(int tiles, int num_kb, int num_sms) {
    const int64_t T = int64_t(tiles) * num_kb;
    const int64_t per_sm = (T / kSkinnyMinShareKb < num_sms) ? T / kSkinnyMinShareKb : num_sms;
    const int64_t cands[5] = {tiles, 2 * int64_t(tiles), 3 * int64_t(tiles), 4 * int64_t(tiles),
                              per_sm};
    int64_t best_g = tiles, best = -1;
    for (int64_t g : cands) {
        if (g > T) g = T;
        if (g > kSkinnyMaxShares) g = kSkinnyMaxShares;
        if (g < 1) g = 1;
        const int64_t cost = skinny_cost(T, g, num_sms, tiles);
        if (best < 0 || cost < best) {
            best = cost;
            best_g = g;
        }
    }
    return best_g;
}

// ---------------------------------------------------------------- launchers
// Each returns cudaSuccess or the launch error; none synchronises.

// Launch as a programmatic dependent of the previous work in the stream: the
// kernel may start (barrier setup, TMEM allocation, descriptor prefetch) while
// that work drains, and waits for it (griddepcontrol.wait) before it touches
// global memory.  Every kernel launched this way makes that wait before its
// first global access.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// a_mn: A is stored K x M (transposed, M contiguous); otherwise M x K.
// b_mn: B is stored K x N (N contiguous); otherwise N x K (transposed).

// Persistent tcgen05 kernel, operands by TMA: tiles of bm x bn, bn in {64, 128,
// 256}, bm = 128 (or 64 with bn = 64: M = 64 MMAs, for problems with few tiles).
int tma_smem_bytes(int bm, int bn);
int tma_stages(int bn);
cudaError_t tma_prepare();
cudaError_t launch_tma(int bm, int bn, bool a_mn, bool b_mn, const CUtensorMap& mapA,
                       const CUtensorMap& mapB, const CUtensorMap& mapC, const Params& p,
                       uint32_t idesc, int grid, cudaStream_t stream);

// Same pipeline, operands staged by ordinary loads (any alignment). bn = 128.
int generic_smem_bytes();
int generic_stages();
cudaError_t generic_prepare();
cudaError_t launch_generic(bool a_mn, bool b_mn, const Params& p, uint32_t idesc, int grid,
                           cudaStream_t stream);

// Skinny M: swap-AB + stream-K. ms in {16, 32, 64} (MMA N = padded M); A is M x K.
int skinny_smem_bytes(int ms);
int skinny_stages(int ms);
cudaError_t skinny_prepare();
cudaError_t launch_skinny(int ms, bool b_mn, const CUtensorMap& mapB, const CUtensorMap& mapA,
                          const Params& p, uint32_t idesc, int grid, cudaStream_t stream);

// CTA-pair (cta_group::2) kernel, 256 x bn pair tiles, operands by TMA. bn in {128, 256}.
int pair_smem_bytes(int bn);
int pair_stages(int bn);
cudaError_t pair_prepare();
int pair_max_clusters(int bn);   // co-resident 2-CTA clusters on the current device (0 = unknown)
cudaError_t launch_pair(int bn, bool a_mn, bool b_mn, const CUtensorMap& mapA,
                        const CUtensorMap& mapB, const CUtensorMap& mapC, const Params& p,
                        uint32_t idesc, int grid, cudaStream_t stream);

// 2-CTA clusters that split each output tile's K loop in halves and exchange half
// of their partials through distributed shared memory.  ms in {16, 32, 64} (M <= 64
// padded: one strip of rows) with bn in {128, 192, 256}, or ms = 128 (tiles of 128
// rows) with bn = 128; grid = 2 x tiles_m x tiles_n; num_kb >= 2; A not transposed.
// b_gen (ms = 128, b_mn only): B is not 16-byte aligned and is read in place with
// ordinary loads (mapB unused).
int splitpair_stages(int ms, int bn, bool b_gen);
cudaError_t splitpair_prepare();
int splitpair_max_clusters();       // co-resident 2-CTA clusters (0 = unknown)
cudaError_t launch_splitpair(int ms, int bn, bool b_mn, bool b_gen, const CUtensorMap& mapA,
                             const CUtensorMap& mapB, const CUtensorMap& mapC, const Params& p,
                             uint32_t idesc, int grid, cudaStream_t stream);

// Copy a rows x cols 16-bit matrix (pitch lds) into dst with pitch ldd (a multiple
// of 8 elements, dst 16-byte aligned), zero-filling columns [cols, ldd).
cudaError_t launch_stage_rows(const uint16_t* src, int64_t lds, uint16_t* dst, int64_t ldd,
                              int64_t rows, int64_t cols, int* status, int num_sms,
                              cudaStream_t stream);

// Wait self-test: one block waits on a barrier nobody completes.
cudaError_t launch_wait_selftest(int* out, uint64_t timeout_ns, cudaStream_t stream);

// A kernel with no work, launched like the GEMM kernels (grid, cluster of 1 or 2,
// programmatic dependent launch): the launch floor.
cudaError_t launch_noop(int grid, int cluster, cudaStream_t stream);

}  // namespace dg
