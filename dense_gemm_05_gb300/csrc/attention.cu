// attention.cu -- attention forward on GB300 (sm_103a): the C ABI declared in
// include/attention.h.
//
// The loop of section "Flash Attention in Triton and online softmax" of "How
// to hand-write Triton kernels for matmul and Flash Attention": each block of
// 128 queries of one head walks the key/value blocks (128 keys each)
// and keeps, per query row, a running maximum m, a running sum l and an
// accumulator O that are rescaled by alpha = exp(m_old - m_new) when m
// grows; O / l is written once at the end.  Causal: key j takes part in row i
// only if j <= i, so query block t needs key blocks 0..t, and only block t is
// masked element by element.  Unlike the page's loop, the maximum the weights
// are taken against moves (and O is rescaled) only when the running maximum
// has grown by more than 2^8 in weight (kRescaleLog2): O / l is the same for
// any reference maximum, and weights up to 2^8 fit every type involved.
//
// GB300 mapping: a persistent grid, one CTA per SM.  A work item is one
// (d = 128) or two (d = 64, tiles A and B sharing every K/V block) query
// tiles of one head; each CTA walks its share of the items with one pipeline
// that does not drain between them (the next item's K/V blocks and Q load
// while the softmax finishes the previous one and writes its O).  TMEM per
// tile: the score buffers S (two at d = 128, one at d = 64), P and O:
//   warp 0      TMA producers: lane 0 each item's Q tiles (once the previous
//               item's S MMAs have read the Q buffer) and then its K blocks,
//               lane 1 the V blocks, each into a ring of 4 (d = 64) or 3
//               (d = 128) stages (3-D tensor maps over [BH, seq, d]).
//   warp 1      S issuer (also owns TMEM): S_t(j) = Q_t K_j^T (M 128, N 128,
//               K d) into score buffer j % kSBufs of tile t once K_j has
//               landed and the tile's softmax has read that buffer.
//   warp 2 + t  P V issuer of tile t: O_t += P_t(j) V_j (M 128, N d, K 128)
//               with P_t(j) read from TMEM once the softmax has stored it
//               there.  With S and each tile's P V on separate warps no MMA
//               waits behind another that is not ready.  A K stage is
//               refilled when every tile's S MMAs that read it have
//               completed, a V stage when its P V MMAs have.  (Warp 3 is idle
//               at d = 128.)
//   warps 4..   one softmax warpgroup per tile, one thread per query row
//               (= TMEM lane): read S_t(j) from TMEM, mask, row max,
//               p = 2^(s*c - m*c) with c = log2(e)/sqrt(d), row sum, P_t(j)
//               rounded to the input type into TMEM (the A operand of the
//               second MMA), and when the reference maximum moves the rescale
//               of O_t in TMEM (load, multiply by alpha, store) after
//               P_t(j-1) V_{j-1} has finished.  At d = 64 they also write
//               O_t / l to global memory at the end of each item, and the two
//               warpgroups interleave on the SM's exponential units and issue
//               slots.
//   warps 8..11 (d = 128) the epilogue warpgroup: the softmax hands it each
//               finished item (1/l and the last P) and goes on with the next;
//               it reads O_t from TMEM after the item's last P V, hands O_t
//               back to the next item's first P V, and writes O_t / l.
// Every mbarrier wait is bounded; a role that gives up raises the CTA's abort
// flag and records the failure in a device status word.
#include <atomic>
#include <cmath>
#include <cstdint>
#include <cstdlib>
#include <mutex>

#include <cuda.h>
#include <cuda_runtime.h>

#include "../../include/attention.h"
#include "common.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace {

__device__ int g_attn_status;

// 32-byte global store of eight 32-bit words; the address must be 32-byte aligned.
__device__ __forceinline__ void st_global_v8(void* ptr, const uint32_t* w) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(ptr), "r"(w[0]), "r"(w[1]),
                 "r"(w[2]), "r"(w[3]), "r"(w[4]), "r"(w[5]), "r"(w[6]), "r"(w[7])
                 : "memory");
}

// 3-D tiled bulk tensor prefetch global -> L2 of one box that lies inside the
// tensor (no shared memory, no barrier).
__device__ __forceinline__ void tma_prefetch_3d(const CUtensorMap* map, int32_t x, int32_t y, int32_t z) {
    asm volatile("cp.async.bulk.prefetch.tensor.3d.L2.global.tile [%0, {%1, %2, %3}];" ::"l"(
                     reinterpret_cast<uint64_t>(map)),
                 "r"(x), "r"(y), "r"(z)
                 : "memory");
}

constexpr int kBQ = 128;                  // queries per tile (TMEM lanes)
constexpr int kBKV = 128;                 // keys per block
constexpr int kAtomBytes = 128 * 128;     // 128 rows x 64 elements of a K-major operand (16 KiB)
constexpr int kSubBytes = 64 * 128;       // 64 keys x 64 d of the MN-major V operand (8 KiB)
constexpr uint32_t kTmemCols = 512;       // per tile t at 256 t: kSBufs score buffers S
constexpr uint32_t kTmemS = 128;          //   (128 columns of fp32 each), then P (64 columns,
constexpr uint32_t kTmemTile = 256;       //   two 16-bit values each), then O (d columns of fp32)
constexpr uint64_t kTimeoutNs = 2000000000ull;

// Lazy rescaling: a row keeps the maximum its weights are taken against until
// the running maximum exceeds it by more than 2^kRescaleLog2 in weight, so
// weights stay <= 2^8 (exact in fp32, and in range for 16-bit P) and O is
// rescaled only on the blocks where some row of the warp crossed that margin.
constexpr float kRescaleLog2 = 8.0f;

template <int D>
struct AttnCfg {
    static constexpr int kAtoms = D / 64;
    static constexpr int kTiles = D == 64 ? 2 : 1;
    // K/V ring depth: 4 at d = 64 (measured +1.4 % over 3; 6 no better), 3 at
    // d = 128 (all the shared memory there is).
    static constexpr int kStages = D == 64 ? 4 : 3;
    // Score buffers per tile: with one tile there is room for two, so that the
    // MMA can compute S(j+2) while the softmax still works on S(j+1) and the
    // P V product of block j is queued.
    static constexpr int kSBufs = kTiles == 1 ? 2 : 1;
    static constexpr uint32_t kTmemP = kSBufs * kTmemS;
    static constexpr uint32_t kTmemO = kTmemP + 64;
    static constexpr int kQBytes = kBQ * D * 2;       // per tile: kAtoms atoms
    static constexpr int kKBytes = kBKV * D * 2;      // kAtoms atoms, N = keys
    static constexpr int kVBytes = kBKV * D * 2;      // [64-key half][64-d sub-tile]
    // With one tile an epilogue warpgroup writes O (read from TMEM, scaled by
    // 1/l) while the softmax warpgroup goes on with the next item: the 16- or
    // 32-byte row stores of 64 KiB of O cost the softmax (the critical path)
    // about 9 % at d = 128.  With two tiles the softmax warpgroups write O
    // themselves (no registers are left for a fourth warpgroup).
    static constexpr bool kEpiWG = kTiles == 1;
    static constexpr int kNumBars = 2 + 4 * kStages + kTiles * (2 * kSBufs + 3) + 1 + (kEpiWG ? 3 * kTiles : 0);
    static constexpr int kInvBytes = kEpiWG ? kTiles * 2 * kBQ * 4 : 0;     // 1/l per row, two items
    static constexpr int kSmemBytes =
        1024 + kTiles * kQBytes + kStages * (kKBytes + kVBytes) + kInvBytes + 8 * kNumBars + 16;
    // Warpgroup 0: the producer warp, the S warp and one P V warp per tile (one
    // idle warp at d = 128); then one softmax warpgroup per tile, then (one
    // tile) the epilogue warpgroup; warpgroup-aligned, for the register split.
    static constexpr int kThreads = 32 * (4 + 4 * kTiles + (kEpiWG ? 4 : 0));
    // 384 threads: the launch allows at most 168 registers a thread, fewer
    // than a softmax thread's 128 scores and 64 packed weights need.  So
    // warpgroup 0 gives registers back (setmaxnreg.dec to kRegsLow), the
    // softmax warpgroups take them (setmaxnreg.inc to kRegsHigh) and the
    // epilogue warpgroup keeps the launch's count.  The increase waits until
    // the decrease has freed enough, so the split needs kRegsLow + kTiles
    // kRegsHigh <= (1 + kTiles) x the launch's registers a thread, i.e. at
    // least kRegsMinLaunch; the launcher checks that before launching.
    static constexpr int kRegsLow = kTiles == 2 ? 64 : 72;
    static constexpr int kRegsHigh = kTiles == 2 ? 208 : 232;
    static constexpr int kRegsMinLaunch = (kRegsLow + kTiles * kRegsHigh + kTiles) / (1 + kTiles);
    static_assert(D == 64 || D == 128, "head dimension");
    static_assert(kSmemBytes <= 232448, "shared memory");
    static_assert(kTmemO + D <= kTmemTile || kTiles == 1, "TMEM per tile");
    static_assert((kTiles - 1) * kTmemTile + kTmemO + D <= kTmemCols, "TMEM");
};

struct AttnParams {
    void* O;
    int64_t ldo, hso;
    int64_t items;         // work items: npairs x heads
    int32_t out_type;      // gemm_out_t
    int32_t o_vec;         // 1: 16-byte stores of O rows are legal, 2: 32-byte stores too
    int32_t seq;
    int32_t causal;
    int32_t ntiles;        // query tiles per head
    int32_t npairs;        // work items per head (tiles kTiles p .. kTiles p + kTiles - 1)
    int32_t heads;
    int32_t d;             // head dimension
    float c;               // log2(e) / sqrt(d)
    uint64_t timeout_ns;
};

// The k-th work item of CTA c among G: items are dealt out in rounds of G,
// alternately forwards and backwards, so that with items in decreasing order
// of work every CTA's total stays close to the mean.
__device__ __forceinline__ int64_t item_of(int64_t k, int c, int G) {
    return k * G + ((k & 1) ? G - 1 - c : c);
}

// Item -> (head, pair).  Causal: the work of a pair grows with its index, so
// items run heaviest first across all heads (the heaviest pair of every
// head, then the next, ...).  Otherwise one head's pairs after another, so
// the CTAs of a round share K and V in L2.
__device__ __forceinline__ void item_coords(const AttnParams& p, int64_t L, int* h, int* pair) {
    if (p.causal) {
        *h = static_cast<int>(L % p.heads);
        *pair = p.npairs - 1 - static_cast<int>(L / p.heads);
    } else {
        *h = static_cast<int>(L / p.npairs);
        *pair = static_cast<int>(L % p.npairs);
    }
}

// Key blocks query tile t of a pair needs (0 for a tile beyond the sequence).
template <int kTiles>
__device__ __forceinline__ int tile_blocks(const AttnParams& p, int pair, int t) {
    const int qt = pair * kTiles + t;
    return qt >= p.ntiles ? 0 : (p.causal ? qt + 1 : (p.seq + kBKV - 1) / kBKV);
}

// A wait for a warp off the critical path (the epilogue warpgroup): each poll
// parks the warp on the mbarrier for up to kParkNs (it wakes when the phase
// completes), then the abort flag and the time limit are checked.  Long parks
// keep the waiting warps from taking issue slots from the softmax warps beside
// them (polls with the 1 us hint of the other roles cost d = 128 about 1.5 %).
template <uint32_t kParkNs = 20000u>
__device__ __forceinline__ bool mbar_wait_parked(uint32_t bar, uint32_t parity, const volatile int* abort_flag,
                                                 uint64_t timeout_ns) {
    const uint64_t t0 = dg::global_timer_ns();
    for (uint32_t it = 0; it < (1u << 30); ++it) {
        if (dg::mbar_try_wait_hint(bar, parity, kParkNs)) return true;
        if (*abort_flag) return false;
        if (dg::global_timer_ns() - t0 > timeout_ns) return false;
    }
    return false;
}

// Columns [col0, col0 + kD) of one row of O (already scaled by 1/l) to global
// memory: 32-byte stores when kWide and the layout allows them (o_vec 2),
// 16-byte (o_vec 1), else one element at a time.  A checked build tests the
// span against the sequence and the row (width p.d).
template <int kD, bool kWide>
__device__ __forceinline__ void store_o_span(const AttnParams& p, int h, int qrow, int col0,
                                             const uint32_t (&o)[kD]) {
    if (qrow >= p.seq ||
        !DG_CHECK(&g_attn_status, dg::kChkC, dg::span_inside(qrow, col0, kD, p.seq, p.d)))
        return;
    const int64_t off = int64_t(h) * p.hso + int64_t(qrow) * p.ldo + col0;
    if (p.out_type == dg::kOutF32) {
        float* dst = static_cast<float*>(p.O) + off;
        if (kWide && p.o_vec == 2) {
#pragma unroll
            for (int i = 0; i < kD / 8; ++i) st_global_v8(dst + 8 * i, o + 8 * i);
        } else if (p.o_vec) {
#pragma unroll
            for (int i = 0; i < kD / 4; ++i)
                reinterpret_cast<float4*>(dst)[i] =
                    make_float4(__uint_as_float(o[4 * i]), __uint_as_float(o[4 * i + 1]),
                                __uint_as_float(o[4 * i + 2]), __uint_as_float(o[4 * i + 3]));
        } else {
#pragma unroll
            for (int i = 0; i < kD; ++i) dst[i] = __uint_as_float(o[i]);
        }
    } else {
        uint16_t* dst = static_cast<uint16_t*>(p.O) + off;
        uint32_t w[kD / 2];
#pragma unroll
        for (int i = 0; i < kD / 2; ++i)
            w[i] = dg::pack_out(__uint_as_float(o[2 * i]), __uint_as_float(o[2 * i + 1]), p.out_type);
        if (kWide && p.o_vec == 2) {
#pragma unroll
            for (int i = 0; i < kD / 16; ++i) st_global_v8(dst + 16 * i, w + 8 * i);
        } else if (p.o_vec) {
#pragma unroll
            for (int i = 0; i < kD / 8; ++i)
                reinterpret_cast<uint4*>(dst)[i] = make_uint4(w[4 * i], w[4 * i + 1], w[4 * i + 2], w[4 * i + 3]);
        } else {
#pragma unroll
            for (int i = 0; i < kD; ++i)
                dst[i] = static_cast<uint16_t>((i & 1) ? (w[i / 2] >> 16) : (w[i / 2] & 0xFFFFu));
        }
    }
}

template <bool BF16, int D>
__global__ void __launch_bounds__(AttnCfg<D>::kThreads, 1)
    attention_fwd_kernel(const __grid_constant__ CUtensorMap mapQ,
                         const __grid_constant__ CUtensorMap mapK,
                         const __grid_constant__ CUtensorMap mapV, const AttnParams p) {
    using Cfg = AttnCfg<D>;
    constexpr int kD = D;
    constexpr int kAtoms = Cfg::kAtoms;
    constexpr int kTiles = Cfg::kTiles;
    constexpr int kStages = Cfg::kStages;
    constexpr int kSBufs = Cfg::kSBufs;
    constexpr int kQBytes = Cfg::kQBytes;
    constexpr int kKBytes = Cfg::kKBytes;
    constexpr int kVBytes = Cfg::kVBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sQ = smem;                                  // tile t at t * kQBytes
    uint8_t* sK = sQ + kTiles * kQBytes;
    uint8_t* sV = sK + kStages * kKBytes;
    float* sInv = reinterpret_cast<float*>(sV + kStages * kVBytes);   // [tile][item parity][row]
    uint64_t* bars = reinterpret_cast<uint64_t*>(sV + kStages * kVBytes + Cfg::kInvBytes);
    uint64_t* q_full = bars;
    uint64_t* q_empty = q_full + 1;
    uint64_t* k_full = q_empty + 1;
    uint64_t* v_full = k_full + kStages;
    uint64_t* k_empty = v_full + kStages;                // freed by the S MMAs of the block
    uint64_t* v_empty = k_empty + kStages;               // one arrival per tile
    uint64_t* s_full = v_empty + kStages;                // [tile][score buffer]
    uint64_t* s_empty = s_full + kTiles * kSBufs;
    uint64_t* p_full = s_empty + kTiles * kSBufs;
    uint64_t* pv_done = p_full + kTiles;
    uint64_t* drain = pv_done + kTiles;                  // [S issuer, then P V issuer t]
    uint64_t* o_full = drain + 1 + kTiles;               // [tile][item parity]: last P, 1/l
    uint64_t* o_free = o_full + 2 * kTiles;              // [tile]: O read by the epilogue
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1 + kTiles + (Cfg::kEpiWG ? 3 * kTiles : 0));
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int cta = static_cast<int>(blockIdx.x);
    const int G = static_cast<int>(gridDim.x);

    if (threadIdx.x == 0) {
        dg::mbar_init(dg::smem_u32(q_full), 1u);
        dg::mbar_init(dg::smem_u32(q_empty), 1u);
        for (int s = 0; s < kStages; ++s) {
            dg::mbar_init(dg::smem_u32(&k_full[s]), 1u);
            dg::mbar_init(dg::smem_u32(&v_full[s]), 1u);
            dg::mbar_init(dg::smem_u32(&k_empty[s]), 1u);
            dg::mbar_init(dg::smem_u32(&v_empty[s]), static_cast<uint32_t>(kTiles));
        }
        for (int t = 0; t < kTiles; ++t) {
            for (int b = 0; b < kSBufs; ++b) {
                dg::mbar_init(dg::smem_u32(&s_full[t * kSBufs + b]), 1u);
                dg::mbar_init(dg::smem_u32(&s_empty[t * kSBufs + b]), 128u);
            }
            dg::mbar_init(dg::smem_u32(&p_full[t]), 128u);
            dg::mbar_init(dg::smem_u32(&pv_done[t]), 1u);
        }
        for (int w = 0; w < 1 + kTiles; ++w) dg::mbar_init(dg::smem_u32(&drain[w]), 1u);
        if constexpr (Cfg::kEpiWG) {
            for (int t = 0; t < kTiles; ++t) {
                dg::mbar_init(dg::smem_u32(&o_full[2 * t]), 128u);
                dg::mbar_init(dg::smem_u32(&o_full[2 * t + 1]), 128u);
                dg::mbar_init(dg::smem_u32(&o_free[t]), 128u);
            }
        }
        *abort_flag = 0;
        dg::fence_mbar_init();
    }
    if (warp == 1) {
        dg::tmem_alloc(dg::smem_u32(tmem_slot), kTmemCols);
        dg::tmem_relinquish();
    }
    if (warp == 0 && lane == 0) {
        dg::prefetch_tmap(&mapQ);
        dg::prefetch_tmap(&mapK);
        dg::prefetch_tmap(&mapV);
    }
    dg::tc_fence_before();
    __syncthreads();
    dg::tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    dg::griddep_wait();              // Q, K, V may be written, O still read, by the previous grid
    dg::griddep_launch_dependents();

    auto fail = [&]() {
        *abort_flag = 1;
        atomicOr(&g_attn_status, dg::kDevTimeout);
    };

    // Every role walks the same items in the same order; its barrier phases
    // continue from one item to the next (K/V ring position, score buffer and
    // P hand-over counts), so the pipeline does not drain between items.
    if (warp < 4) {
        // Warpgroup 0: each register-split instruction heads the code of the
        // warpgroup that executes it, so the compiler sizes each side by it.
        dg::setmaxnreg_dec<Cfg::kRegsLow>();
        if (warp == 0) {
            // ------------------------------------------------------------ TMA producers
            // Lane 0 loads each item's Q tiles (once the previous item's S MMAs
            // have read the Q buffer; S(0) needs Q anyway, so K waits with it)
            // and warms L2 with the next item's Q, then the item's K blocks;
            // lane 1 loads V blocks.  A K stage is freed by the S MMAs that
            // read it, a V stage by every tile's P V MMAs, so K runs ahead of
            // the P V products and V into the next item.
            if (lane < 2) {
                bool ok = true;
                uint32_t g = 0;                                   // ring position
                for (int64_t k = 0; ok; ++k) {
                    const int64_t L = item_of(k, cta, G);
                    if (L >= p.items) break;
                    int h, pair;
                    item_coords(p, L, &h, &pair);
                    if (lane == 0) {
                        if (k > 0 && !dg::mbar_wait(dg::smem_u32(q_empty), static_cast<uint32_t>(k - 1) & 1u,
                                                    abort_flag, p.timeout_ns)) {
                            ok = false;
                            break;
                        }
                        const uint32_t qb = dg::smem_u32(q_full);
                        dg::mbar_arrive_expect_tx(qb, kTiles * kQBytes);
                        for (int t = 0; t < kTiles; ++t)
                            for (int a = 0; a < kAtoms; ++a)
                                dg::tma_load_3d(dg::smem_u32(sQ + t * kQBytes + a * kAtomBytes), &mapQ, qb,
                                                64 * a, (pair * kTiles + t) * kBQ, h);
                        const int64_t Ln = item_of(k + 1, cta, G);
                        if (Ln < p.items) {
                            int hn, pn;
                            item_coords(p, Ln, &hn, &pn);
                            for (int t = 0; t < kTiles; ++t)
                                if ((pn * kTiles + t + 1) * kBQ <= p.seq)
                                    for (int a = 0; a < kAtoms; ++a)
                                        tma_prefetch_3d(&mapQ, 64 * a, (pn * kTiles + t) * kBQ, hn);
                        }
                    }
                    const bool k_lane = lane == 0;
                    const int n0 = tile_blocks<kTiles>(p, pair, 0);
                    const int n1 = tile_blocks<kTiles>(p, pair, kTiles - 1);
                    const int nmax = n1 > n0 ? n1 : n0;
                    uint64_t* empty = k_lane ? k_empty : v_empty;
                    for (int j = 0; j < nmax; ++j, ++g) {
                        const int st = static_cast<int>(g % kStages);
                        const uint32_t ph = (g / kStages) & 1u;
                        // The stage held ring entry g - kStages: its readers must be done.
                        if (g >= kStages &&
                            !dg::mbar_wait(dg::smem_u32(&empty[st]), ph ^ 1u, abort_flag, p.timeout_ns)) {
                            ok = false;
                            break;
                        }
                        if (k_lane) {
                            const uint32_t kb = dg::smem_u32(&k_full[st]);
                            dg::mbar_arrive_expect_tx(kb, kKBytes);
                            for (int a = 0; a < kAtoms; ++a)
                                dg::tma_load_3d(dg::smem_u32(sK + st * kKBytes + a * kAtomBytes), &mapK, kb,
                                                64 * a, j * kBKV, h);
                        } else {
                            const uint32_t vb = dg::smem_u32(&v_full[st]);
                            dg::mbar_arrive_expect_tx(vb, kVBytes);
                            const uint32_t vdst = dg::smem_u32(sV + st * kVBytes);
                            for (int hh = 0; hh < 2; ++hh)
                                for (int a = 0; a < kAtoms; ++a)
                                    dg::tma_load_3d(vdst + (hh * kAtoms + a) * kSubBytes, &mapV, vb, 64 * a,
                                                    j * kBKV + hh * (kBKV / 2), h);
                        }
                    }
                }
                if (!ok) fail();
            }
            __syncwarp();
        } else if (warp == 1 || warp - 2 < kTiles) {
            // ------------------------------------------------------------ MMA issuers
            // Warp 1 issues every tile's S_t(j) = Q_t K_j^T; warp 2 + t issues
            // tile t's O_t += P_t(j) V_j.  So no P V MMA waits behind an S MMA
            // that waits for its K block or for its score buffer to be read, nor
            // behind the other tile's P.  S_t(j) goes into the tile's next score
            // buffer once the tile's softmax has read that buffer's previous
            // scores; P_t(j) V_j once P_t(j) is in TMEM and V_j has landed.  The
            // first P V of an item overwrites O_t: its P hand-over comes after
            // the softmax has read O_t of the tile's previous item.  (An S
            // issuer per tile, as two lanes of warp 1, measured slower.)
            const bool s_role = warp == 1;
            const int pv_tile = warp - 2;
            if (lane == 0) {
                constexpr uint32_t idesc_s = dg::idesc_f16(BF16, false, false, kBQ, kBKV);
                constexpr uint32_t idesc_pv = dg::idesc_f16(BF16, false, true, kBQ, kD);
                bool ok = true;
                uint32_t g = 0;                                   // ring position
                uint32_t cnt[kTiles];                             // S: score buffers filled; P V: P hand-overs
                uint32_t epi_items = 0;                           // P V: items of the tile so far
#pragma unroll
                for (int t = 0; t < kTiles; ++t) cnt[t] = 0;
                for (int64_t k = 0; ok; ++k) {
                    const int64_t L = item_of(k, cta, G);
                    if (L >= p.items) break;
                    int h, pair;
                    item_coords(p, L, &h, &pair);
                    int n[kTiles];
#pragma unroll
                    for (int t = 0; t < kTiles; ++t) n[t] = tile_blocks<kTiles>(p, pair, t);
                    const int nmax = n[kTiles - 1] > n[0] ? n[kTiles - 1] : n[0];
                    if (s_role) {
                        ok = dg::mbar_wait(dg::smem_u32(q_full), static_cast<uint32_t>(k) & 1u, abort_flag,
                                           p.timeout_ns);
                        for (int jj = 0; ok && jj < nmax; ++jj, ++g) {
                            const int st = static_cast<int>(g % kStages);
                            ok = dg::mbar_wait(dg::smem_u32(&k_full[st]), (g / kStages) & 1u, abort_flag,
                                               p.timeout_ns);
                            const uint32_t k_addr = dg::smem_u32(sK + st * kKBytes);
#pragma unroll
                            for (int t = 0; t < kTiles; ++t) {
                                if (!ok || jj >= n[t]) continue;
                                const uint32_t b = cnt[t] % kSBufs;
                                // the buffer's (cnt / kSBufs)-th use: its previous scores were read
                                ok = dg::mbar_wait(dg::smem_u32(&s_empty[t * kSBufs + b]),
                                                   ((cnt[t] / kSBufs) & 1u) ^ 1u, abort_flag, p.timeout_ns);
                                if (!ok) break;
                                dg::tc_fence_after();
                                const uint32_t q_addr = dg::smem_u32(sQ + t * kQBytes);
                                const uint32_t s_tmem = tmem_base + static_cast<uint32_t>(t) * kTmemTile +
                                                        b * kTmemS;
#pragma unroll
                                for (int k16 = 0; k16 < kD / 16; ++k16)
                                    dg::tc_mma_f16(s_tmem,
                                                   dg::operand_desc<false>(q_addr + (k16 >> 2) * kAtomBytes, k16 & 3),
                                                   dg::operand_desc<false>(k_addr + (k16 >> 2) * kAtomBytes, k16 & 3),
                                                   idesc_s, k16 > 0 ? 1u : 0u);
                                dg::tc_commit(dg::smem_u32(&s_full[t * kSBufs + b]));
                                ++cnt[t];
                            }
                            if (ok) dg::tc_commit(dg::smem_u32(&k_empty[st]));
                        }
                        if (ok) dg::tc_commit(dg::smem_u32(q_empty));   // the item's S MMAs read Q
                    } else {
                        const int t = pv_tile;
                        const int nt = t == 0 ? n[0] : n[kTiles - 1];
                        for (int j = 0; ok && j < nmax; ++j, ++g) {
                            const int st = static_cast<int>(g % kStages);
                            ok = dg::mbar_wait(dg::smem_u32(&v_full[st]), (g / kStages) & 1u, abort_flag,
                                               p.timeout_ns);
                            if (!ok) break;
                            if (j < nt) {
                                // With an epilogue warpgroup the first P V of an item
                                // overwrites O_t only once it has read the previous item's.
                                if (Cfg::kEpiWG && j == 0 && epi_items > 0)
                                    ok = dg::mbar_wait(dg::smem_u32(&o_free[t]), (epi_items - 1u) & 1u, abort_flag,
                                                       p.timeout_ns);
                                ok = ok && dg::mbar_wait(dg::smem_u32(&p_full[t]), cnt[0] & 1u, abort_flag,
                                                         p.timeout_ns);
                                if (!ok) break;
                                dg::tc_fence_after();
                                const uint32_t v_addr = dg::smem_u32(sV + st * kVBytes);
                                const uint32_t tile_tmem = tmem_base + static_cast<uint32_t>(t) * kTmemTile;
                                // P_t(j) from TMEM (8 columns = 16 keys per MMA), V_j from
                                // shared memory (N = d: kAtoms sub-tiles 8 KiB apart).
#pragma unroll
                                for (int k16 = 0; k16 < kBKV / 16; ++k16)
                                    dg::tc_mma_f16_ts(tile_tmem + Cfg::kTmemO,
                                                      tile_tmem + Cfg::kTmemP + static_cast<uint32_t>(k16 * 8),
                                                      dg::operand_desc<true>(v_addr + (k16 >> 2) * (kVBytes / 2),
                                                                             k16 & 3),
                                                      idesc_pv, (j > 0 || k16 > 0) ? 1u : 0u);
                                dg::tc_commit(dg::smem_u32(&pv_done[t]));
                                ++cnt[0];
                            }
                            // This tile is done with the stage (also when it did not need the block).
                            dg::tc_commit(dg::smem_u32(&v_empty[st]));
                        }
                        if (nt > 0) ++epi_items;
                    }
                }
                if (!ok) fail();
                // Every MMA this thread issued must have completed (and signalled its
                // barriers) before the CTA's shared memory and TMEM go away.
                const volatile int never = 0;
                uint64_t* my_drain = &drain[s_role ? 0 : 1 + pv_tile];
                dg::tc_commit(dg::smem_u32(my_drain));
                dg::mbar_wait(dg::smem_u32(my_drain), 0u, &never, 100000000ull);
            }
            __syncwarp();
        }
    } else if (warp < 4 + 4 * kTiles) {
        dg::setmaxnreg_inc<Cfg::kRegsHigh>();
        // ------------------------------------------------------------ softmax
        const int t = (warp - 4) >> 2;                  // query tile of this warpgroup
        const int quarter = warp & 3;
        const int r = quarter * 32 + lane;              // query row in the tile == TMEM lane
        const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
        const uint32_t tile_addr = lane_addr + static_cast<uint32_t>(t) * kTmemTile;
        const uint32_t p_addr = tile_addr + Cfg::kTmemP;
        const uint32_t o_addr = tile_addr + Cfg::kTmemO;
        const int ptype = BF16 ? dg::kOutBF16 : dg::kOutF16;
        uint32_t cs = 0;                                 // score buffers read
        uint32_t cp = 0;                                 // P hand-overs
        uint32_t items = 0;                              // items handed to the epilogue warpgroup
        bool ok = true;
        for (int64_t k = 0; ok; ++k) {
            const int64_t L = item_of(k, cta, G);
            if (L >= p.items) break;
            int h, pair;
            item_coords(p, L, &h, &pair);
            const int qt = pair * kTiles + t;
            const int qrow = qt * kBQ + r;
            const int n = tile_blocks<kTiles>(p, pair, t);
            float m = -INFINITY, l = 0.0f;
            for (int j = 0; j < n; ++j, ++cs) {
                const uint32_t sb = cs % kSBufs;              // score buffer of block j
                const uint32_t s_addr = tile_addr + sb * kTmemS;
                const bool got = dg::mbar_wait(dg::smem_u32(&s_full[t * kSBufs + sb]), (cs / kSBufs) & 1u,
                                               abort_flag, p.timeout_ns);
                if (!__all_sync(0xffffffffu, got)) {   // tcgen05.ld is warp-collective
                    ok = false;
                    break;
                }
                dg::tc_fence_after();
                // S_t(j) row: all four 32-column loads in flight before one wait; the
                // score buffer is handed back as soon as the values are in registers.
                uint32_t v0[32], v1[32], v2[32], v3[32];
                dg::tmem_ld_32x32b_x32(s_addr, v0);
                dg::tmem_ld_32x32b_x32(s_addr + 32u, v1);
                dg::tmem_ld_32x32b_x32(s_addr + 64u, v2);
                dg::tmem_ld_32x32b_x32(s_addr + 96u, v3);
                dg::tmem_ld_wait(v0);
                dg::tmem_ld_wait(v1);
                dg::tmem_ld_wait(v2);
                dg::tmem_ld_wait(v3);
                dg::tc_fence_before();
                dg::mbar_arrive(dg::smem_u32(&s_empty[t * kSBufs + sb]));   // the buffer may be refilled
                float x[kBKV];
#pragma unroll
                for (int i = 0; i < 32; ++i) {
                    x[i] = __uint_as_float(v0[i]);
                    x[32 + i] = __uint_as_float(v1[i]);
                    x[64 + i] = __uint_as_float(v2[i]);
                    x[96 + i] = __uint_as_float(v3[i]);
                }
                // Mask (only the diagonal block, and the block holding key seq-1):
                // keys at or beyond seq, and (causal) keys after this query.
                const int kv0 = j * kBKV;
                if ((p.causal && j == qt) || kv0 + kBKV > p.seq) {
                    const int lim = min(p.seq, p.causal ? qrow + 1 : p.seq) - kv0;   // keys [kv0, kv0+lim) stay
#pragma unroll
                    for (int i = 0; i < kBKV; ++i)
                        if (i >= lim) x[i] = -INFINITY;
                }
                // Row maximum (four independent chains of three-input max)
                float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int i = 0; i < kBKV; i += 2) mx[(i >> 1) & 3] = dg::fmax3(mx[(i >> 1) & 3], x[i], x[i + 1]);
                const float mb = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
                const float m_new = fmaxf(m, mb);
                // The reference maximum moves to m_new (and O is rescaled) only when
                // some row of the warp would otherwise get weights above 2^8.
                const bool move = m == -INFINITY || (m_new - m) * p.c > kRescaleLog2;
                const bool rescale = __any_sync(0xffffffffu, move);
                const float m_ref = rescale ? m_new : m;
                const float mc = m_ref * p.c;
                const float alpha = rescale ? dg::ex2_approx(m * p.c - mc) : 1.0f;   // 0 on the first block
                // p = 2^(s*c - m*c), two scores per packed fp32 multiply-add and add,
                // summed in fp32 and packed two per 32-bit word (rounded to the input
                // type) as they are made.
                const float2 c2 = make_float2(p.c, p.c);
                const float2 mc2 = make_float2(-mc, -mc);
                float2 sums[2] = {make_float2(0.0f, 0.0f), make_float2(0.0f, 0.0f)};
                uint32_t pw[kBKV / 2];
#pragma unroll
                for (int i = 0; i < kBKV / 2; ++i) {
                    const float2 t2 = __ffma2_rn(make_float2(x[2 * i], x[2 * i + 1]), c2, mc2);
                    const float2 e2 = make_float2(dg::ex2_approx(t2.x), dg::ex2_approx(t2.y));
                    sums[i & 1] = __fadd2_rn(sums[i & 1], e2);
                    pw[i] = dg::pack_out(e2.x, e2.y, ptype);
                }
                l = l * alpha + ((sums[0].x + sums[1].x) + (sums[0].y + sums[1].y));
                if (Cfg::kEpiWG ? cp > 0 : j > 0) {
                    // The previous P V (of this item or, with an epilogue warpgroup,
                    // of the previous one) must be done: it read the P buffer about
                    // to be rewritten, and O_t must hold its sum before the rescale.
                    const bool done = dg::mbar_wait(dg::smem_u32(&pv_done[t]), (cp - 1u) & 1u, abort_flag,
                                                    p.timeout_ns);
                    if (!__all_sync(0xffffffffu, done)) {
                        ok = false;
                        break;
                    }
                    dg::tc_fence_after();
                }
                // P_t(j) into TMEM: this row's 128 weights, two per 32-bit column
                // (the A operand of the P V MMA).
                {
                    uint32_t w0[32], w1[32];
#pragma unroll
                    for (int i = 0; i < 32; ++i) {
                        w0[i] = pw[i];
                        w1[i] = pw[32 + i];
                    }
                    dg::tmem_st_32x32b_x32(p_addr, w0);
                    dg::tmem_st_32x32b_x32(p_addr + 32u, w1);
                }
                dg::tmem_st_wait();
                if (j > 0 && rescale) {
                    // Rescale O_t to the new reference maximum before P_t(j) V_j is added.
#pragma unroll
                    for (int ch = 0; ch < kD / 32; ++ch) {
                        uint32_t v[32];
                        const uint32_t ta = o_addr + static_cast<uint32_t>(ch * 32);
                        dg::tmem_ld_32x32b_x32(ta, v);
                        dg::tmem_ld_wait(v);
#pragma unroll
                        for (int i = 0; i < 32; ++i)
                            v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
                        dg::tmem_st_32x32b_x32(ta, v);
                    }
                    dg::tmem_st_wait();
                }
                dg::tc_fence_before();
                dg::mbar_arrive(dg::smem_u32(&p_full[t]));
                ++cp;
                m = m_ref;
            }
            if (!ok || n == 0) continue;
            if constexpr (Cfg::kEpiWG) {
                // Hand the item to the epilogue warpgroup: 1/l, then the arrival
                // (after the last P hand-over) that releases it.
                sInv[(t * 2 + (items & 1u)) * kBQ + r] = 1.0f / l;
                dg::mbar_arrive(dg::smem_u32(&o_full[t * 2 + (items & 1u)]));
                ++items;
                continue;
            }
            // The tile's last P V product, then O_t / l to global memory.  The
            // next item's first P hand-over (after these TMEM reads) lets its
            // first P V overwrite O_t.
            const bool done = dg::mbar_wait(dg::smem_u32(&pv_done[t]), (cp - 1u) & 1u, abort_flag,
                                            p.timeout_ns);
            if (!__all_sync(0xffffffffu, done)) {
                ok = false;
                continue;
            }
            dg::tc_fence_after();
            const float inv = 1.0f / l;
            uint32_t o[kD];
#pragma unroll
            for (int ch = 0; ch < kD / 32; ++ch) {
                uint32_t v[32];
                dg::tmem_ld_32x32b_x32(o_addr + static_cast<uint32_t>(ch * 32), v);
                dg::tmem_ld_wait(v);
#pragma unroll
                for (int i = 0; i < 32; ++i) o[ch * 32 + i] = __float_as_uint(__uint_as_float(v[i]) * inv);
            }
            dg::tc_fence_before();
            store_o_span<kD, false>(p, h, qrow, 0, o);
        }
        if (!ok) fail();
    } else {
        // ------------------------------------------------------------ epilogue (one tile)
        // Per item and tile: once the softmax has handed over the last P with
        // 1/l and the last P V product is done, read O from TMEM, hand it back
        // (the next item's first P V may overwrite it), scale and write it.
        // The softmax hands an item over only after seeing P V of its block
        // n - 2 done (and this warpgroup saw the previous item's last one), so
        // the awaited P V completion is never more than one phase away.
        if constexpr (Cfg::kEpiWG) {
            const int quarter = warp & 3;
            const int r = quarter * 32 + lane;
            const uint32_t lane_addr = tmem_base + (static_cast<uint32_t>(quarter * 32) << 16);
            uint32_t cp[kTiles], items[kTiles];          // P V products and items so far, per tile
#pragma unroll
            for (int t = 0; t < kTiles; ++t) cp[t] = items[t] = 0;
            bool ok = true;
            for (int64_t k = 0; ok; ++k) {
                const int64_t L = item_of(k, cta, G);
                if (L >= p.items) break;
                int h, pair;
                item_coords(p, L, &h, &pair);
#pragma unroll
                for (int t = 0; t < kTiles; ++t) {
                    const int n = tile_blocks<kTiles>(p, pair, t);
                    if (!ok || n == 0) continue;
                    cp[t] += static_cast<uint32_t>(n);
                    const uint32_t par = items[t] & 1u;
                    bool got = mbar_wait_parked(dg::smem_u32(&o_full[t * 2 + par]), (items[t] >> 1) & 1u,
                                                abort_flag, p.timeout_ns);
                    got = got && mbar_wait_parked(dg::smem_u32(&pv_done[t]), (cp[t] - 1u) & 1u, abort_flag,
                                                  p.timeout_ns);
                    if (!__all_sync(0xffffffffu, got)) {
                        ok = false;
                        continue;
                    }
                    dg::tc_fence_after();
                    const float inv = sInv[(t * 2 + par) * kBQ + r];
                    const uint32_t o_addr = lane_addr + static_cast<uint32_t>(t) * kTmemTile + Cfg::kTmemO;
                    const int qrow = (pair * kTiles + t) * kBQ + r;
                    ++items[t];
                    // All of the row in registers, O handed back, then the stores
                    // 32 columns at a time.
                    uint32_t v[kD / 32][32];
#pragma unroll
                    for (int ch = 0; ch < kD / 32; ++ch)
                        dg::tmem_ld_32x32b_x32(o_addr + static_cast<uint32_t>(ch * 32), v[ch]);
#pragma unroll
                    for (int ch = 0; ch < kD / 32; ++ch) dg::tmem_ld_wait(v[ch]);
                    dg::tc_fence_before();
                    dg::mbar_arrive(dg::smem_u32(&o_free[t]));
#pragma unroll
                    for (int ch = 0; ch < kD / 32; ++ch) {
#pragma unroll
                        for (int i = 0; i < 32; ++i) v[ch][i] = __float_as_uint(__uint_as_float(v[ch][i]) * inv);
                        store_o_span<32, true>(p, h, qrow, ch * 32, v[ch]);
                    }
                }
            }
            if (!ok) fail();
        }
    }

    if (*abort_flag && threadIdx.x == 0) {
        // Copies already issued may still land in this CTA's shared memory:
        // give them a bounded 2 ms before the CTA leaves.
        const uint64_t t0 = dg::global_timer_ns();
        while (dg::global_timer_ns() - t0 < 2000000ull) {
        }
    }
    dg::tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        dg::tc_fence_after();
        dg::tmem_dealloc(tmem_base, kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* q = nullptr;
        cudaDriverEntryPointQueryResult r{};
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &q, 12000,
                                             cudaEnableDefault, &r) == cudaSuccess &&
            r == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(q);
        else
            (void)cudaGetLastError();
    });
    return fn;
}

// [BH, seq, d] view with row pitch ld and head pitch hs (elements); boxes of
// 64 d (one 128-byte swizzle row) x `rows` rows x 1 head, zero fill beyond seq.
bool encode_qkv(CUtensorMap* map, bool bf16, const void* ptr, int64_t BH, int64_t seq, int64_t d,
                int64_t ld, int64_t hs, uint32_t rows) {
    EncodeTiledFn fn = encode_fn();
    if (fn == nullptr) return false;
    cuuint64_t dims[3] = {static_cast<cuuint64_t>(d), static_cast<cuuint64_t>(seq),
                          static_cast<cuuint64_t>(BH)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(ld) * 2, static_cast<cuuint64_t>(hs) * 2};
    cuuint32_t box[3] = {64u, rows, 1u};
    cuuint32_t estr[3] = {1u, 1u, 1u};
    return fn(map, bf16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16 : CU_TENSOR_MAP_DATA_TYPE_FLOAT16, 3,
              const_cast<void*>(ptr), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
              CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
              CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

struct DeviceFacts {
    bool known = false;
    bool sm103 = false;
    int sms = 0;
};

std::mutex g_mu;
DeviceFacts g_dev[64];
bool g_attr_set[4] = {false, false, false, false};   // [bf16 + 2 * (d == 128)]

bool device_ok(bool* sm103, int* sms) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
        (void)cudaGetLastError();
        return false;
    }
    std::lock_guard<std::mutex> lock(g_mu);
    DeviceFacts& f = g_dev[dev];
    if (!f.known) {
        int major = 0, minor = 0, count = 0;
        if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
            cudaDeviceGetAttribute(&count, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) {
            (void)cudaGetLastError();
            return false;
        }
        f.sm103 = major == 10 && minor == 3;
        f.sms = count;
        f.known = true;
    }
    *sm103 = f.sm103;
    *sms = f.sms;
    return true;
}

// Bytes [begin, end) spanned by a [BH, seq, width] strided view.
void span(const void* ptr, int64_t BH, int64_t seq, int64_t width, int64_t ld, int64_t hs,
          int64_t esize, uintptr_t* b, uintptr_t* e) {
    *b = reinterpret_cast<uintptr_t>(ptr);
    *e = *b + static_cast<uintptr_t>(((BH - 1) * hs + (seq - 1) * ld + width) * esize);
}

gemm_status_t check(const void* Q, const void* K, const void* V, const void* O, int64_t BH,
                    int64_t seq, int64_t d, int64_t ld, int64_t hs, int64_t ldo, int64_t hso,
                    gemm_dtype_t dtype, int32_t out_type) {
    if (BH < 0 || seq < 0 || d < 0 || ld < 0 || hs < 0 || ldo < 0 || hso < 0)
        return GEMM_ERR_INVALID_ARG;
    if (dtype != GEMM_F16 && dtype != GEMM_BF16) return GEMM_ERR_UNSUPPORTED;
    if (out_type != GEMM_OUT_F32 && out_type != GEMM_OUT_F16 && out_type != GEMM_OUT_BF16)
        return GEMM_ERR_UNSUPPORTED;
    if (BH == 0 || seq == 0) return GEMM_OK;
    if (Q == nullptr || K == nullptr || V == nullptr || O == nullptr) return GEMM_ERR_INVALID_ARG;
    if (ld < d || ldo < d) return GEMM_ERR_INVALID_ARG;
    const int64_t osz = out_type == GEMM_OUT_F32 ? 4 : 2;
    if ((reinterpret_cast<uintptr_t>(Q) | reinterpret_cast<uintptr_t>(K) |
         reinterpret_cast<uintptr_t>(V)) % 16u != 0u ||
        reinterpret_cast<uintptr_t>(O) % static_cast<uintptr_t>(osz) != 0u)
        return GEMM_ERR_INVALID_ARG;
    if (d != 64 && d != 128) return GEMM_ERR_UNSUPPORTED;
    // seq <= 2^31 - 256 keeps every row and key index the kernel forms (the
    // first row of the block after the last, a key block's end) inside int32.
    if (ld % 8 != 0 || hs % 8 != 0 || BH > 65535 || seq > int64_t(INT32_MAX) - 255 ||
        ld > (int64_t(1) << 36) || hs > (int64_t(1) << 36) || ldo > (int64_t(1) << 36) ||
        hso > (int64_t(1) << 36))
        return GEMM_ERR_UNSUPPORTED;
    uintptr_t ob, oe;
    span(O, BH, seq, d, ldo, hso, osz, &ob, &oe);
    for (const void* t : {Q, K, V}) {
        uintptr_t tb, te;
        span(t, BH, seq, d, ld, hs, 2, &tb, &te);
        if (ob < te && tb < oe) return GEMM_ERR_INVALID_ARG;
    }
    return GEMM_OK;
}

// Debug settings (attention_set_debug): -1 = debug-sync as GEMM_DEBUG_SYNC says.
std::atomic<int> g_debug_sync{-1};
std::atomic<uint64_t> g_timeout_ns{kTimeoutNs};

bool debug_sync() {
    static const bool env_on = [] {
        const char* e = std::getenv("GEMM_DEBUG_SYNC");
        return e != nullptr && e[0] == '1';
    }();
    const int forced = g_debug_sync.load(std::memory_order_relaxed);
    return forced < 0 ? env_on : forced != 0;
}

}  // namespace

extern "C" {

gemm_status_t attention_set_debug(int32_t sync, uint64_t timeout_ns) {
    if (sync < -1 || sync > 1) return GEMM_ERR_INVALID_ARG;
    g_debug_sync.store(sync, std::memory_order_relaxed);
    g_timeout_ns.store(timeout_ns != 0 ? timeout_ns : kTimeoutNs, std::memory_order_relaxed);
    return GEMM_OK;
}

gemm_status_t attention_fwd_query(const void* Q, const void* K, const void* V, const void* O,
                                  int64_t BH, int64_t seq, int64_t d, int64_t ld,
                                  int64_t head_stride, int64_t ldo, int64_t head_stride_o,
                                  int32_t causal, gemm_dtype_t dtype, int32_t out_type,
                                  attention_config_t* out) {
    if (out == nullptr) return GEMM_ERR_INVALID_ARG;
    const gemm_status_t st =
        check(Q, K, V, O, BH, seq, d, ld, head_stride, ldo, head_stride_o, dtype, out_type);
    if (st != GEMM_OK) return st;
    *out = attention_config_t{};
    out->block_q = kBQ;
    out->block_kv = kBKV;
    out->head_dim = static_cast<int32_t>(d);
    out->stages = d == 64 ? AttnCfg<64>::kStages : AttnCfg<128>::kStages;
    const int tiles_per_cta = d == 64 ? AttnCfg<64>::kTiles : AttnCfg<128>::kTiles;
    out->grid_x = static_cast<int32_t>(((seq + kBQ - 1) / kBQ + tiles_per_cta - 1) / tiles_per_cta);
    out->grid_y = static_cast<int32_t>(BH);
    out->causal = causal ? 1 : 0;
    return GEMM_OK;
}

gemm_status_t attention_fwd(const void* Q, const void* K, const void* V, void* O, int64_t BH,
                            int64_t seq, int64_t d, int64_t ld, int64_t head_stride, int64_t ldo,
                            int64_t head_stride_o, int32_t causal, gemm_dtype_t dtype,
                            int32_t out_type, struct CUstream_st* stream) {
    const gemm_status_t st =
        check(Q, K, V, O, BH, seq, d, ld, head_stride, ldo, head_stride_o, dtype, out_type);
    if (st != GEMM_OK || BH == 0 || seq == 0) return st;
    bool sm103 = false;
    int sms = 0;
    if (!device_ok(&sm103, &sms)) return GEMM_ERR_CUDA;
    if (!sm103 || sms <= 0) return GEMM_ERR_UNSUPPORTED;
    const bool bf16 = dtype == GEMM_BF16;
    CUtensorMap mq, mk, mv;
    if (!encode_qkv(&mq, bf16, Q, BH, seq, d, ld, head_stride, kBQ) ||
        !encode_qkv(&mk, bf16, K, BH, seq, d, ld, head_stride, kBKV) ||
        !encode_qkv(&mv, bf16, V, BH, seq, d, ld, head_stride, kBKV / 2))
        return GEMM_ERR_CUDA;
    using Kernel = void (*)(CUtensorMap, CUtensorMap, CUtensorMap, AttnParams);
    const bool d64 = d == 64;
    const Kernel kernel = d64 ? (bf16 ? attention_fwd_kernel<true, 64> : attention_fwd_kernel<false, 64>)
                              : (bf16 ? attention_fwd_kernel<true, 128> : attention_fwd_kernel<false, 128>);
    const int smem_bytes = d64 ? AttnCfg<64>::kSmemBytes : AttnCfg<128>::kSmemBytes;
    const int threads = d64 ? AttnCfg<64>::kThreads : AttnCfg<128>::kThreads;
    const int tiles_per_cta = d64 ? AttnCfg<64>::kTiles : AttnCfg<128>::kTiles;
    {
        std::lock_guard<std::mutex> lock(g_mu);
        const int which = (bf16 ? 1 : 0) + (d64 ? 0 : 2);
        if (!g_attr_set[which]) {
            if (cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                     smem_bytes) != cudaSuccess) {
                (void)cudaGetLastError();
                return GEMM_ERR_CUDA;
            }
            // The register split needs this many registers a thread at launch
            // (otherwise its increase would wait forever): refuse to launch a
            // build that has fewer.
            {
                cudaFuncAttributes fa{};
                if (cudaFuncGetAttributes(&fa, kernel) != cudaSuccess) {
                    (void)cudaGetLastError();
                    return GEMM_ERR_CUDA;
                }
                if (fa.numRegs < (d64 ? AttnCfg<64>::kRegsMinLaunch : AttnCfg<128>::kRegsMinLaunch))
                    return GEMM_ERR_UNSUPPORTED;
            }
            g_attr_set[which] = true;
        }
    }
    AttnParams p{};
    p.O = O;
    p.ldo = ldo;
    p.hso = head_stride_o;
    p.out_type = out_type;
    const int64_t ovec = out_type == GEMM_OUT_F32 ? 4 : 8;
    p.o_vec = (reinterpret_cast<uintptr_t>(O) % 16u == 0u && ldo % ovec == 0 &&
               head_stride_o % ovec == 0)
                  ? 1
                  : 0;
    if (p.o_vec && reinterpret_cast<uintptr_t>(O) % 32u == 0u && ldo % (2 * ovec) == 0 &&
        head_stride_o % (2 * ovec) == 0)
        p.o_vec = 2;   // 32-byte stores
    p.seq = static_cast<int32_t>(seq);
    p.causal = causal ? 1 : 0;
    p.ntiles = static_cast<int32_t>((seq + kBQ - 1) / kBQ);
    p.npairs = (p.ntiles + tiles_per_cta - 1) / tiles_per_cta;
    p.heads = static_cast<int32_t>(BH);
    p.d = static_cast<int32_t>(d);
    p.items = int64_t(p.npairs) * BH;
    p.c = static_cast<float>(1.4426950408889634 / std::sqrt(static_cast<double>(d)));
    p.timeout_ns = g_timeout_ns.load(std::memory_order_relaxed);
    // Persistent: one CTA per SM (each holds all of an SM's shared memory),
    // walking its share of the items.
    const dim3 grid(static_cast<unsigned>(p.items < sms ? p.items : sms));
    const cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    // Launched as a programmatic dependent (the kernel waits before touching memory).
    if (dg::launch_pdl(kernel, grid, dim3(threads), size_t(smem_bytes), s, mq, mk, mv, p) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return GEMM_ERR_CUDA;
    }
    if (debug_sync()) {
        if (cudaStreamSynchronize(s) != cudaSuccess) {
            (void)cudaGetLastError();
            return GEMM_ERR_CUDA;
        }
        int status = 0;
        if (cudaMemcpyFromSymbol(&status, g_attn_status, sizeof(int)) != cudaSuccess)
            return GEMM_ERR_CUDA;
        if (status != 0) {
            const int zero = 0;
            (void)cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int));
            return (status & dg::kDevBounds) ? GEMM_ERR_BOUNDS : GEMM_ERR_TIMEOUT;
        }
    }
    return GEMM_OK;
}

}  // extern "C"
