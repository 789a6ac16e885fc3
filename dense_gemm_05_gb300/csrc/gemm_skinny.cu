// gemm_skinny.cu -- small-M GEMM for sm_103a: swap-AB + stream-K split of K.
//
// For M <= 64 the product is computed transposed, C^T[N, M] = B^T[N, K] A^T[K, M],
// so N fills the 128 rows of the tcgen05 MMA and the padded M (16, 32 or 64)
// is the MMA's N.  B, the large operand, is read once from HBM: the problem is
// bound by that stream, not by the tensor cores.
//
// To put every SM on the stream, the (tile, K block) iterations of all
// 128-column tiles, taken tile by tile, are cut into G equal contiguous shares
// (one per CTA): each CTA streams the same number of K blocks of B, and a tile
// is computed by at most a few consecutive CTAs, each summing its own run of
// K blocks (the K-sum of "Writing GPU kernels in Triton", section 3.3,
// regrouped; the regrouping is exact up to rounding because the sum is
// associative).  A CTA that covers a whole tile stores C directly.  Otherwise
// it writes its fp32 partial tile to slot (share - first share of the tile) of
// the plan's workspace; the last of the tile's shares to arrive (a per-tile
// counter) adds the partials in slot order 0, 1, ... and writes C, so the
// result is the same bits on every run whatever order the shares finish in.
// It then resets the counter to zero for the next launch.
//
// Warp roles are those of gemm_tc.cu: warp 0 MMA issuer + TMEM owner, warps
// 1..4 epilogue, warp 5 TMA producer.  All three walk the same segments.
#include "common.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace dg {

template <int MS, int STAGES>
struct SkCfg {
    static constexpr int kBtStageBytes = 128 * kBK * 2;   // B^T tile: 128 n x 64 k (two sub-tiles)
    static constexpr int kAStageBytes = MS * kBK * 2;      // A tile: MS m x 64 k, K-major
    static constexpr int kStageBytes = kBtStageBytes + kAStageBytes;
    static constexpr int kTmemCols = (2 * MS < 32) ? 32 : 2 * MS;
    static constexpr int kThreads = 192;
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr int kSmemBytes = 1024 + STAGES * kStageBytes + 8 * kNumBars + 16;
    static_assert(MS == 16 || MS == 32 || MS == 64, "MS");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// One contiguous run of K blocks [kb0, kb1) of one tile, inside one share.
struct Segment {
    int tile;
    int kb0, kb1;
};

// Walks the segments of the shares this CTA owns (share c = blockIdx.x, then
// += gridDim.x), in the same order in every role.
struct SegmentWalker {
    int64_t T, G;
    int num_kb;
    int64_t share, it, end;

    __device__ SegmentWalker(int tiles, int nkb, int shares)
        : T(int64_t(tiles) * nkb), G(shares), num_kb(nkb), share(blockIdx.x) {
        it = share < G ? share_begin(share, T, G) : 0;
        end = share < G ? share_begin(share + 1, T, G) : 0;
    }
    __device__ bool next(Segment& s) {
        while (it >= end) {
            share += gridDim.x;
            if (share >= G) return false;
            it = share_begin(share, T, G);
            end = share_begin(share + 1, T, G);
        }
        s.tile = static_cast<int>(it / num_kb);
        s.kb0 = static_cast<int>(it - int64_t(s.tile) * num_kb);
        const int64_t left = end - it;
        s.kb1 = (num_kb - s.kb0 < left) ? num_kb : s.kb0 + static_cast<int>(left);
        it += s.kb1 - s.kb0;
        return true;
    }
};

template <int MS>
__device__ __forceinline__ void load_acc(uint32_t taddr, float (&v)[MS]) {
    if constexpr (MS == 16) {
        uint32_t r[16];
        tmem_ld_32x32b_x16(taddr, r);
        tmem_ld_wait(r);
#pragma unroll
        for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
    } else {
#pragma unroll
        for (int h = 0; h < MS / 32; ++h) {
            uint32_t r[32];
            tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(h * 32), r);
            tmem_ld_wait(r);
#pragma unroll
            for (int i = 0; i < 32; ++i) v[h * 32 + i] = __uint_as_float(r[i]);
        }
    }
}

template <int MS, int STAGES, bool B_MN>
__global__ void __launch_bounds__(192, 1)
    gemm_skinny_kernel(const __grid_constant__ CUtensorMap mapB,
                       const __grid_constant__ CUtensorMap mapA, const Params p,
                       const uint32_t idesc) {
    using Cfg = SkCfg<MS, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sBt = smem;
    uint8_t* sA = smem + STAGES * Cfg::kBtStageBytes;
    uint64_t* bars = reinterpret_cast<uint64_t*>(sA + STAGES * Cfg::kAStageBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = abort_flag + 1;

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1u);
            mbar_init(smem_u32(&empty[s]), 1u);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1u);
            mbar_init(smem_u32(&tempty[a]), 128u);
        }
        mbar_init(smem_u32(drain), 1u);
        *abort_flag = 0;
        *last_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    if (warp == 5 && lane == 0) {
        prefetch_tmap(&mapA);
        prefetch_tmap(&mapB);
        // Warm L2 with the first K blocks of this CTA's first segment while the
        // previous grid finishes (a prefetch hands no data to this CTA).
        SegmentWalker walk(p.tiles_n, p.num_kb, p.shares);
        Segment sg;
        if (p.prefetch_kb > 0 && walk.next(sg)) {
            const uint64_t pol_stream = l2_policy_evict_first();
            const uint64_t pol_keep = l2_policy_evict_last();
            for (int kb = sg.kb0; kb < sg.kb1 && kb < sg.kb0 + p.prefetch_kb; ++kb) {
                prefetch_operand_hint<B_MN>(&mapB, sg.tile * 128, kb * kBK, 128, pol_stream);
                tma_prefetch_2d_hint(&mapA, kb * kBK, 0, pol_keep);
            }
        }
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();                  // the previous grid's writes (A, B, C, workspace, counters) are done
    griddep_launch_dependents();
    const int num_kb = p.num_kb;

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool failed = false;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            SegmentWalker walk(p.tiles_n, num_kb, p.shares);
            Segment sg;
            while (!failed && walk.next(sg)) {
                if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * MS);
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, p.timeout_ns)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    // MMA A = the B^T tile (N on the MMA's rows), MMA B = the A tile.
                    const uint32_t bt_base = smem_u32(sBt + stage * Cfg::kBtStageBytes);
                    const uint32_t a_base = smem_u32(sA + stage * Cfg::kAStageBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc_mma_f16(d_tmem, operand_desc<B_MN>(bt_base, k),
                                   operand_desc<false>(a_base, k), idesc,
                                   (kb != sg.kb0 || k != 0) ? 1u : 0u);
                    tc_commit(smem_u32(&empty[stage]));
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (failed) break;
                tc_commit(smem_u32(&tfull[acc]));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (failed) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
                const volatile int never = 0;
                tc_commit(smem_u32(drain));
                mbar_wait(smem_u32(drain), 0u, &never, 100000000ull);
            }
        }
        __syncwarp();
    } else if (warp <= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;
        const int r = q * 32 + lane;            // row of the transposed tile = column of C
        const int et = threadIdx.x - 32;        // 0..127
        const int64_t T = int64_t(p.tiles_n) * num_kb;
        int acc = 0;
        uint32_t acc_phase = 0;
        SegmentWalker walk(p.tiles_n, num_kb, p.shares);
        Segment sg;
        while (walk.next(sg)) {
            const bool ok =
                mbar_wait(smem_u32(&tfull[acc]), acc_phase, abort_flag, p.timeout_ns);
            // One decision for all 128 epilogue threads: they share named barriers below.
            if (!named_bar_and(1, 128, ok)) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
                break;
            }
            tc_fence_after();
            float v[MS];
            load_acc<MS>(tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                             static_cast<uint32_t>(acc * MS),
                         v);
            tc_fence_before();
            mbar_arrive(smem_u32(&tempty[acc]));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }

            const int n = sg.tile * 128 + r;
            if (sg.kb0 == 0 && sg.kb1 == num_kb) {
                // This share covers the whole tile: store C directly.
                if (n < p.N) {
#pragma unroll
                    for (int m = 0; m < MS; ++m)
                        if (m < p.M) store_c1(p, m, n, v[m]);
                }
                continue;
            }
            // Partial tile: publish it in this share's slot, then let the last arriver reduce.
            const int64_t first = share_of(int64_t(sg.tile) * num_kb, T, p.shares);
            const int64_t last = share_of(int64_t(sg.tile + 1) * num_kb - 1, T, p.shares);
            const int nslots = static_cast<int>(last - first + 1);
            const int slot = static_cast<int>(walk.share - first);
            // A checked build tests the tile's slots and counter first: the same
            // answer on every epilogue thread, so all of them skip the tile together
            // (its C is then not written).
            if (!DG_CHECK(p.status, kChkWs,
                          nslots <= p.max_slots &&
                              span_inside(0, static_cast<int64_t>(sg.tile) * p.max_slots * (MS * 128),
                                          static_cast<int64_t>(nslots) * (MS * 128), 1, p.ws_len)) ||
                !DG_CHECK(p.status, kChkCounter, span_inside(0, sg.tile, 1, 1, p.counters_len)))
                continue;
            float* tile_ws = p.ws + static_cast<int64_t>(sg.tile) * p.max_slots * (MS * 128);
            float* mine = tile_ws + static_cast<int64_t>(slot) * (MS * 128) + r;
#pragma unroll
            for (int m = 0; m < MS; ++m) __stcg(mine + m * 128, v[m]);
            // The barrier orders every epilogue thread's partial stores before thread 0's
            // release at GPU scope; its acquire half (and the second barrier) make the
            // partials of the shares that arrived earlier visible to the whole CTA.
            named_bar_sync(1, 128);
            if (et == 0) {
                const int old = atomic_add_acq_rel_gpu(&p.counters[sg.tile], 1);
                *last_flag = (old == nslots - 1) ? 1 : 0;
            }
            named_bar_sync(1, 128);
            if (*last_flag) {
                // Sum the slots in order 0, 1, ...; the loads of kBatch slots are issued
                // together so the reduction pays one L2 round trip per batch.
                constexpr int kBatch = MS <= 16 ? 4 : (MS == 32 ? 2 : 1);
                float s[MS];
#pragma unroll
                for (int m = 0; m < MS; ++m) s[m] = 0.0f;
                for (int j0 = 0; j0 < nslots; j0 += kBatch) {
                    float t[kBatch][MS];
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) {
                        const int j = j0 + b;
                        if (j < nslots && j != slot) {
                            const float* src =
                                tile_ws + static_cast<int64_t>(j) * (MS * 128) + r;
#pragma unroll
                            for (int m = 0; m < MS; ++m) t[b][m] = __ldcg(src + m * 128);
                        }
                    }
#pragma unroll
                    for (int b = 0; b < kBatch; ++b) {
                        const int j = j0 + b;
                        if (j < nslots) {
#pragma unroll
                            for (int m = 0; m < MS; ++m) s[m] += (j == slot) ? v[m] : t[b][m];
                        }
                    }
                }
                if (n < p.N) {
#pragma unroll
                    for (int m = 0; m < MS; ++m)
                        if (m < p.M) store_c1(p, m, n, s[m]);
                }
                if (et == 0) store_relaxed_gpu(&p.counters[sg.tile], 0);
            }
        }
    } else {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            bool failed = false;
            int stage = 0;
            uint32_t phase = 0;
            int64_t armed = 0;
            const uint64_t pol_stream = l2_policy_evict_first();   // B: read once
            const uint64_t pol_keep = l2_policy_evict_last();      // A: read by every tile
            SegmentWalker walk(p.tiles_n, num_kb, p.shares);
            Segment sg;
            while (!failed && walk.next(sg)) {
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                   p.timeout_ns)) {
                        failed = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(Cfg::kStageBytes));
                    load_operand_hint<B_MN>(smem_u32(sBt + stage * Cfg::kBtStageBytes), &mapB,
                                            fb, sg.tile * 128, kb * kBK, 128, pol_stream);
                    tma_load_2d_hint(smem_u32(sA + stage * Cfg::kAStageBytes), &mapA, fb,
                                     kb * kBK, 0, pol_keep);
                    ++armed;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (failed) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
                const volatile int never = 0;
                const int64_t rounds = armed / STAGES;
                for (int s = 0; s < STAGES; ++s) {
                    uint32_t parity;
                    if (s < stage) {
                        parity = phase;
                    } else if (rounds >= 1) {
                        parity = phase ^ 1u;
                    } else {
                        continue;
                    }
                    mbar_wait(smem_u32(&full[s]), parity, &never, 50000000ull);
                }
            }
        }
        __syncwarp();
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

namespace {
constexpr int kStages16 = 12;
constexpr int kStages32 = 10;
constexpr int kStages64 = 8;

template <int MS, int STAGES>
cudaError_t set_attrs() {
    cudaError_t e = cudaFuncSetAttribute(gemm_skinny_kernel<MS, STAGES, true>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         SkCfg<MS, STAGES>::kSmemBytes);
    if (e != cudaSuccess) return e;
    return cudaFuncSetAttribute(gemm_skinny_kernel<MS, STAGES, false>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SkCfg<MS, STAGES>::kSmemBytes);
}

template <int MS, int STAGES>
cudaError_t launch(bool b_mn, const CUtensorMap& b, const CUtensorMap& a, const Params& p,
                   uint32_t idesc, int grid, cudaStream_t s) {
    using Cfg = SkCfg<MS, STAGES>;
    if (b_mn)
        return launch_pdl(gemm_skinny_kernel<MS, STAGES, true>, dim3(grid), dim3(Cfg::kThreads),
                          Cfg::kSmemBytes, s, b, a, p, idesc);
    return launch_pdl(gemm_skinny_kernel<MS, STAGES, false>, dim3(grid), dim3(Cfg::kThreads),
                      Cfg::kSmemBytes, s, b, a, p, idesc);
}
}  // namespace

int skinny_smem_bytes(int ms) {
    if (ms == 16) return SkCfg<16, kStages16>::kSmemBytes;
    if (ms == 32) return SkCfg<32, kStages32>::kSmemBytes;
    return SkCfg<64, kStages64>::kSmemBytes;
}

int skinny_stages(int ms) { return ms == 16 ? kStages16 : (ms == 32 ? kStages32 : kStages64); }

cudaError_t skinny_prepare() {
    cudaError_t e = set_attrs<16, kStages16>();
    if (e == cudaSuccess) e = set_attrs<32, kStages32>();
    if (e == cudaSuccess) e = set_attrs<64, kStages64>();
    return e;
}

cudaError_t launch_skinny(int ms, bool b_mn, const CUtensorMap& mapB, const CUtensorMap& mapA,
                          const Params& p, uint32_t idesc, int grid, cudaStream_t stream) {
    if (ms == 16) return launch<16, kStages16>(b_mn, mapB, mapA, p, idesc, grid, stream);
    if (ms == 32) return launch<32, kStages32>(b_mn, mapB, mapA, p, idesc, grid, stream);
    return launch<64, kStages64>(b_mn, mapB, mapA, p, idesc, grid, stream);
}

}  // namespace dg
