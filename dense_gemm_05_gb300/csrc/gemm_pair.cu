// gemm_pair.cu -- persistent tcgen05 GEMM on CTA pairs (cta_group::2), sm_103a.
//
// A cluster of two CTAs on two SMs computes a 256 x BN tile of C with one
// stream of pair MMAs (M = 256): CTA r loads rows [128 r, 128 r + 128) of the
// A tile and columns [r BN/2, (r+1) BN/2) of the B tile into its own shared
// memory, and holds rows [128 r, 128 r + 128) of the accumulator in its own
// TMEM.  Each SM therefore stages half as much B per flop as a one-CTA tile of
// the same width, which is what lets the tensor cores run closer to their
// peak.  No TMA multicast is used: every CTA reads only its own halves.
//
// Same K loop, masking and tile order as gemm_tc.cu ("Writing GPU kernels in
// Triton", sections 3.3 and 4.6; group-major order of "I Wrote a GPU Matmul
// Kernel From Scratch in Triton", Step 4), with pair tiles as the unit.
//
// Roles (both CTAs): warp 0 TMEM owner (and, in CTA 0 only, the MMA issuer),
// warps 1..4 epilogue, warp 5 TMA producer.  Barriers:
//   full[s]   (CTA 0)  one arrive.expect_tx by CTA 0's producer for the bytes
//                      of BOTH CTAs; both producers' TMA loads complete on it
//   empty[s]  (each)   one multicast tcgen05.commit from CTA 0's MMA issuer
//   tfull[a]  (each)   one multicast tcgen05.commit after a tile's last MMA
//   tempty[a] (CTA 0)  256 arrivals: the epilogue threads of both CTAs
#include "common.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace dg {

template <int BN, int STAGES>
struct PairCfg {
    static constexpr int kBHalf = BN / 2;                       // B columns per CTA
    static constexpr int kBStageBytes = kBHalf * kBK * 2;
    static constexpr int kStageBytes = kAStageBytes + kBStageBytes;   // per CTA
    static constexpr int kTmemCols = 2 * BN;                    // two 128 x BN fp32 accumulators
    static constexpr int kThreads = 192;
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr int kSmemBytes =
        1024 + STAGES * kStageBytes + kEpiSmemBytes + 8 * kNumBars + 16;
    static_assert(kBHalf % kSubN == 0, "B half must be whole 64-column sub-tiles");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

template <int BN, int STAGES, bool A_MN, bool B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    gemm_pair_kernel(const __grid_constant__ CUtensorMap mapA,
                     const __grid_constant__ CUtensorMap mapB,
                     const __grid_constant__ CUtensorMap mapC, const Params p,
                     const uint32_t idesc) {
    using Cfg = PairCfg<BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * kAStageBytes;
    uint8_t* sEpi = sB + STAGES * Cfg::kBStageBytes;      // 4 KiB per epilogue warp
    uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + kEpiSmemBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const uint32_t rank = cluster_ctarank();
    const bool leader = rank == 0;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1u);
            mbar_init(smem_u32(&empty[s]), 1u);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1u);
            mbar_init(smem_u32(&tempty[a]), 256u);
        }
        mbar_init(smem_u32(drain), 1u);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc_pair(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish_pair();
    }
    if (warp == 5 && lane == 0) {
        prefetch_tmap(&mapA);
        prefetch_tmap(&mapB);
        if (p.c_tma) prefetch_tmap(&mapC);
    }
    tc_fence_before();
    cluster_sync();      // both CTAs' barriers initialised and TMEM allocated
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;

    const int total = p.tiles_m * p.tiles_n;
    const int num_kb = p.num_kb;
    const int cid = static_cast<int>(cluster_id_x());
    const int ncl = static_cast<int>(nclusters_x());

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer (CTA 0)
        if (leader && lane == 0) {
            bool failed = false;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int t = cid; t < total && !failed; t += ncl) {
                if (!mbar_wait_cluster(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag,
                                       p.timeout_ns)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, p.timeout_ns)) {
                        failed = true;
                        break;
                    }
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + stage * kAStageBytes);
                    const uint32_t b_base = smem_u32(sB + stage * Cfg::kBStageBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc_mma_f16_pair(d_tmem, operand_desc<A_MN>(a_base, k),
                                        operand_desc<B_MN>(b_base, k), idesc,
                                        (kb | k) != 0 ? 1u : 0u);
                    tc_commit_pair_mc(smem_u32(&empty[stage]), 0x3);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
                if (failed) break;
                tc_commit_pair_mc(smem_u32(&tfull[acc]), 0x3);
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1u;
                }
            }
            if (failed) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicExch(p.status, kDevTimeout);
                const volatile int never = 0;
                tc_commit_pair_mc(smem_u32(drain), 0x1);
                mbar_wait(smem_u32(drain), 0u, &never, 100000000ull);
            }
        }
        __syncwarp();
    } else if (warp <= 4) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int row_in_tile = static_cast<int>(rank) * 128 + q * 32 + lane;
        const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
        const uint32_t tempty1 = mapa_shared(smem_u32(&tempty[1]), 0);
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = cid; t < total; t += ncl) {
            int tm, tn;
            tile_coord32(t, p.tiles_m, p.tiles_n, p.group, tm, tn);
            const bool ok =
                mbar_wait(smem_u32(&tfull[acc]), acc_phase, abort_flag, p.timeout_ns);
            if (!__all_sync(0xffffffffu, ok)) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicExch(p.status, kDevTimeout);
                break;
            }
            tc_fence_after();
            const int row = tm * 256 + row_in_tile;
            const int col0 = tn * BN;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            const uint32_t tempty_peer0 = acc == 0 ? tempty0 : tempty1;
            if (p.c_tma) {
                epilogue_tma<BN>(p, &mapC, smem_u32(sEpi) + (warp - 1) * kEpiBufBytes, taddr, lane,
                                 row - lane, col0, [&] {
                                     tc_fence_before();
                                     mbar_arrive_cluster(tempty_peer0);
                                 });
            } else {
                const int64_t row_off = static_cast<int64_t>(row) * p.ldc + col0;
                const bool row_ok = row < p.M;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c * 32), v);
                    tmem_ld_wait(v);
                    if (c == BN / 32 - 1) {
                        tc_fence_before();
                        mbar_arrive_cluster(tempty_peer0);
                    }
                    if (row_ok) store_c32(p, row_off + c * 32, v, p.N - (col0 + c * 32));
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    } else {
        // ------------------------------------------------------------ TMA producer (both CTAs)
        if (lane == 0) {
            bool failed = false;
            int stage = 0;
            uint32_t phase = 0;
            for (int t = cid; t < total && !failed; t += ncl) {
                int tm, tn;
                tile_coord32(t, p.tiles_m, p.tiles_n, p.group, tm, tn);
                const int a_row = tm * 256 + static_cast<int>(rank) * 128;
                const int b_col = tn * BN + static_cast<int>(rank) * Cfg::kBHalf;
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                   p.timeout_ns)) {
                        failed = true;
                        break;
                    }
                    const uint32_t fb_local = smem_u32(&full[stage]);
                    const uint32_t fb = mapa_shared(fb_local, 0);   // CTA 0's full[stage]
                    if (leader) mbar_arrive_expect_tx(fb_local, 2u * Cfg::kStageBytes);
                    load_operand_pair<A_MN>(smem_u32(sA + stage * kAStageBytes), &mapA, fb, a_row,
                                            kb * kBK, kBM);
                    load_operand_pair<B_MN>(smem_u32(sB + stage * Cfg::kBStageBytes), &mapB, fb,
                                            b_col, kb * kBK, Cfg::kBHalf);
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (!failed) {
                // Every stage must be handed back (the last multicast commits have landed
                // in this CTA) before the pair may exit.
                for (int i = 0; i < STAGES; ++i) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                   p.timeout_ns)) {
                        failed = true;
                        break;
                    }
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (failed) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicExch(p.status, kDevTimeout);
                // Copies already issued complete on CTA 0's barriers, which this CTA
                // cannot observe: give them a bounded 2 ms to land before leaving.
                const uint64_t t0 = global_timer_ns();
                while (global_timer_ns() - t0 < 2000000ull) {
                }
            }
        }
        __syncwarp();
    }

    // The TMA stores of C must have completed before the CTA's shared memory goes away.
    if (warp >= 1 && warp <= 4 && lane == 0 && p.c_tma) bulk_wait_group0();
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // neither CTA leaves while its peer may still signal it
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc_pair(tmem_base, Cfg::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

namespace {
constexpr int kPairStages256 = 6;
constexpr int kPairStages128 = 8;

template <int BN, int STAGES, bool A_MN, bool B_MN>
cudaError_t set_attrs_one() {
    return cudaFuncSetAttribute(gemm_pair_kernel<BN, STAGES, A_MN, B_MN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                PairCfg<BN, STAGES>::kSmemBytes);
}

template <int BN, int STAGES>
cudaError_t set_attrs() {
    cudaError_t e = set_attrs_one<BN, STAGES, false, true>();
    if (e == cudaSuccess) e = set_attrs_one<BN, STAGES, false, false>();
    if (e == cudaSuccess) e = set_attrs_one<BN, STAGES, true, true>();
    if (e == cudaSuccess) e = set_attrs_one<BN, STAGES, true, false>();
    return e;
}

template <int BN, int STAGES, bool A_MN, bool B_MN>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                       const Params& p, uint32_t idesc, int grid, cudaStream_t s) {
    gemm_pair_kernel<BN, STAGES, A_MN, B_MN>
        <<<grid, PairCfg<BN, STAGES>::kThreads, PairCfg<BN, STAGES>::kSmemBytes, s>>>(a, b, c, p,
                                                                                   idesc);
    return cudaGetLastError();
}

template <int BN, int STAGES>
cudaError_t launch(bool a_mn, bool b_mn, const CUtensorMap& a, const CUtensorMap& b,
                   const CUtensorMap& c, const Params& p, uint32_t idesc, int grid,
                   cudaStream_t s) {
    if (!a_mn && b_mn) return launch_one<BN, STAGES, false, true>(a, b, c, p, idesc, grid, s);
    if (!a_mn && !b_mn) return launch_one<BN, STAGES, false, false>(a, b, c, p, idesc, grid, s);
    if (a_mn && b_mn) return launch_one<BN, STAGES, true, true>(a, b, c, p, idesc, grid, s);
    return launch_one<BN, STAGES, true, false>(a, b, c, p, idesc, grid, s);
}

// All four layout instantiations have the same resources, so one query serves them.
template <int BN, int STAGES>
int max_clusters() {
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(PairCfg<BN, STAGES>::kThreads, 1, 1);
    cfg.dynamicSmemBytes = PairCfg<BN, STAGES>::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_pair_kernel<BN, STAGES, false, true>, &cfg) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}
}  // namespace

int pair_smem_bytes(int bn) {
    return bn == 256 ? PairCfg<256, kPairStages256>::kSmemBytes
                     : PairCfg<128, kPairStages128>::kSmemBytes;
}

int pair_stages(int bn) { return bn == 256 ? kPairStages256 : kPairStages128; }

cudaError_t pair_prepare() {
    cudaError_t e = set_attrs<256, kPairStages256>();
    if (e == cudaSuccess) e = set_attrs<128, kPairStages128>();
    return e;
}

int pair_max_clusters(int bn) {
    return bn == 256 ? max_clusters<256, kPairStages256>() : max_clusters<128, kPairStages128>();
}

cudaError_t launch_pair(int bn, bool a_mn, bool b_mn, const CUtensorMap& mapA,
                        const CUtensorMap& mapB, const CUtensorMap& mapC, const Params& p,
                        uint32_t idesc, int grid, cudaStream_t stream) {
    if (bn == 256)
        return launch<256, kPairStages256>(a_mn, b_mn, mapA, mapB, mapC, p, idesc, grid, stream);
    return launch<128, kPairStages128>(a_mn, b_mn, mapA, mapB, mapC, p, idesc, grid, stream);
}

}  // namespace dg
