// gemm_splitpair.cu -- GEMM for sm_103a whose output tiles are too few to
// occupy every SM: each tile's K loop is split over the two CTAs of a cluster,
// without a global split-K reduction.
//
// C[M, N] is cut into tiles of MS rows x BN columns (MS = 16, 32 or 64 for
// M <= 64: one strip of rows; MS = 128 otherwise, tile rows tm = 0, 1, ...);
// each tile is computed by a cluster of two CTAs, one per half of the K loop
// (the K-sum of "Writing GPU kernels in Triton", section 3.3, cut in two; exact
// up to rounding because the sum is associative).  N on the MMA's N side: the
// A tile (MS rows, zero-filled beyond M by the tensor-memory-access engine) is
// the MMA's A operand of 128 rows, and the B tile the MMA's B operand, so at
// small M one tcgen05.mma consumes BN x 16 elements of B -- the stream that
// bounds the problem -- and the tensor core stays far below the rate that the
// B stream needs (a swap-AB MMA with M = 16 as its N would move only 128 x 16
// elements of B per instruction).  With MS < 128, rows MS..127 of the 128-row
// A window hold whatever follows the A tile in shared memory; they only feed
// accumulator rows that are never read.
//
// When both halves are summed, each CTA keeps one half of the strip's columns:
// it sends the other half of its fp32 partial into the peer CTA's shared memory
// (distributed shared memory of the cluster), receives the peer's half of its
// own columns, adds the two (a + b: one rounding, the same bits whichever CTA
// adds) and stores C: with 16-byte stores of fp32 C each thread writes its row
// directly; otherwise (a C pitch that is not a 16-byte multiple, 16-bit C) the
// sums go back into the exchange buffer and C is written from it row by row,
// each warp store covering contiguous columns of one row (measured: the
// 1023 x 1000 x 1029 workload, whose C rows are not 16-byte aligned, 15.1 ->
// 13.4 us; with aligned fp32 rows the direct stores are faster).  No workspace,
// counter or second pass.
//
// Warp roles: warp 0 MMA issuer + TMEM owner, warps 1..4 epilogue (warp w reads
// TMEM lanes 32 (w % 4) ..; rows of C are lanes), warp 5 TMA producer.
//
// The kernel is short (about 20 us at M = 16, N = 14336, K = 4096), so its
// fixed costs are kept off the critical path: the producer issues its first
// loads right after the CTA's barriers exist (the cluster barrier that guards
// the remote arrive is waited for only by the epilogue, the TMEM address is
// handed over by a named barrier), and it is launched as a programmatic
// dependent of the previous kernel in the stream: its prologue overlaps that
// kernel's tail and every load waits for it to finish.  Before that wait, with
// one row of tiles, the producer prefetches its first K blocks into L2 (the
// host sets how many in Params::prefetch_kb; graph-replayed at M = 16, N =
// 14336: 20.8 -> 19.7 us).
#include "common.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace dg {

template <int MS, int BN, int STAGES>
struct SplitPairCfg {
    static constexpr int kAStageBytes = MS * kBK * 2;       // A tile: MS rows x 64 k, K-major
    static constexpr int kBStageBytes = BN * kBK * 2;       // B tile: BN n x 64 k
    static constexpr int kHalf = BN / 2;                    // columns kept by each CTA
    static constexpr int kXPitch = kHalf + 4;               // floats per exchange row (bank spread)
    static constexpr int kXBytes = MS * kXPitch * 4;
    static constexpr int kTmemCols = 256;
    static constexpr int kThreads = 192;
    static constexpr int kEpiWarps = (MS + 31) / 32;        // epilogue warps holding rows
    static constexpr int kNumBars = 2 * STAGES + 3;
    static constexpr int kSmemBytes =
        1024 + STAGES * (kAStageBytes + kBStageBytes) + kXBytes + 8 * kNumBars + 16;
    static_assert(MS == 16 || MS == 32 || MS == 64 || MS == 128, "MS");
    static_assert(BN % 64 == 0 && BN >= 128 && BN <= 256, "BN");
    // The MMA reads a 128-row (16 KiB) A window from each A stage; the B ring
    // behind the A stages keeps the last window inside the allocation.
    static_assert(STAGES * kBStageBytes >= kBM * kBK * 2, "A window");
    static_assert(kAStageBytes % 1024 == 0 && kBStageBytes % 1024 == 0, "swizzle atoms");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

template <int MS, int BN, int STAGES, bool B_MN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    gemm_splitpair_kernel(const __grid_constant__ CUtensorMap mapA,
                       const __grid_constant__ CUtensorMap mapB, const Params p,
                       const uint32_t idesc) {
    using Cfg = SplitPairCfg<MS, BN, STAGES>;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                                       // STAGES packed A tiles
    uint8_t* sB = sA + STAGES * Cfg::kAStageBytes;
    float* sX = reinterpret_cast<float*>(sB + STAGES * Cfg::kBStageBytes);   // peer's half
    uint64_t* bars = reinterpret_cast<uint64_t*>(reinterpret_cast<uint8_t*>(sX) + Cfg::kXBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* xfull = tfull + 1;     // the peer's MS rows have arrived in sX
    uint64_t* drain = xfull + 1;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    bool arrived = false;            // this thread's arrival on the closing cluster barrier
    const uint32_t rank = cluster_ctarank();
    const uint32_t peer = rank ^ 1u;
    const int tile = static_cast<int>(cluster_id_x());
    const int tm = tile / p.tiles_n;                 // 0 unless MS == 128
    const int n0 = (tile - tm * p.tiles_n) * BN;
    const int m0 = tm * kBM;
    const int num_kb = p.num_kb;
    const int kb_half = num_kb / 2;                  // num_kb >= 2: both halves non-empty
    const int kb0 = rank ? kb_half : 0;
    const int kb1 = rank ? num_kb : kb_half;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), 1u);
            mbar_init(smem_u32(&empty[s]), 1u);
        }
        mbar_init(smem_u32(tfull), 1u);
        mbar_init(smem_u32(xfull), static_cast<uint32_t>(MS));
        mbar_init(smem_u32(drain), 1u);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 5 && lane == 0) {
        prefetch_tmap(&mapA);
        prefetch_tmap(&mapB);
    }
    __syncthreads();
    // Released here, waited for (by every thread) before the first remote arrive
    // and before leaving: the peer's barriers are initialised when it is passed.
    cluster_arrive_release();
    griddep_launch_dependents();

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
        tc_fence_before();
        named_bar_sync(2, 160);          // TMEM address -> the epilogue warps
        tc_fence_after();
        const uint32_t tmem_base = *tmem_slot;
        if (lane == 0) {
            bool failed = false;
            int stage = 0;
            uint32_t phase = 0;
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, p.timeout_ns)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t a_base = smem_u32(sA + stage * Cfg::kAStageBytes);
                const uint32_t b_base = smem_u32(sB + stage * Cfg::kBStageBytes);
#pragma unroll
                for (int k = 0; k < kBK / 16; ++k)
                    tc_mma_f16(tmem_base, operand_desc<false>(a_base, k),
                               operand_desc<B_MN>(b_base, k), idesc,
                               (kb != kb0 || k != 0) ? 1u : 0u);
                tc_commit(smem_u32(&empty[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (!failed) {
                tc_commit(smem_u32(tfull));
            } else {
                *abort_flag = 1;
                if (p.status != nullptr) atomicExch(p.status, kDevTimeout);
                const volatile int never = 0;
                tc_commit(smem_u32(drain));
                mbar_wait(smem_u32(drain), 0u, &never, 100000000ull);
            }
        }
        __syncwarp();
        cluster_wait_acquire();
    } else if (warp <= 4) {
        // ------------------------------------------------------------ epilogue
        named_bar_sync(2, 160);
        tc_fence_after();
        const uint32_t tmem_base = *tmem_slot;
        griddep_wait();                               // C may still be read by the previous grid
        cluster_wait_acquire();                       // the peer's exchange barrier exists
        const int q = warp & 3;                       // TMEM lane quadrant of this warp
        const bool direct = p.c_type == kOutF32 && p.c_vec;   // the same in every thread
        if (q * 32 < MS) {
            const int r = q * 32 + lane;              // row of C (TMEM lane)
            bool ok = mbar_wait(smem_u32(tfull), 0u, abort_flag, p.timeout_ns);
            // tcgen05.ld is warp-collective: one decision per warp.
            ok = __all_sync(0xffffffffu, ok);
            if (ok) {
                tc_fence_after();
                const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
                // 1. The peer's half of the columns goes to the peer's exchange buffer.
                const uint32_t x_remote =
                    mapa_shared(smem_u32(sX) + static_cast<uint32_t>(r * Cfg::kXPitch * 4), peer);
#pragma unroll 1
                for (int c = 0; c < Cfg::kHalf; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(trow + peer * Cfg::kHalf + c, v);
                    tmem_ld_wait(v);
                    if (r < MS) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            st_cluster_v4_b32(x_remote + static_cast<uint32_t>((c + 4 * j) * 4),
                                              make_uint4(v[4 * j], v[4 * j + 1], v[4 * j + 2],
                                                         v[4 * j + 3]));
                    }
                }
                if (r < MS) mbar_arrive_cluster(mapa_shared(smem_u32(xfull), peer));
                // This thread touches the peer's shared memory no more: its arrival on
                // the closing cluster barrier can go now.
                cluster_arrive_release();
                arrived = true;
                // 2. This CTA's half: own partial + the peer's.  With 16-byte stores of
                // fp32 C each thread writes its own row straight away; otherwise the
                // sums go back into the exchange buffer and step 3 writes them out.
                const bool got = mbar_wait_cluster(smem_u32(xfull), 0u, abort_flag, p.timeout_ns);
                if (!got) {
                    *abort_flag = 1;
                    if (p.status != nullptr) atomicExch(p.status, kDevTimeout);
                }
                if (__all_sync(0xffffffffu, got) && direct) {
                    const float* xrow = sX + r * Cfg::kXPitch;
                    const int col_base = n0 + static_cast<int>(rank) * Cfg::kHalf;
                    const int row = m0 + r;
#pragma unroll 1
                    for (int c = 0; c < Cfg::kHalf; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(trow + rank * Cfg::kHalf + c, v);
                        tmem_ld_wait(v);
                        const int col = col_base + c;
                        if (r < MS && row < p.M && col < p.N) {
#pragma unroll
                            for (int j = 0; j < 32; ++j)
                                v[j] = __float_as_uint(__uint_as_float(v[j]) + xrow[c + j]);
                            store_c32(p, static_cast<int64_t>(row) * p.ldc + col, v, p.N - col);
                        }
                    }
                } else if (__all_sync(0xffffffffu, got)) {
                    float* xrow = sX + r * Cfg::kXPitch;
#pragma unroll 1
                    for (int c = 0; c < Cfg::kHalf; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(trow + rank * Cfg::kHalf + c, v);
                        tmem_ld_wait(v);
                        if (r < MS) {
#pragma unroll
                            for (int j = 0; j < 32; j += 4) {
                                float4* x4 = reinterpret_cast<float4*>(xrow + c + j);
                                float4 t = *x4;
                                t.x += __uint_as_float(v[j]);
                                t.y += __uint_as_float(v[j + 1]);
                                t.z += __uint_as_float(v[j + 2]);
                                t.w += __uint_as_float(v[j + 3]);
                                *x4 = t;
                            }
                        }
                    }
                }
            } else {
                *abort_flag = 1;
                if (p.status != nullptr) atomicExch(p.status, kDevTimeout);
            }
            // 3. (Not direct) C from the exchange buffer, row by row: every row of
            // this CTA's half is complete once all epilogue warps holding rows have
            // passed the barrier; each warp store covers contiguous columns of a row.
            if (!direct) named_bar_sync(3, 32 * Cfg::kEpiWarps);
            if (!direct && *abort_flag == 0) {
                const int col_base = n0 + static_cast<int>(rank) * Cfg::kHalf;
                for (int rr = q; rr < MS && m0 + rr < p.M; rr += Cfg::kEpiWarps) {
                    const float* xr = sX + rr * Cfg::kXPitch;
                    const int64_t off = static_cast<int64_t>(m0 + rr) * p.ldc;
#pragma unroll 4
                    for (int cc = lane; cc < Cfg::kHalf; cc += 32) {
                        const int col = col_base + cc;
                        if (col < p.N) store_c1(p, off + col, xr[cc]);
                    }
                }
            }
        }
    } else {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            bool failed = false;
            int stage = 0;
            uint32_t phase = 0;
            int armed = 0;
            const uint64_t pol_stream = l2_policy_evict_first();   // B: read once
            const uint64_t pol_keep = l2_policy_evict_last();      // A: read by every tile of its rows
            // While the previous grid finishes, warm L2 with this CTA's first K
            // blocks: a prefetch hands no data to this CTA, so it needs no wait,
            // and the first loads after the wait then find their lines in L2.
            for (int kb = kb0; kb < kb1 && kb < kb0 + p.prefetch_kb; ++kb) {
                tma_prefetch_2d_hint(&mapA, kb * kBK, m0, pol_keep);
                prefetch_operand_hint<B_MN>(&mapB, n0, kb * kBK, BN, pol_stream);
            }
            griddep_wait();                   // A and B may be written by the previous grid
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p.timeout_ns)) {
                    failed = true;
                    break;
                }
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(
                    fb, static_cast<uint32_t>(Cfg::kAStageBytes + Cfg::kBStageBytes));
                tma_load_2d_hint(smem_u32(sA + stage * Cfg::kAStageBytes), &mapA, fb, kb * kBK, m0,
                                 pol_keep);
                load_operand_hint<B_MN>(smem_u32(sB + stage * Cfg::kBStageBytes), &mapB, fb, n0,
                                        kb * kBK, BN, pol_stream);
                ++armed;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (failed) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicExch(p.status, kDevTimeout);
                // Copies already issued must land before the shared memory goes away.
                const volatile int never = 0;
                const int rounds = armed / STAGES;
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
        cluster_wait_acquire();
    }

    tc_fence_before();
    __syncthreads();
    // No CTA leaves while its peer may still write to its shared memory.
    if (!arrived) cluster_arrive_release();
    cluster_wait_acquire();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(*tmem_slot, Cfg::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

namespace {

// Ring depth per (MS, BN): as deep as fits next to the exchange buffer.
template <int MS, int BN>
constexpr int stages_for() {
    constexpr int per = MS * kBK * 2 + BN * kBK * 2;
    constexpr int fixed = 1024 + MS * (BN / 2 + 4) * 4 + 8 * 40 + 16;
    constexpr int s = (232448 - fixed) / per;
    return s > 8 ? 8 : s;
}

template <int MS, int BN, bool B_MN>
cudaError_t set_attr_one() {
    constexpr int S = stages_for<MS, BN>();
    return cudaFuncSetAttribute(gemm_splitpair_kernel<MS, BN, S, B_MN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                SplitPairCfg<MS, BN, S>::kSmemBytes);
}

template <int MS, int BN>
cudaError_t set_attrs_bn() {
    cudaError_t e = set_attr_one<MS, BN, true>();
    if (e == cudaSuccess) e = set_attr_one<MS, BN, false>();
    return e;
}

template <int MS>
cudaError_t set_attrs_ms() {
    cudaError_t e = set_attrs_bn<MS, 128>();
    if constexpr (MS != 128) {                       // 128-row tiles: 128 columns only
        if (e == cudaSuccess) e = set_attrs_bn<MS, 192>();
        if (e == cudaSuccess) e = set_attrs_bn<MS, 256>();
    }
    return e;
}

// Launched as a programmatic dependent of the previous work in the stream (the
// kernel waits for it before touching global memory).
template <int MS, int BN>
cudaError_t launch_bn(bool b_mn, const CUtensorMap& a, const CUtensorMap& b, const Params& p,
                      uint32_t idesc, int grid, cudaStream_t s) {
    constexpr int S = stages_for<MS, BN>();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.gridDim = dim3(static_cast<unsigned>(grid), 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = SplitPairCfg<MS, BN, S>::kSmemBytes;
    cfg.stream = s;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    if (b_mn) return cudaLaunchKernelEx(&cfg, gemm_splitpair_kernel<MS, BN, S, true>, a, b, p, idesc);
    return cudaLaunchKernelEx(&cfg, gemm_splitpair_kernel<MS, BN, S, false>, a, b, p, idesc);
}

template <int MS>
cudaError_t launch_ms(int bn, bool b_mn, const CUtensorMap& a, const CUtensorMap& b,
                      const Params& p, uint32_t idesc, int grid, cudaStream_t s) {
    if constexpr (MS == 128) {
        return launch_bn<MS, 128>(b_mn, a, b, p, idesc, grid, s);
    } else {
        if (bn == 128) return launch_bn<MS, 128>(b_mn, a, b, p, idesc, grid, s);
        if (bn == 192) return launch_bn<MS, 192>(b_mn, a, b, p, idesc, grid, s);
        return launch_bn<MS, 256>(b_mn, a, b, p, idesc, grid, s);
    }
}

template <int MS, int BN>
int max_clusters_one() {
    constexpr int S = stages_for<MS, BN>();
    cudaLaunchConfig_t cfg = {};
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2, 1, 1);
    cfg.blockDim = dim3(192, 1, 1);
    cfg.dynamicSmemBytes = SplitPairCfg<MS, BN, S>::kSmemBytes;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, gemm_splitpair_kernel<MS, BN, S, true>, &cfg) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}
}  // namespace

int splitpair_stages(int ms, int bn) {
    if (ms == 16) return bn == 128 ? stages_for<16, 128>() : (bn == 192 ? stages_for<16, 192>() : stages_for<16, 256>());
    if (ms == 32) return bn == 128 ? stages_for<32, 128>() : (bn == 192 ? stages_for<32, 192>() : stages_for<32, 256>());
    if (ms == 128) return stages_for<128, 128>();
    return bn == 128 ? stages_for<64, 128>() : (bn == 192 ? stages_for<64, 192>() : stages_for<64, 256>());
}

cudaError_t splitpair_prepare() {
    cudaError_t e = set_attrs_ms<16>();
    if (e == cudaSuccess) e = set_attrs_ms<32>();
    if (e == cudaSuccess) e = set_attrs_ms<64>();
    if (e == cudaSuccess) e = set_attrs_ms<128>();
    return e;
}

// All (MS, BN) instantiations hold one CTA per SM, so one query serves them.
int splitpair_max_clusters() { return max_clusters_one<64, 256>(); }

cudaError_t launch_splitpair(int ms, int bn, bool b_mn, const CUtensorMap& mapA,
                          const CUtensorMap& mapB, const Params& p, uint32_t idesc, int grid,
                          cudaStream_t stream) {
    if (ms == 16) return launch_ms<16>(bn, b_mn, mapA, mapB, p, idesc, grid, stream);
    if (ms == 32) return launch_ms<32>(bn, b_mn, mapA, mapB, p, idesc, grid, stream);
    if (ms == 128) return launch_ms<128>(bn, b_mn, mapA, mapB, p, idesc, grid, stream);
    return launch_ms<64>(bn, b_mn, mapA, mapB, p, idesc, grid, stream);
}

}  // namespace dg
