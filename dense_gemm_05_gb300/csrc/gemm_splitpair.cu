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
// When both halves are summed, each CTA keeps one half of the strip's columns.
// After the K loop its operand ring is idle, so each CTA writes the other half
// of its fp32 partial there ([4 columns][row] float4s, 512 contiguous bytes
// per warp store) and one thread sends it to the peer with a single bulk
// shared-to-shared copy (cp.async.bulk.shared::cluster), which completes on the
// peer's barrier.  (Per-thread remote stores of the same 32 KiB took 2.3 us
// per launch; the bulk copy runs at the copy engine's rate.)  Each CTA then adds
// the peer's half of its own columns to its own partial (a + b: one rounding,
// the same bits whichever CTA adds) and stores C through the chunk epilogue of
// tiles.cuh: tensor-memory-access stores where C allows them, otherwise
// 16-byte stores wherever a row's alignment allows.  No workspace, counter or
// second pass.  A bounded wait that runs out claims the receiving CTA's
// exchange slot (a compare-and-swap the sender also makes before it sends), so
// a copy is never in flight into a CTA that has left.
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

// B read in place (B_GEN): raw-row stages of bulk copies in flight per loader warp.
constexpr int kSplitPairRawStages = 3;

template <int MS, int BN, int STAGES, int RAW = 0>
struct SplitPairCfg {
    static constexpr int kAStageBytes = MS * kBK * 2;       // A tile: MS rows x 64 k, K-major
    static constexpr int kBStageBytes = BN * kBK * 2;       // B tile: BN n x 64 k
    static constexpr int kHalf = BN / 2;                    // columns kept by each CTA
    static constexpr int kXBytes = MS * kHalf * 4;          // one half of the fp32 partial
    static constexpr int kRingBytes = STAGES * (kAStageBytes + kBStageBytes);
    // After the K loop the operand ring is free: it holds the half sent to the
    // peer, then (from a 1 KiB boundary) the epilogue warps' chunk buffers.
    static constexpr int kEpiOffset = (kXBytes + 1023) / 1024 * 1024;
    static constexpr int kTmemCols = 256;
    static constexpr int kThreads = 192;
    static constexpr int kEpiWarps = (MS + 31) / 32;        // epilogue warps holding rows
    // B read in place: RAW stages of raw rows (kRawStageBytes each), one barrier
    // per stage and loader warp.
    static constexpr int kRawBytes = RAW * kRawStageBytes;
    static constexpr int kNumBars = 2 * STAGES + 3 + 4 * RAW;
    static constexpr int kSmemBytes =
        1024 + kRingBytes + kXBytes + kRawBytes + 8 * kNumBars + 16;
    static_assert(MS == 16 || MS == 32 || MS == 64 || MS == 128, "MS");
    static_assert(BN % 64 == 0 && BN >= 128 && BN <= 256, "BN");
    // The MMA reads a 128-row (16 KiB) A window from each A stage; the B ring
    // behind the A stages keeps the last window inside the allocation.
    static_assert(STAGES * kBStageBytes >= kBM * kBK * 2, "A window");
    static_assert(kAStageBytes % 1024 == 0 && kBStageBytes % 1024 == 0, "swizzle atoms");
    static_assert(kEpiOffset + kEpiSmemBytes <= kRingBytes, "epilogue buffers fit the ring");
    static_assert(kXBytes % 16 == 0, "bulk copy size");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// B_GEN: B (stored K x N) is not 16-byte aligned and is read in place by the
// four epilogue warps with ordinary loads while the K loop runs (the
// unaligned-rows loader of tiles.cuh); A still comes by TMA.  Only with 128-row
// tiles of 128 columns.
template <int MS, int BN, int STAGES, bool B_MN, bool B_GEN>
__global__ void __cluster_dims__(2, 1, 1) __launch_bounds__(192, 1)
    gemm_splitpair_kernel(const __grid_constant__ CUtensorMap mapA,
                          const __grid_constant__ CUtensorMap mapB,
                          const __grid_constant__ CUtensorMap mapC, const Params p,
                          const uint32_t idesc) {
    constexpr int RAW = B_GEN ? kSplitPairRawStages : 0;
    using Cfg = SplitPairCfg<MS, BN, STAGES, RAW>;
    static_assert(!B_GEN || (MS == 128 && BN == 128 && B_MN), "in-place B loads: 128 x 128 tiles");
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;                                       // STAGES packed A tiles
    uint8_t* sB = sA + STAGES * Cfg::kAStageBytes;
    float4* sX = reinterpret_cast<float4*>(sB + STAGES * Cfg::kBStageBytes);   // peer's half
    uint8_t* sRaw = reinterpret_cast<uint8_t*>(sX) + Cfg::kXBytes;             // B_GEN raw rows
    uint64_t* bars = reinterpret_cast<uint64_t*>(sRaw + Cfg::kRawBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* xfull = tfull + 1;     // the peer's half has landed in sX
    uint64_t* drain = xfull + 1;
    uint64_t* rawfull = drain + 1;   // [RAW][4]: raw rows of a stage landed, per loader warp
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(rawfull + 4 * RAW);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    int* xstate = const_cast<int*>(abort_flag) + 1;   // 0, then 1 = peer sends, 2 = gave up
    float4* sSend = reinterpret_cast<float4*>(smem);  // the ring, once the K loop is done

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
            // B_GEN: the producer's TMA arrival for A plus the 128 loader threads for B
            mbar_init(smem_u32(&full[s]), B_GEN ? 129u : 1u);
            mbar_init(smem_u32(&empty[s]), 1u);
        }
        mbar_init(smem_u32(tfull), 1u);
        mbar_init(smem_u32(xfull), 1u);
        mbar_init(smem_u32(drain), 1u);
        for (int i = 0; i < 4 * RAW; ++i) mbar_init(smem_u32(&rawfull[i]), 32u);   // a warp's lanes
        *abort_flag = 0;
        *xstate = 0;
        // The peer's bulk copy of its half completes on xfull.
        mbar_arrive_expect_tx(smem_u32(xfull), static_cast<uint32_t>(Cfg::kXBytes));
        fence_mbar_init();
    }
    if (warp == 5 && lane == 0) {
        prefetch_tmap(&mapA);
        if (!B_GEN) prefetch_tmap(&mapB);
        if (p.c_tma) prefetch_tmap(&mapC);
    }
    __syncthreads();
    // Released here, waited for (by every thread) before the first remote access
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
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
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
        griddep_wait();                               // C (and B) may still be used by the previous grid
        cluster_wait_acquire();                       // the peer's barriers exist
        if constexpr (B_GEN) {
            // ---------------------------------------------------- B loader (K loop)
            // Warp w4 copies its 16 rows of each stage into the raw ring (RAW
            // stages ahead of the MMA), then moves them into the swizzled B stage.
            const int w4 = warp - 1;
            const uint32_t raw0 = smem_u32(sRaw);
            int stage = 0;
            uint32_t phase = 0;
            int issued = 0, placed = 0;       // stages of this CTA's K half
            const int nkb = kb1 - kb0;
            auto issue = [&](int j) {         // j-th stage of the half into raw slot j % RAW
                const int slot = j % RAW;
                unaligned_rows_issue(raw0 + static_cast<uint32_t>(slot * kRawStageBytes),
                                     smem_u32(&rawfull[slot * 4 + w4]), p.B, p.ldb, n0,
                                     (kb0 + j) * kBK, p.N, p.K, w4, lane, p.status, kChkB);
            };
            for (; issued < RAW && issued < nkb; ++issued) issue(issued);
            bool failed = false;
#pragma unroll 1
            for (; placed < nkb; ++placed) {
                const int slot = placed % RAW;
                const uint32_t rphase = static_cast<uint32_t>(placed / RAW) & 1u;
                bool ok = mbar_wait(smem_u32(&rawfull[slot * 4 + w4]), rphase, abort_flag,
                                    p.timeout_ns);
                ok = ok && mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p.timeout_ns);
                if (!__all_sync(0xffffffffu, ok)) {
                    failed = true;
                    break;
                }
                unaligned_rows_place(smem_u32(sB + stage * Cfg::kBStageBytes),
                                     raw0 + static_cast<uint32_t>(slot * kRawStageBytes), p.B, p.ldb,
                                     n0, (kb0 + placed) * kBK, p.N, p.K, w4, lane, p.status,
                                     kChkB);
                // generic stores -> the MMA's operand reads; generic reads of the raw
                // slot -> the next bulk copy into it
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&full[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
                __syncwarp();
                if (issued < nkb) issue(issued++);
            }
            if (failed) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
                // Bulk copies already issued must land before the shared memory goes away.
                const volatile int never = 0;
                for (int j = placed; j < issued; ++j)
                    mbar_wait(smem_u32(&rawfull[(j % RAW) * 4 + w4]),
                              static_cast<uint32_t>(j / RAW) & 1u, &never, 50000000ull);
            }
        }
        const int q = warp & 3;                       // TMEM lane quadrant of this warp
        if (q * 32 < MS) {
            const int r = q * 32 + lane;              // row of the tile (TMEM lane)
            const uint32_t trow = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
            bool ok = mbar_wait(smem_u32(tfull), 0u, abort_flag, p.timeout_ns);
            // tcgen05.ld is warp-collective: one decision per warp.
            ok = __all_sync(0xffffffffu, ok);
            // 1. The peer's half of the columns goes to the peer in one bulk copy
            // through this CTA's now idle operand ring, laid out [4 columns][row]
            // as float4 (a warp writes 512 contiguous bytes).  The producer warp,
            // idle once the K loop is issued, sends it (step 1b below), so that no
            // epilogue thread has a copy of its own in flight.
            if (ok) {
                tc_fence_after();
                fence_proxy_async_smem();   // the ring was last used by TMA and the MMAs
#pragma unroll 1
                for (int c = 0; c < Cfg::kHalf; c += 32) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(trow + peer * Cfg::kHalf + c, v);
                    tmem_ld_wait(v);
                    if (r < MS) {
#pragma unroll
                        for (int j = 0; j < 8; ++j)
                            sSend[(c / 4 + j) * MS + r] =
                                make_float4(__uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                            __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                    }
                }
                fence_proxy_async_smem();
            } else {
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
            }
            named_bar_arrive(4, 32 * Cfg::kEpiWarps + 32);
            // 2. The peer's half of this CTA's columns.  A wait that runs out claims
            // the exchange slot so that the peer sends nothing afterwards; if the
            // peer had already claimed it, its copy is on the way and is waited
            // for (with a long bound) before this CTA may leave.
            bool got = mbar_wait_cluster(smem_u32(xfull), 0u, abort_flag, p.timeout_ns);
            if (!got) {
                if (atom_cas_shared_cluster(smem_u32(xstate), 0, 2) == 1) {
                    const volatile int never = 0;
                    mbar_wait_cluster(smem_u32(xfull), 0u, &never, 100000000ull);
                }
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
            }
            // Nothing more arrives in this CTA's shared memory once the peer's copy
            // has landed, and this thread touches no other CTA's memory: the closing
            // arrival can go now, without release semantics.
            cluster_arrive_relaxed();
            arrived = true;
            got = __all_sync(0xffffffffu, got) && ok;
            // 3. This CTA's half: own partial + the peer's (a + b, one rounding, the
            // same bits whichever CTA adds), then C through the chunk epilogue
            // (tensor-memory-access stores where C allows them).
            const uint32_t ebuf =
                smem_u32(smem) + Cfg::kEpiOffset + static_cast<uint32_t>((warp - 1) * kEpiWarpBytes);
            uint32_t eseq = 0;
            const int col_base = n0 + static_cast<int>(rank) * Cfg::kHalf;
            const int row0 = m0 + q * 32;
            if (MS <= 64 && p.c_type == kOutF32 && p.c_vec) {
                // A strip of at most 64 rows with 16-byte-aligned fp32 C: each thread
                // writes its own row's sums straight to C (16-byte stores), which
                // measured faster here than staging 32-row chunks of which only the
                // strip's rows exist.  Every lane runs the (warp-collective) TMEM
                // loads; only the rows of the strip are stored.
                if (got) {
                    const int row = m0 + r;
                    const int rx = r < MS ? r : 0;
#pragma unroll 1
                    for (int c = 0; c < Cfg::kHalf; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(trow + rank * Cfg::kHalf + c, v);
                        tmem_ld_wait(v);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 x = sX[(c / 4 + j) * MS + rx];
                            v[4 * j] = __float_as_uint(__uint_as_float(v[4 * j]) + x.x);
                            v[4 * j + 1] = __float_as_uint(__uint_as_float(v[4 * j + 1]) + x.y);
                            v[4 * j + 2] = __float_as_uint(__uint_as_float(v[4 * j + 2]) + x.z);
                            v[4 * j + 3] = __float_as_uint(__uint_as_float(v[4 * j + 3]) + x.w);
                        }
                        if (r < MS && row < p.M) store_c32(p, row, col_base + c, v);
                    }
                }
            } else if (p.c_type == kOutF32 || Cfg::kHalf % 64 == 0) {
                if (got) {
                    const int cw = epi_chunk_cols(p.c_type);
#pragma unroll 1
                    for (int c = 0; c < Cfg::kHalf; c += cw) {
                        uint32_t lo[32], hi[32];
                        tmem_ld_32x32b_x32(trow + rank * Cfg::kHalf + c, lo);
                        if (cw == 64) tmem_ld_32x32b_x32(trow + rank * Cfg::kHalf + c + 32, hi);
                        tmem_ld_wait(lo);
                        if (cw == 64) tmem_ld_wait(hi);
                        const int rx = r < MS ? r : 0;   // rows beyond a short strip: masked at M
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            const float4 x = sX[(c / 4 + j) * MS + rx];
                            lo[4 * j] = __float_as_uint(__uint_as_float(lo[4 * j]) + x.x);
                            lo[4 * j + 1] = __float_as_uint(__uint_as_float(lo[4 * j + 1]) + x.y);
                            lo[4 * j + 2] = __float_as_uint(__uint_as_float(lo[4 * j + 2]) + x.z);
                            lo[4 * j + 3] = __float_as_uint(__uint_as_float(lo[4 * j + 3]) + x.w);
                        }
                        if (cw == 64) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                const float4 x = sX[(c / 4 + 8 + j) * MS + rx];
                                hi[4 * j] = __float_as_uint(__uint_as_float(hi[4 * j]) + x.x);
                                hi[4 * j + 1] = __float_as_uint(__uint_as_float(hi[4 * j + 1]) + x.y);
                                hi[4 * j + 2] = __float_as_uint(__uint_as_float(hi[4 * j + 2]) + x.z);
                                hi[4 * j + 3] = __float_as_uint(__uint_as_float(hi[4 * j + 3]) + x.w);
                            }
                        }
                        epi_store_chunk(p, &mapC, ebuf, eseq, lane, row0, col_base + c, lo, hi);
                    }
                    // The tensor-memory-access stores must have read their buffers
                    // before the shared memory goes away.
                    if (lane == 0 && p.c_tma) bulk_wait_group0();
                }
            } else {
                // 16-bit C with 96 columns per CTA (not whole 64-column chunks): the
                // sums go back into the exchange buffer and are written row by row.
                if (got) {
#pragma unroll 1
                    for (int c = 0; c < Cfg::kHalf; c += 32) {
                        uint32_t v[32];
                        tmem_ld_32x32b_x32(trow + rank * Cfg::kHalf + c, v);
                        tmem_ld_wait(v);
                        if (r < MS) {
#pragma unroll
                            for (int j = 0; j < 8; ++j) {
                                float4& x = sX[(c / 4 + j) * MS + r];
                                x.x += __uint_as_float(v[4 * j]);
                                x.y += __uint_as_float(v[4 * j + 1]);
                                x.z += __uint_as_float(v[4 * j + 2]);
                                x.w += __uint_as_float(v[4 * j + 3]);
                            }
                        }
                    }
                }
                // Every warp holding rows passes this barrier, whatever its waits gave.
                if (named_bar_and(3, 32 * Cfg::kEpiWarps, got)) {
                    const float* xs = reinterpret_cast<const float*>(sX);
                    for (int rr = q; rr < MS && m0 + rr < p.M; rr += Cfg::kEpiWarps) {
#pragma unroll 4
                        for (int cc = lane; cc < Cfg::kHalf; cc += 32) {
                            const int col = col_base + cc;
                            if (col < p.N)
                                store_c1(p, m0 + rr, col, xs[((cc >> 2) * MS + rr) * 4 + (cc & 3)]);
                        }
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
                if (!B_GEN) prefetch_operand_hint<B_MN>(&mapB, n0, kb * kBK, BN, pol_stream);
            }
            griddep_wait();                   // A and B may be written by the previous grid
            for (int kb = kb0; kb < kb1; ++kb) {
                if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p.timeout_ns)) {
                    failed = true;
                    break;
                }
                const uint32_t fb = smem_u32(&full[stage]);
                mbar_arrive_expect_tx(fb, static_cast<uint32_t>(B_GEN ? Cfg::kAStageBytes
                                                                      : Cfg::kAStageBytes +
                                                                            Cfg::kBStageBytes));
                tma_load_2d_hint(smem_u32(sA + stage * Cfg::kAStageBytes), &mapA, fb, kb * kBK, m0,
                                 pol_keep);
                if (!B_GEN)
                    load_operand_hint<B_MN>(smem_u32(sB + stage * Cfg::kBStageBytes), &mapB, fb,
                                            n0, kb * kBK, BN, pol_stream);
                ++armed;
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (failed) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
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
        cluster_wait_acquire();             // the peer's barriers exist
        // 1b. Once the epilogue warps holding rows have written the peer's half
        // (named barrier 4), claim the peer's exchange slot and send the half.
        // A peer that has given up (a bounded wait ran out) has claimed the slot
        // first, and then nothing is sent; nor is anything after a wait of this
        // CTA gave up (the abort flag).
        named_bar_sync(4, 32 * Cfg::kEpiWarps + 32);
        if (lane == 0) {
            if (*abort_flag == 0 &&
                atom_cas_shared_cluster(mapa_shared(smem_u32(xstate), peer), 0, 1) == 0) {
                bulk_copy_s2s_cluster(mapa_shared(smem_u32(sX), peer), smem_u32(sSend),
                                      static_cast<uint32_t>(Cfg::kXBytes),
                                      mapa_shared(smem_u32(xfull), peer));
            } else {
                *abort_flag = 1;
            }
        }
        __syncwarp();
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
    constexpr int fixed = 1024 + MS * (BN / 2) * 4 + 8 * 40 + 16;
    constexpr int s = (232448 - fixed) / per;
    return s > 8 ? 8 : s;
}

// B read in place: a shallower operand ring next to the raw rows.
constexpr int kSplitPairGenStages = 4;

template <int MS, int BN, bool B_GEN>
constexpr int stages_of() {
    return B_GEN ? kSplitPairGenStages : stages_for<MS, BN>();
}

template <int MS, int BN, bool B_GEN>
constexpr int smem_of() {
    return SplitPairCfg<MS, BN, stages_of<MS, BN, B_GEN>(), B_GEN ? kSplitPairRawStages : 0>::kSmemBytes;
}

template <int MS, int BN, bool B_MN, bool B_GEN = false>
cudaError_t set_attr_one() {
    constexpr int S = stages_of<MS, BN, B_GEN>();
    return cudaFuncSetAttribute(gemm_splitpair_kernel<MS, BN, S, B_MN, B_GEN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize,
                                smem_of<MS, BN, B_GEN>());
}

template <int MS, int BN>
cudaError_t set_attrs_bn() {
    cudaError_t e = set_attr_one<MS, BN, true>();
    if (e == cudaSuccess) e = set_attr_one<MS, BN, false>();
    if constexpr (MS == 128 && BN == 128) {
        if (e == cudaSuccess) e = set_attr_one<MS, BN, true, true>();
    }
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
cudaError_t launch_bn(bool b_mn, bool b_gen, const CUtensorMap& a, const CUtensorMap& b,
                      const CUtensorMap& c, const Params& p, uint32_t idesc, int grid,
                      cudaStream_t s) {
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
    if constexpr (MS == 128 && BN == 128) {
        if (b_gen) {
            constexpr int SG = stages_of<MS, BN, true>();
            cfg.dynamicSmemBytes = smem_of<MS, BN, true>();
            return cudaLaunchKernelEx(&cfg, gemm_splitpair_kernel<MS, BN, SG, true, true>, a, b, c,
                                      p, idesc);
        }
    }
    if (b_gen) return cudaErrorInvalidValue;
    if (b_mn)
        return cudaLaunchKernelEx(&cfg, gemm_splitpair_kernel<MS, BN, S, true, false>, a, b, c, p,
                                  idesc);
    return cudaLaunchKernelEx(&cfg, gemm_splitpair_kernel<MS, BN, S, false, false>, a, b, c, p,
                              idesc);
}

template <int MS>
cudaError_t launch_ms(int bn, bool b_mn, bool b_gen, const CUtensorMap& a, const CUtensorMap& b,
                      const CUtensorMap& c, const Params& p, uint32_t idesc, int grid,
                      cudaStream_t s) {
    if constexpr (MS == 128) {
        return launch_bn<MS, 128>(b_mn, b_gen, a, b, c, p, idesc, grid, s);
    } else {
        if (bn == 128) return launch_bn<MS, 128>(b_mn, b_gen, a, b, c, p, idesc, grid, s);
        if (bn == 192) return launch_bn<MS, 192>(b_mn, b_gen, a, b, c, p, idesc, grid, s);
        return launch_bn<MS, 256>(b_mn, b_gen, a, b, c, p, idesc, grid, s);
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
    if (cudaOccupancyMaxActiveClusters(&n, gemm_splitpair_kernel<MS, BN, S, true, false>, &cfg) !=
        cudaSuccess) {
        (void)cudaGetLastError();
        return 0;
    }
    return n;
}
}  // namespace

int splitpair_stages(int ms, int bn, bool b_gen) {
    if (b_gen) return kSplitPairGenStages;
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

cudaError_t launch_splitpair(int ms, int bn, bool b_mn, bool b_gen, const CUtensorMap& mapA,
                             const CUtensorMap& mapB, const CUtensorMap& mapC, const Params& p,
                             uint32_t idesc, int grid, cudaStream_t stream) {
    if (ms == 16) return launch_ms<16>(bn, b_mn, b_gen, mapA, mapB, mapC, p, idesc, grid, stream);
    if (ms == 32) return launch_ms<32>(bn, b_mn, b_gen, mapA, mapB, mapC, p, idesc, grid, stream);
    if (ms == 128)
        return launch_ms<128>(bn, b_mn, b_gen, mapA, mapB, mapC, p, idesc, grid, stream);
    return launch_ms<64>(bn, b_mn, b_gen, mapA, mapB, mapC, p, idesc, grid, stream);
}

}  // namespace dg
