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
    static constexpr int kNumBars = 2 * STAGES + 6;
    static constexpr int kSmemBytes =
        1024 + STAGES * kStageBytes + kEpiSmemBytes + 8 * kNumBars + 32;
    static_assert(kBHalf % kSubN == 0, "B half must be whole 64-column sub-tiles");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

// The work of one cluster, in order: its stream-K share of the tiles
// [0, sk_tiles) -- one contiguous run of the (tile, K block) iterations of
// those tiles, cut into per-tile segments -- and the whole tiles
// sk_tiles + cid, sk_tiles + cid + clusters, ...; the share comes first, or
// after the first whole tile when the cluster has at least two.  Keeping the
// split tiles before most whole tiles lets their fix-ups (run by the epilogue
// warps) overlap the MMAs of the whole tiles that follow.
struct PairSeg {
    int tile;
    int kb0, kb1;     // K blocks [kb0, kb1) of the tile
    int share;        // stream-K share, or -1 for a whole data-parallel tile
};

struct PairWalker {
    int num_kb, ncl, total, next_dp, share;
    bool dp_first;       // one whole tile still to be walked before the stream-K share
    int64_t t_sk, g, it, end;

    __device__ PairWalker(const Params& p, int cid, int nclusters)
        : num_kb(p.num_kb), ncl(nclusters), total(p.tiles_m * p.tiles_n), share(cid) {
        const int sk = p.shares > 0 ? p.sk_tiles : 0;
        // With at least two whole tiles per cluster, the first whole tile runs
        // before the stream-K share: the share then reads operands the first
        // wave has brought into L2 (a cold share streamed at about 0.5 us per K
        // block against 0.3), and its fix-up still overlaps later whole tiles.
        dp_first = sk > 0 && total - sk >= 2 * nclusters;
        t_sk = int64_t(sk) * num_kb;
        g = p.shares;
        if (sk > 0 && cid < g) {
            it = share_begin(cid, t_sk, g);
            end = share_begin(cid + 1, t_sk, g);
        } else {
            it = end = 0;
        }
        next_dp = sk + cid;
    }
    __device__ bool next(PairSeg& s) {
        if (dp_first) {
            dp_first = false;
            if (next_dp < total) {
                s.tile = next_dp;
                s.kb0 = 0;
                s.kb1 = num_kb;
                s.share = -1;
                next_dp += ncl;
                return true;
            }
        }
        if (it < end) {
            s.tile = static_cast<int>(it / num_kb);
            s.kb0 = static_cast<int>(it - int64_t(s.tile) * num_kb);
            const int64_t left = end - it;
            s.kb1 = (num_kb - s.kb0 < left) ? num_kb : s.kb0 + static_cast<int>(left);
            s.share = share;
            it += s.kb1 - s.kb0;
            return true;
        }
        if (next_dp < total) {
            s.tile = next_dp;
            s.kb0 = 0;
            s.kb1 = num_kb;
            s.share = -1;
            next_dp += ncl;
            return true;
        }
        return false;
    }
    // Partial-tile slot of share `sh` for `tile`: 0 if the share begins inside the
    // tile, 1 if it ends inside it (a share holds at most these two partial tiles).
    __device__ int slot_of(int64_t sh, int tile) const {
        return share_begin(sh, t_sk, g) / num_kb == tile ? 0 : 1;
    }
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
    uint64_t* final_bar = drain + 1;   // after an abort: the last multicast commit of CTA 0
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(final_bar + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
    volatile int* last_flag = abort_flag + 1;   // "this CTA sums a stream-K tile"
    volatile int* n_issued = last_flag + 1;     // K-block stages this CTA's producer issued
    volatile int* n_consumed = n_issued + 1;    // CTA 0: stages whose full barrier the MMA passed

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
        mbar_init(smem_u32(final_bar), 1u);
        *abort_flag = 0;
        *last_flag = 0;
        *n_issued = 0;
        *n_consumed = 0;
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
    griddep_wait();      // the previous grid's writes (A, B, C, workspace, counters) are done
    griddep_launch_dependents();

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
            int consumed = 0;
            PairWalker walk(p, cid, ncl);
            PairSeg sg;
            while (!failed && walk.next(sg)) {
                if (!mbar_wait_cluster(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag,
                                       p.timeout_ns)) {
                    failed = true;
                    break;
                }
                tc_fence_after();
                const uint32_t d_tmem = tmem_base + static_cast<uint32_t>(acc * BN);
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
                    if (!mbar_wait(smem_u32(&full[stage]), phase, abort_flag, p.timeout_ns)) {
                        failed = true;
                        break;
                    }
                    ++consumed;
                    tc_fence_after();
                    const uint32_t a_base = smem_u32(sA + stage * kAStageBytes);
                    const uint32_t b_base = smem_u32(sB + stage * Cfg::kBStageBytes);
#pragma unroll
                    for (int k = 0; k < kBK / 16; ++k)
                        tc_mma_f16_pair(d_tmem, operand_desc<A_MN>(a_base, k),
                                        operand_desc<B_MN>(b_base, k), idesc,
                                        (kb != sg.kb0 || k != 0) ? 1u : 0u);
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
            *n_consumed = consumed;
            if (failed) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
                const volatile int never = 0;
                tc_commit_pair_mc(smem_u32(drain), 0x1);
                mbar_wait(smem_u32(drain), 0u, &never, 100000000ull);
            }
        }
        __syncwarp();
    } else if (warp <= 4) {
        // ------------------------------------------------------------ epilogue (both CTAs)
        const int q = warp & 3;
        const int lrow = q * 32 + lane;          // TMEM lane = row of this CTA's half tile
        const int row_in_tile = static_cast<int>(rank) * 128 + lrow;
        const int et = threadIdx.x - 32;         // 0..127
        const uint32_t tempty0 = mapa_shared(smem_u32(&tempty[0]), 0);
        const uint32_t tempty1 = mapa_shared(smem_u32(&tempty[1]), 0);
        const uint32_t ebuf = smem_u32(sEpi) + (warp - 1) * kEpiWarpBytes;
        uint32_t eseq = 0;                       // chunk counter of this warp's two buffers
        int acc = 0;
        uint32_t acc_phase = 0;
        PairWalker walk(p, cid, ncl);
        PairSeg sg;
        while (walk.next(sg)) {
            int tm, tn;
            tile_coord32(sg.tile, p.tiles_m, p.tiles_n, p.group, tm, tn);
            const bool waited =
                mbar_wait(smem_u32(&tfull[acc]), acc_phase, abort_flag, p.timeout_ns);
            if (!waited && p.status != nullptr) atomicOr(p.status, kDevTimeout);
            bool in_range = true;
#if DG_CHECKED
            // A checked build tests a partial tile's counter and workspace parts
            // first; a failure stops the cluster like a wait that gave up.
            if (sg.kb0 != 0 || sg.kb1 != num_kb) {
                const int64_t f = share_of(int64_t(sg.tile) * num_kb, walk.t_sk, walk.g);
                const int64_t l = share_of(int64_t(sg.tile + 1) * num_kb - 1, walk.t_sk, walk.g);
                in_range = DG_CHECK(p.status, kChkCounter,
                                    span_inside(0, int64_t(sg.tile) * 2 + rank, 1, 1, p.counters_len));
                for (int64_t sh = f; sh <= l && in_range; ++sh)
                    in_range = DG_CHECK(
                        p.status, kChkWs,
                        span_inside(0, ((sh * 2 + walk.slot_of(sh, sg.tile)) * 2 + rank) * (BN * 128),
                                    BN * 128, 1, p.ws_len));
            }
#endif
            // One decision for all 128 epilogue threads: they share named barriers below.
            if (!named_bar_and(1, 128, waited && in_range)) {
                *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const int row = tm * 256 + row_in_tile;
            const int col0 = tn * BN;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            const uint32_t tempty_peer0 = acc == 0 ? tempty0 : tempty1;
            if (sg.kb0 != 0 || sg.kb1 != num_kb) {
                // ---- a stream-K partial tile.  The shares [first, last] that cover it
                // each hold a partial sum; C = ((p_first + p_first+1) + ...) + p_last.
                // Partials live in the workspace as [share][slot][rank][BN/4][128][4]
                // floats: one float4 per (4 columns, row), so a warp moves 512
                // contiguous bytes per access.  Work goes 64 columns per round.
                const int64_t first = share_of(int64_t(sg.tile) * num_kb, walk.t_sk, walk.g);
                const int64_t last = share_of(int64_t(sg.tile + 1) * num_kb - 1, walk.t_sk, walk.g);
                const int nparts = static_cast<int>(last - first + 1);
                int* counter = p.counters + sg.tile * 2 + static_cast<int>(rank);
                auto part_of = [&](int64_t sh) -> float4* {
                    return reinterpret_cast<float4*>(
                        p.ws + ((sh * 2 + walk.slot_of(sh, sg.tile)) * 2 + rank) * (BN * 128));
                };
                auto own_round = [&](int c0, uint32_t (&lo)[32], uint32_t (&hi)[32]) {
                    tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c0), lo);
                    tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c0 + 32), hi);
                    tmem_ld_wait(lo);
                    if (c0 + 64 == BN) {
                        tc_fence_before();
                        mbar_arrive_cluster(tempty_peer0);
                    }
                };
                auto load_round = [&](const float4* src, int c0, float4 (&t)[16]) {
#pragma unroll
                    for (int j = 0; j < 16; ++j) t[j] = __ldcg(src + (c0 / 4 + j) * 128 + lrow);
                };
                auto store_round = [&](int c0, uint32_t (&lo)[32], uint32_t (&hi)[32]) {
                    if (p.c_type == kOutF32) {
                        epi_store_chunk(p, &mapC, ebuf, eseq, lane, row - lane, col0 + c0, lo, hi);
                        epi_store_chunk(p, &mapC, ebuf, eseq, lane, row - lane, col0 + c0 + 32, hi,
                                        lo);
                    } else {
                        epi_store_chunk(p, &mapC, ebuf, eseq, lane, row - lane, col0 + c0, lo, hi);
                    }
                };
                // Sum one 64-column round of the tile in share order.  fold: this
                // share's own partial comes straight from TMEM (it never published).
                auto sum_round = [&](int c0, bool fold, uint32_t (&lo)[32], uint32_t (&hi)[32]) {
                    float4 s4[16];
#pragma unroll 1
                    for (int64_t sh = first; sh <= last; ++sh) {
                        float4 t[16];
                        if (fold && sh == sg.share) {
#pragma unroll
                            for (int h = 0; h < 2; ++h) {
                                uint32_t v[32];
                                tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c0 + 32 * h), v);
                                tmem_ld_wait(v);
#pragma unroll
                                for (int j = 0; j < 8; ++j)
                                    t[8 * h + j] = make_float4(
                                        __uint_as_float(v[4 * j]), __uint_as_float(v[4 * j + 1]),
                                        __uint_as_float(v[4 * j + 2]), __uint_as_float(v[4 * j + 3]));
                            }
                            if (c0 + 64 == BN) {
                                tc_fence_before();
                                mbar_arrive_cluster(tempty_peer0);
                            }
                        } else {
                            load_round(part_of(sh), c0, t);
                        }
                        if (sh == first) {
#pragma unroll
                            for (int j = 0; j < 16; ++j) s4[j] = t[j];
                        } else {
#pragma unroll
                            for (int j = 0; j < 16; ++j) {
                                s4[j].x += t[j].x;
                                s4[j].y += t[j].y;
                                s4[j].z += t[j].z;
                                s4[j].w += t[j].w;
                            }
                        }
                    }
#pragma unroll
                    for (int j = 0; j < 8; ++j) {
                        lo[4 * j] = __float_as_uint(s4[j].x);
                        lo[4 * j + 1] = __float_as_uint(s4[j].y);
                        lo[4 * j + 2] = __float_as_uint(s4[j].z);
                        lo[4 * j + 3] = __float_as_uint(s4[j].w);
                        hi[4 * j] = __float_as_uint(s4[j + 8].x);
                        hi[4 * j + 1] = __float_as_uint(s4[j + 8].y);
                        hi[4 * j + 2] = __float_as_uint(s4[j + 8].z);
                        hi[4 * j + 3] = __float_as_uint(s4[j + 8].w);
                    }
                };
                // Fold: when every other share of the tile has already published, this
                // share adds their partials to its accumulator without publishing its
                // own.  Both ways sum in share order, so the bits are the same.
                if (et == 0) *last_flag = (load_acquire_gpu(counter) == nparts - 1) ? 2 : 0;
                named_bar_sync(1, 128);
                if (*last_flag == 2) {
#pragma unroll 1
                    for (int c0 = 0; c0 < BN; c0 += 64) {
                        uint32_t lo[32], hi[32];
                        sum_round(c0, true, lo, hi);
                        store_round(c0, lo, hi);
                    }
                    if (et == 0) store_relaxed_gpu(counter, 0);
                } else {
                    // Publish this share's partial, then count it in; the share that
                    // arrives last sums every partial.
                    float4* mine = part_of(sg.share);
#pragma unroll 1
                    for (int c0 = 0; c0 < BN; c0 += 64) {
                        uint32_t lo[32], hi[32];
                        own_round(c0, lo, hi);
#pragma unroll
                        for (int j = 0; j < 8; ++j) {
                            __stcg(mine + (c0 / 4 + j) * 128 + lrow,
                                   make_float4(__uint_as_float(lo[4 * j]), __uint_as_float(lo[4 * j + 1]),
                                               __uint_as_float(lo[4 * j + 2]), __uint_as_float(lo[4 * j + 3])));
                            __stcg(mine + (c0 / 4 + j + 8) * 128 + lrow,
                                   make_float4(__uint_as_float(hi[4 * j]), __uint_as_float(hi[4 * j + 1]),
                                               __uint_as_float(hi[4 * j + 2]), __uint_as_float(hi[4 * j + 3])));
                        }
                    }
                    named_bar_sync(1, 128);
                    if (et == 0) {
                        const int old = atomic_add_acq_rel_gpu(counter, 1);
                        *last_flag = (old == nparts - 1) ? 1 : 0;
                    }
                    named_bar_sync(1, 128);
                    if (*last_flag) {
#pragma unroll 1
                        for (int c0 = 0; c0 < BN; c0 += 64) {
                            uint32_t lo[32], hi[32];
                            sum_round(c0, false, lo, hi);
                            store_round(c0, lo, hi);
                        }
                        if (et == 0) store_relaxed_gpu(counter, 0);
                    }
                }
            } else {
                epilogue_staged<BN>(p, &mapC, ebuf, eseq, taddr, lane,
                                 row - lane, col0, [&] {
                                     tc_fence_before();
                                     mbar_arrive_cluster(tempty_peer0);
                                 });
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
            int issued = 0;
            PairWalker walk(p, cid, ncl);
            PairSeg sg;
            while (!failed && walk.next(sg)) {
                int tm, tn;
                tile_coord32(sg.tile, p.tiles_m, p.tiles_n, p.group, tm, tn);
                const int a_row = tm * 256 + static_cast<int>(rank) * 128;
                const int b_col = tn * BN + static_cast<int>(rank) * Cfg::kBHalf;
                for (int kb = sg.kb0; kb < sg.kb1; ++kb) {
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
                    ++issued;
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
            *n_issued = issued;
            if (failed) {
                *abort_flag = 1;
                if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
            }
        }
        __syncwarp();
    }

    // The TMA stores of C must have completed before the CTA's shared memory goes away.
    if (warp >= 1 && warp <= 4 && lane == 0 && p.c_tma) bulk_wait_group0();
    tc_fence_before();
    __syncthreads();
    cluster_sync();      // #1: no role of either CTA issues anything any more
    // After a wait gave up in either CTA, copies may still be on their way into
    // both CTAs' shared memory, and those of CTA 1 complete on CTA 0's barriers,
    // which CTA 1 cannot observe.  CTA 0 therefore brings every stage that either
    // producer issued but the MMA did not consume to completion -- arming the
    // ones only CTA 1 issued, cancelling the bytes of CTA 1's half where only
    // CTA 0 issued -- and waits for each (bounded); the second cluster barrier
    // then keeps both CTAs until they have landed.  (At most STAGES stages are
    // outstanding: a producer issues stage i only after the MMA freed i - STAGES.)
    // Multicast commits of CTA 0's MMA issuer (the empty and tfull arrivals) may
    // also still be on their way into CTA 1 when a role that waited for them gave
    // up: a last commit to both CTAs, which arrives after every earlier one, is
    // waited for by both.
    const uint32_t peer = rank ^ 1u;
    if ((leader && warp == 5 && lane == 0) || (warp == 0 && lane == 0)) {
        const bool any_abort =
            *abort_flag != 0 ||
            ld_shared_cluster_s32(mapa_shared(smem_u32(const_cast<int*>(abort_flag)), peer)) != 0;
        if (any_abort && warp == 0) {
            const volatile int never = 0;
            if (leader) tc_commit_pair_mc(smem_u32(final_bar), 0x3);
            mbar_wait(smem_u32(final_bar), 0u, &never, 100000000ull);
        }
        if (any_abort && warp == 5) {
            const int n0 = *n_issued;
            const int n1 = ld_shared_cluster_s32(mapa_shared(smem_u32(const_cast<int*>(n_issued)), 1));
            const int c = *n_consumed;
            const int n = n0 > n1 ? n0 : n1;
            const volatile int never = 0;
            for (int i = c; i < n; ++i) {
                const uint32_t fb = smem_u32(&full[i % STAGES]);
                if (i >= n0)
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(Cfg::kStageBytes));
                else if (i >= n1)
                    mbar_complete_tx(fb, static_cast<uint32_t>(Cfg::kStageBytes));
                mbar_wait(fb, static_cast<uint32_t>(i / STAGES) & 1u, &never, 100000000ull);
            }
        }
    }
    cluster_sync();      // #2: neither CTA leaves while a copy or commit may still land in it
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
    return launch_pdl(gemm_pair_kernel<BN, STAGES, A_MN, B_MN>, dim3(grid),
                      dim3(PairCfg<BN, STAGES>::kThreads), PairCfg<BN, STAGES>::kSmemBytes, s, a, b,
                      c, p, idesc);
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
