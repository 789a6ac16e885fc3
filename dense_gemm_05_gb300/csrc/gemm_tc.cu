// gemm_tc.cu -- persistent, warp-specialised tcgen05 GEMM for sm_103a.
//
// One CTA per SM walks output tiles of BM x BN (BM = 128, or 64 for small
// problems: M = 64 MMAs) in the scheduler's order.
// Each tile is the K-loop of "acc += A_tile @ B_tile" ("Writing GPU kernels in
// Triton: Vector Add, Softmax, MatMul", section 3.3; "Triton 04", section
// "Why have acc"), with the fp32 accumulator held in tensor memory.
//
// Warp roles (one CTA):
//   warp 0        MMA issuer (one thread) and TMEM owner
//   warps 1..4    epilogue: TMEM -> registers -> masked global stores of C
//   warp 5        TMA producer (TMA variant), or
//   warps 5..8    load/store producer (generic variant, any alignment)
//
// Shared memory holds a ring of STAGES {A BMx64, B 64xBN} tiles in the
// 128-byte-swizzled layouts of tiles.cuh (A_MN / B_MN: the operand is stored
// with M / N contiguous, i.e. A transposed, or B in its natural K x N layout);
// "full" barriers hand a stage to the MMA issuer, "empty" barriers
// (tcgen05.commit) hand it back.  Two TMEM accumulators of BM x BN fp32 let
// the epilogue drain tile i while the MMAs of tile i+1 run.
//
// Masking: TMA fills elements outside the global tensor with zeros (the
// masked load with other=0 of "I Wrote a GPU Matmul Kernel From Scratch in
// Triton", Step 3); the generic producer writes zeros itself; the epilogue
// stores only rows < M and columns < N (the masked store).
#include "common.cuh"
#include "ptx.cuh"
#include "tiles.cuh"

namespace dg {

template <int BM, int BN, int STAGES, bool GENERIC>
struct TcCfg {
    static_assert(BM == 128 || (BM == 64 && !GENERIC), "tile rows");
    static constexpr int kAStageBytes = BM * kBK * 2;
    static constexpr int kBStageBytes = BN * kBK * 2;
    static constexpr int kStageBytes = kAStageBytes + kBStageBytes;
    // Accumulator rows each epilogue warp holds: an M = 128 MMA puts row r in
    // TMEM lane r; an M = 64 one puts rows 16 q .. 16 q + 15 in lanes 0 .. 15 of
    // lane quarter q.
    static constexpr int kRowsPerWarp = BM / 4;
    static constexpr int kTmemCols = 2 * BN;               // two fp32 accumulators, power of 2
    static constexpr int kProducerWarps = GENERIC ? 4 : 1;
    static constexpr int kThreads = 32 * (1 + 4 + kProducerWarps);
    static constexpr int kNumBars = 2 * STAGES + 5;
    static constexpr int kEpiBytes = GENERIC ? 0 : kEpiSmemBytes;   // TMA-store staging
    static constexpr int kSmemBytes = 1024 + STAGES * kStageBytes + kEpiBytes + 8 * kNumBars + 16;
    static_assert(BN % kSubN == 0 && BN >= 64 && BN <= 256, "BN");
    static_assert(kSmemBytes <= 232448, "shared memory");
};

__device__ __forceinline__ void raise_abort(const Params& p, volatile int* abort_flag) {
    *abort_flag = 1;
    if (p.status != nullptr) atomicOr(p.status, kDevTimeout);
}

// Eight consecutive 16-bit elements of a stored rows x cols matrix (pitch ld),
// from (row, col) on; elements beyond cols, or all of them when row >= rows,
// read as zero.  In a checked build each load is tested against the rectangle
// first (`kind`: the operand's status bit).
__device__ __forceinline__ uint4 load8(const uint16_t* base, int64_t ld, int row, int col,
                                       int rows, int cols, int vec, int* status, int kind) {
    uint4 r = make_uint4(0u, 0u, 0u, 0u);
    const int remaining = cols - col;
    if (row >= rows || remaining <= 0) return r;
    const uint16_t* ptr = base + static_cast<int64_t>(row) * ld + col;
    if (vec && remaining >= 8) {
        if (!DG_CHECK(status, kind, span_inside(row, col, 8, rows, cols))) return r;
        return __ldg(reinterpret_cast<const uint4*>(ptr));
    }
    uint32_t e[8];
#pragma unroll
    for (int i = 0; i < 8; ++i)
        e[i] = (i < remaining && DG_CHECK(status, kind, span_inside(row, col + i, 1, rows, cols)))
                   ? static_cast<uint32_t>(__ldg(ptr + i))
                   : 0u;
    r.x = e[0] | (e[1] << 16);
    r.y = e[2] | (e[3] << 16);
    r.z = e[4] | (e[5] << 16);
    r.w = e[6] | (e[7] << 16);
    return r;
}

// One operand tile (ROWS M/N rows x 64 K) staged by 128 threads with ordinary
// loads into the same swizzled layout TMA would produce.  MN_MAJOR: the stored
// operand has K rows of contiguous M/N elements; otherwise M/N rows of
// contiguous K elements.  Out-of-range elements are written as zeros.
template <bool MN_MAJOR, int ROWS>
__device__ __forceinline__ void load_tile_generic(uint32_t dst, const uint16_t* base, int64_t ld,
                                                  int mn0, int k0, int mn_total, int k_total,
                                                  int vec, int pt, int* status, int kind) {
    constexpr int kChunks = ROWS * kBK / 8;      // 16-byte chunks in the tile
    constexpr int kPer = kChunks / 128;
    constexpr int kRowChunks = MN_MAJOR ? ROWS / 8 : kBK / 8;
    uint4 v[kPer];
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int q = pt + i * 128;
        const int r = q / kRowChunks, c = q % kRowChunks;
        if constexpr (MN_MAJOR) {
            v[i] = load8(base, ld, k0 + r, mn0 + c * 8, k_total, mn_total, vec, status, kind);
        } else {
            v[i] = load8(base, ld, mn0 + r, k0 + c * 8, mn_total, k_total, vec, status, kind);
        }
    }
#pragma unroll
    for (int i = 0; i < kPer; ++i) {
        const int q = pt + i * 128;
        const int r = q / kRowChunks, c = q % kRowChunks;
        st_shared_v4_b32(dst + chunk_offset<MN_MAJOR>(r, c), v[i]);
    }
}

template <int BM, int BN, int STAGES, bool GENERIC, bool A_MN, bool B_MN>
__global__ void __launch_bounds__(TcCfg<BM, BN, STAGES, GENERIC>::kThreads, 1)
    gemm_tc_kernel(const __grid_constant__ CUtensorMap mapA,
                   const __grid_constant__ CUtensorMap mapB,
                   const __grid_constant__ CUtensorMap mapC, const Params p,
                   const uint32_t idesc) {
    using Cfg = TcCfg<BM, BN, STAGES, GENERIC>;
    constexpr int kAStageBytes = Cfg::kAStageBytes;
    extern __shared__ uint8_t smem_raw[];
    uint8_t* smem = reinterpret_cast<uint8_t*>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    uint8_t* sA = smem;
    uint8_t* sB = smem + STAGES * kAStageBytes;
    uint8_t* sEpi = sB + STAGES * Cfg::kBStageBytes;      // TMA-store staging (not in GENERIC)
    uint64_t* bars = reinterpret_cast<uint64_t*>(sEpi + Cfg::kEpiBytes);
    uint64_t* full = bars;
    uint64_t* empty = bars + STAGES;
    uint64_t* tfull = bars + 2 * STAGES;
    uint64_t* tempty = tfull + 2;
    uint64_t* drain = tempty + 2;
    uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
    volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;

    if (threadIdx.x == 0) {
        for (int s = 0; s < STAGES; ++s) {
            mbar_init(smem_u32(&full[s]), GENERIC ? 128u : 1u);
            mbar_init(smem_u32(&empty[s]), 1u);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(smem_u32(&tfull[a]), 1u);
            mbar_init(smem_u32(&tempty[a]), 128u);
        }
        mbar_init(smem_u32(drain), 1u);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) {
        tmem_alloc(smem_u32(tmem_slot), Cfg::kTmemCols);
        tmem_relinquish();
    }
    if (!GENERIC && warp == 5 && lane == 0) {
        prefetch_tmap(&mapA);
        prefetch_tmap(&mapB);
        if (p.c_tma) prefetch_tmap(&mapC);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem_base = *tmem_slot;
    griddep_wait();                  // the previous grid's writes (A, B, C, workspace) are done
    griddep_launch_dependents();

    const int total = p.tiles_m * p.tiles_n;
    const int num_kb = p.num_kb;

    if (warp == 0) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            bool failed = false;
            int stage = 0;
            uint32_t phase = 0;
            int acc = 0;
            uint32_t acc_phase = 0;
            for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
                if (!mbar_wait(smem_u32(&tempty[acc]), acc_phase ^ 1u, abort_flag, p.timeout_ns)) {
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
                        tc_mma_f16(d_tmem, operand_desc<A_MN>(a_base, k),
                                   operand_desc<B_MN>(b_base, k), idesc, (kb | k) != 0 ? 1u : 0u);
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
                raise_abort(p, abort_flag);
                // Let every MMA already issued finish before TMEM is released.
                const volatile int never = 0;
                tc_commit(smem_u32(drain));
                mbar_wait(smem_u32(drain), 0u, &never, 100000000ull);
            }
        }
        __syncwarp();
    } else if (warp <= 4) {
        // ------------------------------------------------------------ epilogue
        const int q = warp & 3;                 // TMEM lane quarter this warp may access
        uint32_t eseq = 0;                      // chunk counter of this warp's two buffers
        const int row_in_tile = q * Cfg::kRowsPerWarp + lane;   // valid for lane < kRowsPerWarp
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            int tm, tn;
            tile_coord32(t, p.tiles_m, p.tiles_n, p.group, tm, tn);
            const bool ok =
                mbar_wait(smem_u32(&tfull[acc]), acc_phase, abort_flag, p.timeout_ns);
            if (!__all_sync(0xffffffffu, ok)) {
                raise_abort(p, abort_flag);
                break;
            }
            tc_fence_after();
            const int row = tm * BM + row_in_tile;
            const int col0 = tn * BN;
            const uint32_t taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) +
                                   static_cast<uint32_t>(acc * BN);
            const uint32_t tempty_bar = smem_u32(&tempty[acc]);
            if (!GENERIC) {
                epilogue_staged<BN, Cfg::kRowsPerWarp>(p, &mapC, smem_u32(sEpi) + (warp - 1) * kEpiWarpBytes, eseq,
                                    taddr, lane,
                                 row - lane, col0, [&] {
                                     tc_fence_before();
                                     mbar_arrive(tempty_bar);
                                 });
            } else {
                const bool row_ok = row < p.M && lane < Cfg::kRowsPerWarp;
#pragma unroll 1
                for (int c = 0; c < BN / 32; ++c) {
                    uint32_t v[32];
                    tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(c * 32), v);
                    tmem_ld_wait(v);
                    if (c == BN / 32 - 1) {
                        tc_fence_before();
                        mbar_arrive(tempty_bar);
                    }
                    if (row_ok) store_c32(p, row, col0 + c * 32, v);
                }
            }
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1u;
            }
        }
    } else if (!GENERIC) {
        // ------------------------------------------------------------ TMA producer
        if (lane == 0) {
            bool failed = false;
            int stage = 0;
            uint32_t phase = 0;
            int64_t armed = 0;
            for (int t = blockIdx.x; t < total && !failed; t += gridDim.x) {
                int tm, tn;
                tile_coord32(t, p.tiles_m, p.tiles_n, p.group, tm, tn);
                for (int kb = 0; kb < num_kb; ++kb) {
                    if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag,
                                   p.timeout_ns)) {
                        failed = true;
                        break;
                    }
                    const uint32_t fb = smem_u32(&full[stage]);
                    mbar_arrive_expect_tx(fb, static_cast<uint32_t>(Cfg::kStageBytes));
                    load_operand<A_MN>(smem_u32(sA + stage * kAStageBytes), &mapA, fb, tm * BM,
                                       kb * kBK, BM);
                    load_operand<B_MN>(smem_u32(sB + stage * Cfg::kBStageBytes), &mapB, fb,
                                       tn * BN, kb * kBK, BN);
                    ++armed;
                    if (++stage == STAGES) {
                        stage = 0;
                        phase ^= 1u;
                    }
                }
            }
            if (failed) {
                raise_abort(p, abort_flag);
                // Wait (bounded) for the copies already issued to land before the CTA exits.
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
    } else {
        // ------------------------------------------------------------ generic producer
        const int pt = threadIdx.x - 160;     // 0..127
        int stage = 0;
        uint32_t phase = 0;
        for (int t = blockIdx.x; t < total; t += gridDim.x) {
            int tm, tn;
            tile_coord32(t, p.tiles_m, p.tiles_n, p.group, tm, tn);
            bool failed = false;
            for (int kb = 0; kb < num_kb; ++kb) {
                if (!mbar_wait(smem_u32(&empty[stage]), phase ^ 1u, abort_flag, p.timeout_ns)) {
                    failed = true;
                    break;
                }
                load_tile_generic<A_MN, BM>(smem_u32(sA + stage * kAStageBytes), p.A, p.lda,
                                            tm * BM, kb * kBK, p.M, p.K, p.a_vec, pt, p.status,
                                             kChkA);
                load_tile_generic<B_MN, BN>(smem_u32(sB + stage * Cfg::kBStageBytes), p.B, p.ldb,
                                            tn * BN, kb * kBK, p.N, p.K, p.b_vec, pt, p.status,
                                            kChkB);
                fence_proxy_async_smem();
                mbar_arrive(smem_u32(&full[stage]));
                if (++stage == STAGES) {
                    stage = 0;
                    phase ^= 1u;
                }
            }
            if (failed) {
                raise_abort(p, abort_flag);
                break;
            }
        }
    }

    // The TMA stores of C must have completed before the CTA's shared memory goes away.
    if (!GENERIC && warp >= 1 && warp <= 4 && lane == 0 && p.c_tma) bulk_wait_group0();
    tc_fence_before();
    __syncthreads();
    if (warp == 0) {
        tc_fence_after();
        tmem_dealloc(tmem_base, Cfg::kTmemCols);
    }
}

// ---------------------------------------------------------------- host side

namespace {
constexpr int kTmaStages256 = 4;
constexpr int kTmaStages128 = 6;
constexpr int kTmaStages64 = 6;
constexpr int kGenericStages = 4;

template <int BM, int BN, int STAGES, bool GENERIC, bool A_MN, bool B_MN>
cudaError_t set_attrs_one() {
    using Cfg = TcCfg<BM, BN, STAGES, GENERIC>;
    return cudaFuncSetAttribute(gemm_tc_kernel<BM, BN, STAGES, GENERIC, A_MN, B_MN>,
                                cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg::kSmemBytes);
}

template <int BM, int BN, int STAGES, bool GENERIC>
cudaError_t set_attrs() {
    cudaError_t e = set_attrs_one<BM, BN, STAGES, GENERIC, false, true>();
    if (e == cudaSuccess) e = set_attrs_one<BM, BN, STAGES, GENERIC, false, false>();
    if (e == cudaSuccess) e = set_attrs_one<BM, BN, STAGES, GENERIC, true, true>();
    if (e == cudaSuccess) e = set_attrs_one<BM, BN, STAGES, GENERIC, true, false>();
    return e;
}

template <int BM, int BN, int STAGES, bool GENERIC, bool A_MN, bool B_MN>
cudaError_t launch_one(const CUtensorMap& a, const CUtensorMap& b, const CUtensorMap& c,
                       const Params& p, uint32_t idesc, int grid, cudaStream_t s) {
    using Cfg = TcCfg<BM, BN, STAGES, GENERIC>;
    return launch_pdl(gemm_tc_kernel<BM, BN, STAGES, GENERIC, A_MN, B_MN>, dim3(grid),
                      dim3(Cfg::kThreads), Cfg::kSmemBytes, s, a, b, c, p, idesc);
}

template <int BM, int BN, int STAGES, bool GENERIC>
cudaError_t launch(bool a_mn, bool b_mn, const CUtensorMap& a, const CUtensorMap& b,
                   const CUtensorMap& c, const Params& p, uint32_t idesc, int grid,
                   cudaStream_t s) {
    if (!a_mn && b_mn)
        return launch_one<BM, BN, STAGES, GENERIC, false, true>(a, b, c, p, idesc, grid, s);
    if (!a_mn && !b_mn)
        return launch_one<BM, BN, STAGES, GENERIC, false, false>(a, b, c, p, idesc, grid, s);
    if (a_mn && b_mn)
        return launch_one<BM, BN, STAGES, GENERIC, true, true>(a, b, c, p, idesc, grid, s);
    return launch_one<BM, BN, STAGES, GENERIC, true, false>(a, b, c, p, idesc, grid, s);
}
}  // namespace

int tma_smem_bytes(int bm, int bn) {
    if (bn == 256) return TcCfg<128, 256, kTmaStages256, false>::kSmemBytes;
    if (bn == 64)
        return bm == 64 ? TcCfg<64, 64, kTmaStages64, false>::kSmemBytes
                        : TcCfg<128, 64, kTmaStages64, false>::kSmemBytes;
    return TcCfg<128, 128, kTmaStages128, false>::kSmemBytes;
}

int tma_stages(int bn) {
    return bn == 256 ? kTmaStages256 : (bn == 64 ? kTmaStages64 : kTmaStages128);
}

cudaError_t tma_prepare() {
    cudaError_t e = set_attrs<128, 256, kTmaStages256, false>();
    if (e == cudaSuccess) e = set_attrs<128, 128, kTmaStages128, false>();
    if (e == cudaSuccess) e = set_attrs<128, 64, kTmaStages64, false>();
    if (e == cudaSuccess) e = set_attrs<64, 64, kTmaStages64, false>();
    return e;
}

cudaError_t launch_tma(int bm, int bn, bool a_mn, bool b_mn, const CUtensorMap& mapA,
                       const CUtensorMap& mapB, const CUtensorMap& mapC, const Params& p,
                       uint32_t idesc, int grid, cudaStream_t stream) {
    if (bn == 256)
        return launch<128, 256, kTmaStages256, false>(a_mn, b_mn, mapA, mapB, mapC, p, idesc,
                                                      grid, stream);
    if (bn == 64 && bm == 64)
        return launch<64, 64, kTmaStages64, false>(a_mn, b_mn, mapA, mapB, mapC, p, idesc, grid,
                                                   stream);
    if (bn == 64)
        return launch<128, 64, kTmaStages64, false>(a_mn, b_mn, mapA, mapB, mapC, p, idesc, grid,
                                                    stream);
    return launch<128, 128, kTmaStages128, false>(a_mn, b_mn, mapA, mapB, mapC, p, idesc, grid,
                                                  stream);
}

int generic_smem_bytes() { return TcCfg<128, 128, kGenericStages, true>::kSmemBytes; }

int generic_stages() { return kGenericStages; }

cudaError_t generic_prepare() { return set_attrs<128, 128, kGenericStages, true>(); }

cudaError_t launch_generic(bool a_mn, bool b_mn, const Params& p, uint32_t idesc, int grid,
                           cudaStream_t stream) {
    CUtensorMap dummy;
    memset(&dummy, 0, sizeof(dummy));
    return launch<128, 128, kGenericStages, true>(a_mn, b_mn, dummy, dummy, dummy, p, idesc,
                                                  grid, stream);
}

}  // namespace dg
