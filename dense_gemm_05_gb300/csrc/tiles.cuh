// tiles.cuh -- operand tiles in shared memory and the C epilogue store, shared
// by the kernels.  Every operand tile is 64 deep in K and uses the 128-byte
// swizzle; it is either
//   K-major : rows of 64 K elements (128 B) -- A stored M x K, or B stored N x K
//             (the transposed, "weight" layout); one TMA box {64 k, rows}
//   MN-major: sub-tiles of 64 M/N elements x 64 K rows (8 KiB each) -- A stored
//             K x M (transposed), or B stored K x N; TMA boxes {64 mn, 64 k}
// and the tcgen05 shared-memory descriptor of each kind, advanced by one
// 16-deep K step, is described below.
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>

#include "common.cuh"
#include "ptx.cuh"

namespace dg {

// Output element types of the epilogue.
enum : int { kOutF32 = 0, kOutF16 = 1, kOutBF16 = 2 };

// Descriptor of the operand tile at shared address `base`, advanced by `k16`
// steps of 16 K elements.  K-major: 8-row core groups 1024 B apart, a K step is
// 32 B inside the swizzled row.  MN-major: 64-wide sub-tiles 8 KiB apart
// (leading offset), 8-row K groups 1024 B apart, a K step is 16 rows of 128 B.
template <bool MN_MAJOR>
__device__ __forceinline__ uint64_t operand_desc(uint32_t base, int k16) {
    if constexpr (MN_MAJOR)
        return sdesc_sw128(base + static_cast<uint32_t>(k16 * 16 * 128),
                           static_cast<uint32_t>(kSubTileBytes), 1024u);
    else
        return sdesc_sw128(base + static_cast<uint32_t>(k16 * 32), 16u, 1024u);
}

// TMA of one operand tile of `rows` M/N rows (K-major: one box; MN-major: rows/64
// boxes) at M/N offset mn0 and K offset k0, completing on `bar`.
template <bool MN_MAJOR>
__device__ __forceinline__ void load_operand(uint32_t dst, const CUtensorMap* map, uint32_t bar,
                                             int mn0, int k0, int rows) {
    if constexpr (MN_MAJOR) {
        for (int j = 0; j < rows / kSubN; ++j)
            tma_load_2d(dst + static_cast<uint32_t>(j * kSubTileBytes), map, bar, mn0 + j * kSubN,
                        k0);
    } else {
        tma_load_2d(dst, map, bar, k0, mn0);
    }
}

// Same with an L2 cache policy on every box.
template <bool MN_MAJOR>
__device__ __forceinline__ void load_operand_hint(uint32_t dst, const CUtensorMap* map,
                                                  uint32_t bar, int mn0, int k0, int rows,
                                                  uint64_t policy) {
    if constexpr (MN_MAJOR) {
        for (int j = 0; j < rows / kSubN; ++j)
            tma_load_2d_hint(dst + static_cast<uint32_t>(j * kSubTileBytes), map, bar,
                             mn0 + j * kSubN, k0, policy);
    } else {
        tma_load_2d_hint(dst, map, bar, k0, mn0, policy);
    }
}

// The boxes of load_operand_hint, prefetched into L2 only.
template <bool MN_MAJOR>
__device__ __forceinline__ void prefetch_operand_hint(const CUtensorMap* map, int mn0, int k0,
                                                      int rows, uint64_t policy) {
    if constexpr (MN_MAJOR) {
        for (int j = 0; j < rows / kSubN; ++j)
            tma_prefetch_2d_hint(map, mn0 + j * kSubN, k0, policy);
    } else {
        tma_prefetch_2d_hint(map, k0, mn0, policy);
    }
}

// Same for a CTA of a pair: completion is counted on `bar_cluster`, which may
// be the peer CTA's barrier.
template <bool MN_MAJOR>
__device__ __forceinline__ void load_operand_pair(uint32_t dst, const CUtensorMap* map,
                                                  uint32_t bar_cluster, int mn0, int k0, int rows) {
    if constexpr (MN_MAJOR) {
        for (int j = 0; j < rows / kSubN; ++j)
            tma_load_2d_pair(dst + static_cast<uint32_t>(j * kSubTileBytes), map, bar_cluster,
                             mn0 + j * kSubN, k0);
    } else {
        tma_load_2d_pair(dst, map, bar_cluster, k0, mn0);
    }
}

// Shared-memory byte offset of the 16-byte chunk holding elements
// [8c, 8c + 8) of row `r` of a K-major tile, or of K row `r` at M/N elements
// [8c, 8c + 8) of an MN-major tile (c counts 8-element chunks along the
// contiguous dimension of the stored operand).
template <bool MN_MAJOR>
__device__ __forceinline__ uint32_t chunk_offset(int r, int c) {
    if constexpr (MN_MAJOR)
        return static_cast<uint32_t>((c >> 3) * kSubTileBytes + r * 128 + (((c & 7) ^ (r & 7)) << 4));
    else
        return static_cast<uint32_t>(r * 128 + ((c ^ (r & 7)) << 4));
}

__device__ __forceinline__ uint32_t pack_out(float a, float b, int type) {
    if (type == kOutF16) {
        const __half2 h = __floats2half2_rn(a, b);
        return *reinterpret_cast<const uint32_t*>(&h);
    }
    const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);
    return *reinterpret_cast<const uint32_t*>(&h);
}

// Store 32 consecutive accumulator values of C row `row` from column `col` on,
// those below N, converting to the output type with round-to-nearest-even.
// `vec`: the row start is 16-byte aligned (C base and ldc allow 16-byte
// stores).  A checked build tests the row's range first.
__device__ __forceinline__ void store_c32(const Params& p, int row, int col,
                                          const uint32_t (&v)[32]) {
    const int ncols = p.N - col;
    if (ncols <= 0 ||
        !DG_CHECK(p.status, kChkC, span_inside(row, col, ncols < 32 ? ncols : 32, p.M, p.N)))
        return;
    const int64_t off = static_cast<int64_t>(row) * p.ldc + col;
    if (p.c_type == kOutF32) {
        float* dst = static_cast<float*>(p.C) + off;
        if (p.c_vec && ncols >= 32) {
            float4* d4 = reinterpret_cast<float4*>(dst);
#pragma unroll
            for (int i = 0; i < 8; ++i)
                d4[i] = make_float4(__uint_as_float(v[4 * i]), __uint_as_float(v[4 * i + 1]),
                                    __uint_as_float(v[4 * i + 2]), __uint_as_float(v[4 * i + 3]));
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i)
                if (i < ncols) dst[i] = __uint_as_float(v[i]);
        }
        return;
    }
    uint16_t* dst = static_cast<uint16_t*>(p.C) + off;
    if (p.c_vec && ncols >= 32) {
        uint4* d4 = reinterpret_cast<uint4*>(dst);
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            uint4 w;
            w.x = pack_out(__uint_as_float(v[8 * i]), __uint_as_float(v[8 * i + 1]), p.c_type);
            w.y = pack_out(__uint_as_float(v[8 * i + 2]), __uint_as_float(v[8 * i + 3]), p.c_type);
            w.z = pack_out(__uint_as_float(v[8 * i + 4]), __uint_as_float(v[8 * i + 5]), p.c_type);
            w.w = pack_out(__uint_as_float(v[8 * i + 6]), __uint_as_float(v[8 * i + 7]), p.c_type);
            d4[i] = w;
        }
    } else {
#pragma unroll
        for (int i = 0; i < 32; ++i)
            if (i < ncols)
                dst[i] = static_cast<uint16_t>(pack_out(__uint_as_float(v[i]), 0.0f, p.c_type) &
                                               0xFFFFu);
    }
}

// ---------------------------------------------------------------- staged epilogue
// One epilogue warp owns 32 accumulator rows.  It writes C in chunks 128 bytes
// wide (32 fp32 or 64 16-bit columns): the chunk goes to a 4 KiB shared buffer
// of the warp in the 128-byte-swizzled layout (row r at r * 128, 16-byte piece
// j at piece j ^ (r % 8), which spreads the warp's rows over all banks).  With
// c_tma, lane 0 stores it with one TMA box {chunk columns, 32 rows}, which the
// hardware clips to the M x N rectangle.  Otherwise (a C that TMA cannot
// address) the warp writes it back row by row, each row as 128 contiguous
// bytes across the lanes, masked at M and N -- coalesced, where storing each
// lane's own row directly would touch 32 rows per instruction.
constexpr int kEpiBufBytes = 4096;             // one chunk
constexpr int kEpiWarpBytes = 2 * kEpiBufBytes;    // two chunk buffers per epilogue warp
constexpr int kEpiSmemBytes = 4 * kEpiWarpBytes;

// Columns of one chunk for the output type (128 bytes of C).
__device__ __forceinline__ int epi_chunk_cols(int c_type) { return c_type == kOutF32 ? 32 : 64; }

// lo (and hi, for 16-bit output) hold the chunk's accumulator values for this
// lane's row: 32 fp32 bit patterns, or 64 values to be rounded to 16 bits.
// The warp's two chunk buffers (at warp_buf) alternate by `seq`, which the
// warp keeps across all its chunks, so a chunk is written while the previous
// one is still being stored.
__device__ __forceinline__ void epi_store_chunk(const Params& p, const CUtensorMap* mapC,
                                                uint32_t warp_buf, uint32_t& seq, int lane,
                                                int row0, int col, const uint32_t (&lo)[32],
                                                const uint32_t (&hi)[32], int rows = 32) {
    // A chunk wholly outside C (rows from row0 or columns from col beyond M or N)
    // is skipped without touching a buffer: the two buffers then alternate over
    // the stores actually issued, so the wait below always covers the store that
    // last read the buffer about to be rewritten.  (row0 and col are the same on
    // every lane.)
    if (row0 >= p.M || col >= p.N) return;
    const uint32_t buf = warp_buf + (seq & 1u) * static_cast<uint32_t>(kEpiBufBytes);
    ++seq;
    // The store that last read this buffer (two stores ago) must have read it.
    if (p.c_tma && lane == 0) bulk_wait_group_read1();
    __syncwarp();
    const uint32_t row = buf + static_cast<uint32_t>(lane * 128);
    if (p.c_type == kOutF32) {
#pragma unroll
        for (int j = 0; j < 8; ++j)
            st_shared_v4_b32(row + static_cast<uint32_t>((j ^ (lane & 7)) << 4),
                             make_uint4(lo[4 * j], lo[4 * j + 1], lo[4 * j + 2], lo[4 * j + 3]));
    } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t (&h)[32] = j < 4 ? lo : hi;
            const int b = (j & 3) * 8;
            uint4 w;
            w.x = pack_out(__uint_as_float(h[b]), __uint_as_float(h[b + 1]), p.c_type);
            w.y = pack_out(__uint_as_float(h[b + 2]), __uint_as_float(h[b + 3]), p.c_type);
            w.z = pack_out(__uint_as_float(h[b + 4]), __uint_as_float(h[b + 5]), p.c_type);
            w.w = pack_out(__uint_as_float(h[b + 6]), __uint_as_float(h[b + 7]), p.c_type);
            st_shared_v4_b32(row + static_cast<uint32_t>((j ^ (lane & 7)) << 4), w);
        }
    }
    if (p.c_tma) {
        fence_proxy_async_smem();              // generic stores -> visible to the TMA engine
        __syncwarp();
        if (lane == 0) {
            tma_store_2d(mapC, buf, col, row0);
            bulk_commit_group();
        }
        return;
    }
    __syncwarp();
    if (p.c_type == kOutF32 && col + 32 <= p.N) {
        // fp32 C whose rows are only 4-byte aligned, chunk wholly inside N.  A
        // warp store costs about the same whatever its width, so the chunk is
        // written with as few stores as the alignment allows: first every
        // 16-byte slot that lies inside a row (7 or 8 per row: 8 stores of
        // float4 across the warp), then each row's head and tail (the 1-3
        // floats before its first and after its last aligned slot) with at
        // most four 4- and 8-byte stores, one row per lane.
        float* cbase = static_cast<float*>(p.C);
#pragma unroll
        for (int t = 0; t < 8; ++t) {
            const int i = lane + 32 * t;
            const int rr = i >> 3, k = i & 7;
            const int r = row0 + rr;
            const int64_t off = static_cast<int64_t>(r) * p.ldc + col;
            const int h = static_cast<int>((4u - ((reinterpret_cast<uintptr_t>(cbase + off) >> 2) & 3u)) & 3u);
            if (rr < rows && r < p.M && h + 4 * k + 4 <= 32 &&
                DG_CHECK(p.status, kChkC, span_inside(r, col + h + 4 * k, 4, p.M, p.N))) {
                const int e = h + 4 * k;
                const uint32_t rowb = buf + static_cast<uint32_t>(rr * 128);
                float4 v;
                v.x = __uint_as_float(ld_shared_b32(rowb + (static_cast<uint32_t>(((e >> 2) ^ (rr & 7))) << 4) + (e & 3) * 4));
                v.y = __uint_as_float(ld_shared_b32(rowb + (static_cast<uint32_t>((((e + 1) >> 2) ^ (rr & 7))) << 4) + ((e + 1) & 3) * 4));
                v.z = __uint_as_float(ld_shared_b32(rowb + (static_cast<uint32_t>((((e + 2) >> 2) ^ (rr & 7))) << 4) + ((e + 2) & 3) * 4));
                v.w = __uint_as_float(ld_shared_b32(rowb + (static_cast<uint32_t>((((e + 3) >> 2) ^ (rr & 7))) << 4) + ((e + 3) & 3) * 4));
                *reinterpret_cast<float4*>(cbase + off + e) = v;
            }
        }
        const int r = row0 + lane;
        const int64_t off = static_cast<int64_t>(r) * p.ldc + col;
        const int h = static_cast<int>((4u - ((reinterpret_cast<uintptr_t>(cbase + off) >> 2) & 3u)) & 3u);
        if (lane < rows && r < p.M && h != 0 &&
            DG_CHECK(p.status, kChkC, span_inside(r, col, 32, p.M, p.N))) {
            const uint32_t rowb = buf + static_cast<uint32_t>(lane * 128);
            auto elem = [&](int e) {
                return __uint_as_float(ld_shared_b32(
                    rowb + (static_cast<uint32_t>(((e >> 2) ^ (lane & 7))) << 4) + (e & 3) * 4));
            };
            // h = 3: head e0 (4 B) + e1..2 (8 B), tail e31 (4 B); h = 2: head e0..1,
            // tail e30..31 (8 B each); h = 1: head e0 (4 B), tail e29..30 (8 B) + e31.
            if (h & 1) cbase[off] = elem(0);
            if (h >= 2) *reinterpret_cast<float2*>(cbase + off + h - 2) = make_float2(elem(h - 2), elem(h - 1));
            if (h <= 2) *reinterpret_cast<float2*>(cbase + off + 28 + h) = make_float2(elem(28 + h), elem(29 + h));
            if (h & 1) cbase[off + 31] = elem(31);
        }
        return;
    }
    // Lane l reads 32-bit word l of each 128-byte row (in 16-byte piece l / 4).
    const uint32_t word = static_cast<uint32_t>(lane & 3) * 4u;
#pragma unroll 4
    for (int rr = 0; rr < rows; ++rr) {
        const int r = row0 + rr;
        if (r >= p.M) break;
        const uint32_t w = ld_shared_b32(buf + static_cast<uint32_t>(rr * 128) +
                                         ((static_cast<uint32_t>((lane >> 2) ^ (rr & 7))) << 4) +
                                         word);
        const int64_t off = static_cast<int64_t>(r) * p.ldc;
        if (p.c_type == kOutF32) {
            const int c = col + lane;
            if (c < p.N && DG_CHECK(p.status, kChkC, span_inside(r, c, 1, p.M, p.N)))
                static_cast<float*>(p.C)[off + c] = __uint_as_float(w);
        } else {
            const int c = col + 2 * lane;
            uint16_t* dst = static_cast<uint16_t*>(p.C) + off;
            if (c < p.N && DG_CHECK(p.status, kChkC, span_inside(r, c, 1, p.M, p.N)))
                dst[c] = static_cast<uint16_t>(w & 0xFFFFu);
            if (c + 1 < p.N && DG_CHECK(p.status, kChkC, span_inside(r, c + 1, 1, p.M, p.N)))
                dst[c + 1] = static_cast<uint16_t>(w >> 16);
        }
    }
}

// The epilogue of one warp's 32 rows x BN columns of an accumulator at TMEM
// address `taddr` (this warp's lanes), through the staged chunks above.  `release` is called
// after the last TMEM load, so the MMA issuer may reuse the accumulator while
// the final chunks are still being stored.
// ROWS: the accumulator rows this warp holds in its lanes 0 .. ROWS-1 (32, or 16
// for a 64-row tile; the TMA box of mapC is then ROWS rows high).
template <int BN, int ROWS = 32, typename Release>
__device__ __forceinline__ void epilogue_staged(const Params& p, const CUtensorMap* mapC,
                                             uint32_t warp_buf, uint32_t& seq, uint32_t taddr,
                                             int lane, int row0, int col0, Release release) {
    const int cw = epi_chunk_cols(p.c_type);
    const int nchunks = BN / cw;
    if (cw == 32) {
        // fp32 C: two chunks' TMEM loads in flight before one wait, so the load
        // latency is paid once per 64 columns.  (The destination registers of a
        // tcgen05.ld are undefined until tcgen05.wait::ld, so a load must not be
        // left in flight across other code: the compiler may move or spill them.)
        static_assert(BN % 64 == 0, "chunk pairs");
#pragma unroll 1
        for (int ch = 0; ch < BN / 32; ch += 2) {
            uint32_t a[32], b[32], none[32];
            tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(ch * 32), a);
            tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>((ch + 1) * 32), b);
            tmem_ld_wait(a);
            tmem_ld_wait(b);
            if (ch + 2 == BN / 32) release();
            epi_store_chunk(p, mapC, warp_buf, seq, lane, row0, col0 + ch * 32, a, none, ROWS);
            epi_store_chunk(p, mapC, warp_buf, seq, lane, row0, col0 + (ch + 1) * 32, b, none, ROWS);
        }
        return;
    }
#pragma unroll 1
    for (int ch = 0; ch < nchunks; ++ch) {
        uint32_t lo[32], hi[32];
        tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(ch * cw), lo);
        if (cw == 64) {
            tmem_ld_32x32b_x32(taddr + static_cast<uint32_t>(ch * cw + 32), hi);
            tmem_ld_wait(hi);
        } else {
#pragma unroll
            for (int i = 0; i < 32; ++i) hi[i] = 0u;
        }
        tmem_ld_wait(lo);
        if (ch == nchunks - 1) release();
        epi_store_chunk(p, mapC, warp_buf, seq, lane, row0, col0 + ch * cw, lo, hi, ROWS);
    }
}

// ---------------------------------------------------------------- unaligned MN-major rows
// A 64 (K) x 128 (M/N) MN-major operand tile from a matrix whose rows are only
// 2-byte aligned (e.g. a K x N operand with an odd leading dimension, which
// TMA cannot address), for the 4 warps of a warpgroup: warp w4 takes K rows
// w4, w4 + 4, ..., 60 + w4.  The 16-byte-aligned span around each row's 256
// bytes (at most 17 pieces of 16 bytes) is copied by asynchronous 16-byte
// copies (cp.async) into a raw row slot of 272 bytes -- many copies in flight
// per SM, no registers held -- and the elements are then moved into the
// 128-byte-swizzled tile at their 2-byte offset.  A row whose aligned span
// would leave the matrix's footprint [base, base + (K - 1) * ld + MN) -- row 0
// of a base that is not 16-byte aligned, the last row -- is read element by
// element instead.  Elements beyond K or MN are written as zeros.
constexpr int kRawRowBytes = 272;
constexpr int kRawStageBytes = 64 * kRawRowBytes;

struct RowSpan {
    uintptr_t a;      // byte address of the row's first element
    uint32_t d;       // a - (a rounded down to 16 bytes)
    uint32_t pieces;  // 16-byte pieces of the aligned span to copy (0: element-wise or beyond K)
};

// Row k0 + w4 + 4 i of the warp's 16 (i = 0..15).
__device__ __forceinline__ RowSpan unaligned_row_span(const uint16_t* base, int64_t ld, int mn0,
                                                      int k, int mn_total, int k_total) {
    RowSpan r{0, 0, 0};
    if (k >= k_total) return r;
    const uintptr_t lo = reinterpret_cast<uintptr_t>(base);
    const uintptr_t hi =
        reinterpret_cast<uintptr_t>(base + (static_cast<int64_t>(k_total) - 1) * ld + mn_total);
    const int ncols = mn_total - mn0 < 128 ? mn_total - mn0 : 128;
    r.a = reinterpret_cast<uintptr_t>(base + static_cast<int64_t>(k) * ld + mn0);
    const uintptr_t a16 = r.a & ~static_cast<uintptr_t>(15);
    r.d = static_cast<uint32_t>(r.a - a16);
    const uintptr_t e16 = (r.a + 2u * static_cast<uintptr_t>(ncols) + 15u) & ~static_cast<uintptr_t>(15);
    if (a16 >= lo && e16 <= hi) r.pieces = static_cast<uint32_t>(e16 - a16) >> 4;
    return r;
}

// Whether every one of the tile's 64 rows at K offset k0 has its whole aligned
// span inside the footprint: no row 0 of a misaligned base, no last row, no
// row beyond K, and rows at least 8 elements apart (so that the up to 14 bytes
// a span reaches past a row lie in the next or previous row).  Such a stage
// takes the fast paths below.
__device__ __forceinline__ bool unaligned_stage_interior(const uint16_t* base, int64_t ld, int mn0,
                                                         int k0, int k_total) {
    const bool first_ok = k0 > 0 || mn0 > 0 || (reinterpret_cast<uintptr_t>(base) & 15u) == 0u;
    return first_ok && ld >= 8 && k0 + 64 < k_total;   // rows k0 .. k0 + 63 below the last
}

// Issue this warp's copies of its 16 rows of the tile at K offset k0 into the
// raw stage at `raw` (row kk at kk * kRawRowBytes); every lane then arrives on
// `bar` (32 expected arrivals) when its copies have landed.  Half-warp h takes
// rows i = h, h + 2, ..., h + 14 (K rows w4 + 4 i), lane c of it the 16-byte
// piece c of each (lane 0 also piece 16): a warp instruction copies two rows'
// 256 contiguous bytes.  All rows of a half-warp sit at the same offset from a
// 16-byte boundary (their distance, 16 ld bytes, is a multiple of 16), so on
// an interior stage one row's span serves all eight.
__device__ __forceinline__ void unaligned_rows_issue(uint32_t raw, uint32_t bar,
                                                     const uint16_t* base, int64_t ld, int mn0,
                                                     int k0, int mn_total, int k_total, int w4,
                                                     int lane, int* status, int kind) {
    const int h = lane >> 4, c = lane & 15;
#if DG_CHECKED
    // A checked build tests every 16-byte copy against the matrix's footprint.
    const uintptr_t foot_lo = reinterpret_cast<uintptr_t>(base);
    const uintptr_t foot_hi =
        reinterpret_cast<uintptr_t>(base + (static_cast<int64_t>(k_total) - 1) * ld + mn_total);
    auto copy16 = [&](uint32_t dst, uintptr_t src) {
        if (DG_CHECK(status, kind, bytes_inside(src, 16u, foot_lo, foot_hi)))
            cp_async_16(dst, reinterpret_cast<const void*>(src));
    };
#else
    (void)status;
    (void)kind;
    auto copy16 = [&](uint32_t dst, uintptr_t src) {
        cp_async_16(dst, reinterpret_cast<const void*>(src));
    };
#endif
    if (unaligned_stage_interior(base, ld, mn0, k0, k_total)) {
        const RowSpan r0 = unaligned_row_span(base, ld, mn0, k0 + w4 + 4 * h, mn_total, k_total);
        const uintptr_t a16 = r0.a - r0.d;
        const uintptr_t step = static_cast<uintptr_t>(16 * ld);       // 8 K rows, in bytes
        const uint32_t dst0 = raw + static_cast<uint32_t>((w4 + 4 * h) * kRawRowBytes);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            const uint32_t dst = dst0 + static_cast<uint32_t>(j * 8 * kRawRowBytes);
            const uintptr_t src = a16 + static_cast<uintptr_t>(j) * step;
            if (static_cast<uint32_t>(c) < r0.pieces) copy16(dst + 16u * c, src + 16u * c);
            if (c == 0 && r0.pieces > 16) copy16(dst + 256u, src + 256u);
        }
    } else {
#pragma unroll 1
        for (int j = 0; j < 8; ++j) {
            const int kk = w4 + 4 * (h + 2 * j);
            const RowSpan r = unaligned_row_span(base, ld, mn0, k0 + kk, mn_total, k_total);
            const uintptr_t a16 = r.a - r.d;
            const uint32_t dst = raw + static_cast<uint32_t>(kk * kRawRowBytes);
            if (static_cast<uint32_t>(c) < r.pieces) copy16(dst + 16u * c, a16 + 16u * c);
            if (c == 0 && r.pieces > 16) copy16(dst + 256u, a16 + 256u);
        }
    }
    cp_async_arrive(bar);
}

// Move this warp's 16 rows from the raw stage into the swizzled tile at `dst`:
// lane c of half-warp h takes the 16-byte chunk c (elements mn0 + 8c ..) of
// rows h, h + 2, ..., h + 14.
__device__ __forceinline__ void unaligned_rows_place(uint32_t dst, uint32_t raw,
                                                     const uint16_t* base, int64_t ld, int mn0,
                                                     int k0, int mn_total, int k_total, int w4,
                                                     int lane, int* status, int kind) {
    const int h = lane >> 4, c = lane & 15;
    const int n = mn0 + 8 * c;
    uint32_t keep[4];                              // masks of the elements below MN
#pragma unroll
    for (int e = 0; e < 4; ++e)
        keep[e] = (n + 2 * e < mn_total ? 0x0000FFFFu : 0u) | (n + 2 * e + 1 < mn_total ? 0xFFFF0000u : 0u);
    const int kk0 = w4 + 4 * h;                    // rows kk0 + 8 j: same swizzle phase (kk & 7)
    if (unaligned_stage_interior(base, ld, mn0, k0, k_total)) {
        const RowSpan r0 = unaligned_row_span(base, ld, mn0, k0 + kk0, mn_total, k_total);
        const uint32_t d = r0.d;                   // the same for the eight rows
        const uint32_t src0 = raw + static_cast<uint32_t>(kk0 * kRawRowBytes) + 16u * c + (d & ~3u);
        const uint32_t dst0 = dst + chunk_offset<true>(kk0, c);
        const uint32_t sh = 8u * (d & 3u);
#pragma unroll
        for (int j = 0; j < 8; ++j) {
            // bytes [d + 16c, d + 16c + 16) of the raw row (d even); bytes past the
            // copied span are masked below
            const uint32_t src = src0 + static_cast<uint32_t>(j * 8 * kRawRowBytes);
            uint32_t x[5];
#pragma unroll
            for (int t = 0; t < 5; ++t) x[t] = ld_shared_b32(src + 4u * t);
            uint32_t w[4];
#pragma unroll
            for (int t = 0; t < 4; ++t) w[t] = __funnelshift_r(x[t], x[t + 1], sh) & keep[t];
            st_shared_v4_b32(dst0 + static_cast<uint32_t>(j * 8 * 128), make_uint4(w[0], w[1], w[2], w[3]));
        }
        return;
    }
#pragma unroll 1
    for (int j = 0; j < 8; ++j) {
        const int kk = kk0 + 8 * j;
        const int k = k0 + kk;
        const RowSpan r = unaligned_row_span(base, ld, mn0, k, mn_total, k_total);
        uint32_t w[4] = {0u, 0u, 0u, 0u};
        if (r.pieces) {
            const uint32_t src = raw + static_cast<uint32_t>(kk * kRawRowBytes) + 16u * c + (r.d & ~3u);
            uint32_t x[5];
#pragma unroll
            for (int t = 0; t < 5; ++t) x[t] = ld_shared_b32(src + 4u * t);
#pragma unroll
            for (int t = 0; t < 4; ++t) w[t] = __funnelshift_r(x[t], x[t + 1], 8u * (r.d & 3u));
        } else if (k < k_total) {
            const uint16_t* row = base + static_cast<int64_t>(k) * ld;
#pragma unroll
            for (int e = 0; e < 8; ++e)
                if (n + e < mn_total &&
                    DG_CHECK(status, kind, span_inside(k, n + e, 1, k_total, mn_total)))
                    w[e >> 1] |= static_cast<uint32_t>(__ldg(reinterpret_cast<const unsigned short*>(row + n + e)))
                                 << (16 * (e & 1));
        }
        st_shared_v4_b32(dst + chunk_offset<true>(kk, c),
                         make_uint4(w[0] & keep[0], w[1] & keep[1], w[2] & keep[2], w[3] & keep[3]));
    }
}

// Store one accumulator value at C[row, col] (scattered columns).
__device__ __forceinline__ void store_c1(const Params& p, int row, int col, float x) {
    if (!DG_CHECK(p.status, kChkC, span_inside(row, col, 1, p.M, p.N))) return;
    const int64_t off = static_cast<int64_t>(row) * p.ldc + col;
    if (p.c_type == kOutF32)
        static_cast<float*>(p.C)[off] = x;
    else
        static_cast<uint16_t*>(p.C)[off] =
            static_cast<uint16_t>(pack_out(x, 0.0f, p.c_type) & 0xFFFFu);
}

}  // namespace dg
