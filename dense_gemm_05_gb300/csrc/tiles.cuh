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

// Store 32 consecutive accumulator values of one C row starting at element
// `off` (= row * ldc + col), the first `ncols` of them in range, converting to
// the output type with round-to-nearest-even.  `vec`: the row start is
// 16-byte aligned (C base and ldc allow 16-byte stores).
__device__ __forceinline__ void store_c32(const Params& p, int64_t off, const uint32_t (&v)[32],
                                          int ncols) {
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

// Store one accumulator value (skinny epilogue, scattered columns).
__device__ __forceinline__ void store_c1(const Params& p, int64_t off, float x) {
    if (p.c_type == kOutF32)
        static_cast<float*>(p.C)[off] = x;
    else
        static_cast<uint16_t*>(p.C)[off] =
            static_cast<uint16_t>(pack_out(x, 0.0f, p.c_type) & 0xFFFFu);
}

}  // namespace dg
