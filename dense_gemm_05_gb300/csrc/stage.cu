// stage.cu -- copy a row-major 16-bit matrix whose base or row pitch is not a
// multiple of 16 bytes into a buffer whose rows start on 16-byte boundaries,
// so that the tensor-memory-access kernels can read it (TMA boxes need 16-byte
// aligned rows).  One thread writes one 16-byte piece (8 elements) of a
// destination row; the columns from `cols` up to the padded pitch are zero.
#include "common.cuh"
#include "ptx.cuh"

namespace dg {

namespace {

__global__ void __launch_bounds__(256)
    stage_rows_kernel(const uint16_t* __restrict__ src, int64_t lds, uint16_t* __restrict__ dst,
                      int64_t ldd, int64_t rows, int64_t cols, int* status) {
    griddep_wait();        // src may be written, dst still read, by the previous grid
    griddep_launch_dependents();
    const int64_t pieces = (cols + 7) / 8;          // per row; ldd >= 8 * pieces
    const int64_t total = rows * pieces;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < total;
         i += int64_t(gridDim.x) * blockDim.x) {
        const int64_t r = i / pieces;
        const int64_t c0 = (i - r * pieces) * 8;
        const uint16_t* s = src + r * lds + c0;
        uint32_t w[4];
#pragma unroll
        for (int e = 0; e < 4; ++e) {
            const uint32_t lo = (c0 + 2 * e < cols &&
                                 DG_CHECK(status, kChkStage, span_inside(r, c0 + 2 * e, 1, rows, cols)))
                                    ? s[2 * e] : 0u;
            const uint32_t hi = (c0 + 2 * e + 1 < cols &&
                                 DG_CHECK(status, kChkStage, span_inside(r, c0 + 2 * e + 1, 1, rows, cols)))
                                    ? s[2 * e + 1] : 0u;
            w[e] = lo | (hi << 16);
        }
        if (DG_CHECK(status, kChkStage, span_inside(r, c0, 8, rows, ldd)))
            *reinterpret_cast<uint4*>(dst + r * ldd + c0) = make_uint4(w[0], w[1], w[2], w[3]);
    }
}

}  // namespace

cudaError_t launch_stage_rows(const uint16_t* src, int64_t lds, uint16_t* dst, int64_t ldd,
                              int64_t rows, int64_t cols, int* status, int num_sms,
                              cudaStream_t stream) {
    const int64_t total = rows * ((cols + 7) / 8);
    const int64_t blocks = (total + 255) / 256;
    const int64_t cap = int64_t(num_sms) * 8;
    return launch_pdl(stage_rows_kernel, dim3(static_cast<unsigned>(blocks < cap ? blocks : cap)),
                      dim3(256), 0, stream, src, lds, dst, ldd, rows, cols, status);
}

}  // namespace dg
