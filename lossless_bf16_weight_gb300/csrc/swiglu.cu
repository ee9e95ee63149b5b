// Element-wise glue around the matmuls.
//   swiglu    h = bf16(silu(g) * u), silu(z) = z / (1 + e^-z) in fp32 with
//             CUDA's expf.  Memory bound: 8 values per thread per 16-byte
//             load, grid-stride.
//   pad_rows  rows of `cols` values copied into rows of `cp` (a multiple of
//             64) with zeros after them: the activations (and, for the
//             uncompressed matmul, the weights) of a matrix whose rows are
//             stored extended with filler weights.
#include <cuda_bf16.h>

#include "kernels.h"

namespace uw {

namespace {

__device__ __forceinline__ float bf(uint16_t b) { return __uint_as_float(uint32_t(b) << 16); }

__device__ __forceinline__ uint16_t swiglu1(uint16_t g, uint16_t u) {
    const float z = bf(g);
    const float s = z / (1.0f + expf(-z));
    return __bfloat16_as_ushort(__float2bfloat16_rn(s * bf(u)));
}

__global__ void swiglu_kernel(const uint16_t *__restrict__ g, const uint16_t *__restrict__ u,
                              uint16_t *__restrict__ h, int64_t n) {
    grid_dep_launch();
    grid_dep_wait();  // g and u come from the kernels before
    const int64_t n8 = n / 8;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n8; i += stride) {
        const uint4 gv = __ldg(reinterpret_cast<const uint4 *>(g) + i);
        const uint4 uv = __ldg(reinterpret_cast<const uint4 *>(u) + i);
        const uint16_t *ga = reinterpret_cast<const uint16_t *>(&gv);
        const uint16_t *ua = reinterpret_cast<const uint16_t *>(&uv);
        uint4 hv;
        uint16_t *ha = reinterpret_cast<uint16_t *>(&hv);
#pragma unroll
        for (int k = 0; k < 8; k++)
            ha[k] = swiglu1(ga[k], ua[k]);
        reinterpret_cast<uint4 *>(h)[i] = hv;
    }
    for (int64_t i = n8 * 8 + int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride)
        h[i] = swiglu1(g[i], u[i]);
}

__global__ void pad_rows_kernel(const uint16_t *__restrict__ src, int64_t rows, int64_t cols,
                                uint16_t *__restrict__ dst, int64_t cp) {
    grid_dep_launch();
    grid_dep_wait();  // src may come from the kernel before; dst may still be read by it
    const int64_t per_row = cp / 8;
    const int64_t n = rows * per_row;
    const int64_t stride = int64_t(gridDim.x) * blockDim.x;
    for (int64_t i = int64_t(blockIdx.x) * blockDim.x + threadIdx.x; i < n; i += stride) {
        const int64_t r = i / per_row, k0 = (i - r * per_row) * 8;
        const uint16_t *row = src + r * cols;
        uint4 v;
        uint16_t *h = reinterpret_cast<uint16_t *>(&v);
#pragma unroll
        for (int k = 0; k < 8; k++)
            h[k] = k0 + k < cols ? row[k0 + k] : uint16_t(0);
        reinterpret_cast<uint4 *>(dst)[i] = v;
    }
}

}  // namespace

uw_status launch_pad_rows(const uint16_t *src, int64_t rows, int64_t cols, uint16_t *dst, int64_t cp,
                          cudaStream_t stream) {
    if (rows <= 0)
        return UW_OK;
    if (cp % kGroup || cp < cols || (reinterpret_cast<uintptr_t>(dst) & 15u))
        return UW_ERR_INVALID_ARG;
    int64_t blocks = (rows * (cp / 8) + 255) / 256;
    if (blocks > 152 * 16)
        blocks = 152 * 16;
    return launch_overlapped(pad_rows_kernel, dim3(unsigned(blocks)), dim3(256), 0, stream, src, rows, cols, dst,
                             cp) == cudaSuccess
               ? UW_OK
               : UW_ERR_CUDA;
}

uw_status launch_swiglu(const uint16_t *g, const uint16_t *u, uint16_t *h, int64_t n, cudaStream_t stream) {
    if (n <= 0)
        return UW_OK;
    const bool aligned = ((reinterpret_cast<uintptr_t>(g) | reinterpret_cast<uintptr_t>(u) |
                           reinterpret_cast<uintptr_t>(h)) & 15u) == 0;
    if (!aligned)
        return UW_ERR_INVALID_ARG;
    int64_t blocks = (n / 8 + 255) / 256;
    if (blocks < 1)
        blocks = 1;
    if (blocks > 152 * 16)
        blocks = 152 * 16;
    return launch_overlapped(swiglu_kernel, dim3(unsigned(blocks)), dim3(256), 0, stream, g, u, h, n) == cudaSuccess
               ? UW_OK
               : UW_ERR_CUDA;
}

}  // namespace uw
