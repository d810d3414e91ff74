// Bank packing (rank-local slicing copy) and the dequantisation debug export.
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {

// dst[r][0:width) = src[r][0:width) for r < height: a strided byte copy. Each thread
// moves 16 bytes when both rows are 16-byte aligned, single bytes otherwise.
__global__ void copy2d_kernel(const uint8_t *__restrict__ src, size_t src_pitch, uint8_t *__restrict__ dst,
                              size_t dst_pitch, size_t width, size_t height, int vec)
{
    pdl_enter();
    const size_t per_row = vec ? width / 16 : width;
    const size_t total = per_row * height;
    for (size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x; i < total; i += (size_t)gridDim.x * blockDim.x) {
        const size_t r = i / per_row, col = i - r * per_row;
        if (vec) {
            reinterpret_cast<uint4 *>(dst + r * dst_pitch)[col] = reinterpret_cast<const uint4 *>(src + r * src_pitch)[col];
        } else {
            dst[r * dst_pitch + col] = src[r * src_pitch + col];
        }
    }
}

cudaError_t launch_pack_copy2d(const uint8_t *src, size_t src_pitch, uint8_t *dst, size_t dst_pitch, size_t width,
                               size_t height, cudaStream_t s)
{
    if (width == 0 || height == 0) return cudaSuccess;
    const int vec = ((reinterpret_cast<uintptr_t>(src) | reinterpret_cast<uintptr_t>(dst) | src_pitch | dst_pitch |
                      width) & 15u) == 0;
    const size_t total = (vec ? width / 16 : width) * height;
    size_t blocks = (total + 255) / 256;
    const size_t cap = (size_t)sm_count() * 16;
    if (blocks > cap) blocks = cap;
    FT_LAUNCH(copy2d_kernel, dim3((unsigned)blocks), dim3(256), 0, s, src, src_pitch, dst, dst_pitch, width,
              height, vec);
    count_launches(1);
    return cudaGetLastError();
}

// out[n][k] = bf16(e2m1(code[n][k]) * e4m3(scale[n][k/group])) through dequant8, the
// routine the fused kernels use. One thread per 4 code bytes (8 elements).
__global__ void dequant_kernel(const uint8_t *__restrict__ codes, const uint8_t *__restrict__ scales, int rows,
                               int K, int group, uint16_t *__restrict__ out)
{
    pdl_enter();
    const size_t words = (size_t)rows * (K / 8);
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= words) return;
    const size_t n = i / (K / 8), w = i - n * (K / 8);
    const int k0 = (int)w * 8;
    const uint32_t code4 = reinterpret_cast<const uint32_t *>(codes + n * (K / 2))[w];
    const uint32_t sbyte = scales[n * (K / group) + k0 / group];
    uint32_t s0, s1;
    e4m3x2_to_bf16x2_scaled(sbyte, s0, s1);
    uint32_t v[4];
    dequant8(code4, s0, v);
    uint4 o = make_uint4(v[0], v[1], v[2], v[3]);
    *reinterpret_cast<uint4 *>(out + n * K + k0) = o;
}

cudaError_t launch_dequant(const uint8_t *codes, const uint8_t *scales, int rows, int K, int group, uint16_t *out,
                           cudaStream_t s)
{
    const size_t words = (size_t)rows * (K / 8);
    if (words == 0) return cudaSuccess;
    FT_LAUNCH(dequant_kernel, dim3((unsigned)((words + 255) / 256)), dim3(256), 0, s, codes, scales, rows, K,
              group, out);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
