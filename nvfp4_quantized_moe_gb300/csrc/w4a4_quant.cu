// NVFP4 activation rows for the W4A4 variant (native block-scaled FP4 tensor cores, which
// the pages' sm_86/sm_89 cards lack: "[TP=2] Quantized MoE expert parallelism ... NVFP4
// port", section 2). The pages give no activation recipe; the reading is NVFP4's two-level
// scaling per row: glob = amax / (6 * 448), per 16 elements the e4m3 scale
// s = e4m3(block max / (6 * glob)), codes q = e2m1(x * r) with the block's reciprocal
// r = 1 / (s * glob); every step one correctly rounded fp32 operation, both conversions
// rounding to nearest-even with saturation, so that the codes are a function of the fp32
// inputs alone.
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {

namespace {

// e4m3 byte of a non-negative fp32 value, nearest-even, saturating at 448.
__device__ __forceinline__ uint32_t e4m3_rn_sat(float v)
{
    uint16_t b;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(b) : "f"(0.0f), "f"(v));
    return b & 0xFFu;  // the second operand lands in the low byte
}

// Two e2m1 codes (lo = even element in the low nibble), nearest-even, saturating at 6.
__device__ __forceinline__ uint32_t e2m1x2_rn_sat(float lo, float hi)
{
    uint32_t r;
    asm("{\n\t.reg .b8 t;\n\tcvt.rn.satfinite.e2m1x2.f32 t, %1, %2;\n\tcvt.u32.u8 %0, t;\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return r & 0xFFu;
}

// e4m3 value of a byte (every e4m3 value is an f16 value, hence exact in fp32).
__device__ __forceinline__ float e4m3_value(uint32_t b)
{
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(b));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// The 16 elements of block b of a row as fp32 (two or four 16-byte loads).
template <bool F32_SRC>
__device__ __forceinline__ void load_block(const void *row, int b, float (&v)[16])
{
    if constexpr (F32_SRC) {
        const float4 *p = reinterpret_cast<const float4 *>(row) + 4 * b;
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const float4 q = __ldg(p + i);
            v[4 * i] = q.x; v[4 * i + 1] = q.y; v[4 * i + 2] = q.z; v[4 * i + 3] = q.w;
        }
    } else {
        const uint4 *p = reinterpret_cast<const uint4 *>(row) + 2 * b;
#pragma unroll
        for (int i = 0; i < 2; ++i) {
            const uint4 q = __ldg(p + i);
            const uint32_t w[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                v[8 * i + 2 * j] = __uint_as_float(w[j] << 16);
                v[8 * i + 2 * j + 1] = __uint_as_float(w[j] & 0xFFFF0000u);
            }
        }
    }
}

}  // namespace

// One warp per position row: the source row is the token of sorted_slot[pos] (gate_up's
// expert-sorted copy of x), or pos itself; padding positions (beyond the count, or a
// sentinel slot) get zero codes, scales and row scale. Lanes take the 16-element blocks
// round robin.
template <bool F32_SRC>
__global__ void __launch_bounds__(256) quant_nvfp4_rows_kernel(const void *__restrict__ src, int K,
                                                                 const int *__restrict__ sorted_slot,
                                                                 const int *__restrict__ n_pos_dev, int n_pos_static,
                                                                 int n_slots, int top_k, uint8_t *__restrict__ codes,
                                                                 uint8_t *__restrict__ scales, float *__restrict__ glob,
                                                                 int cap, int *status)
{
    pdl_enter();
    const int n_pos = n_pos_dev ? chk_count(*n_pos_dev, 1, cap, status) : n_pos_static;
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    const int nb = K / 16;
    const size_t esz = F32_SRC ? 4 : 2;  // (rows start 16-byte aligned: K is a multiple of 16)
    for (int pos = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; pos < n_pos; pos += warps) {
        int row = pos;
        if (sorted_slot) {
            const int sl = chk_slot(__ldg(sorted_slot + pos), n_slots, status);
            row = sl < n_slots ? sl / top_k : -1;
        } else if (pos >= n_slots) {
            row = -1;
        }
        uint8_t *cr = codes + (size_t)pos * (K / 2);
        uint8_t *sr = scales + (size_t)pos * nb;
        if (row < 0) {
            for (int b = lane; b < nb; b += 32) {
                *reinterpret_cast<uint2 *>(cr + 8 * b) = make_uint2(0u, 0u);
                sr[b] = 0;
            }
            if (lane == 0) glob[pos] = 0.f;
            continue;
        }
        const void *xr = static_cast<const char *>(src) + (size_t)row * K * esz;
        float amax = 0.f;
        for (int b = lane; b < nb; b += 32) {
            float v[16];
            load_block<F32_SRC>(xr, b, v);
#pragma unroll
            for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(v[i]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xFFFFFFFFu, amax, off));
        const float g = __fdiv_rn(amax, 2688.0f);
        for (int b = lane; b < nb; b += 32) {
            float v[16];
            load_block<F32_SRC>(xr, b, v);  // (the row is in L1 from the first pass)
            float bmax = 0.f;
#pragma unroll
            for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(v[i]));
            uint32_t sc = 0;
            if (g > 0.f) sc = e4m3_rn_sat(__fdiv_rn(bmax, __fmul_rn(6.0f, g)));
            const float d = __fmul_rn(e4m3_value(sc), g);
            uint32_t w[2] = {0u, 0u};
            if (d > 0.f) {
                const float rcp = __fdiv_rn(1.0f, d);
#pragma unroll
                for (int i = 0; i < 16; i += 2)
                    w[i >> 3] |= e2m1x2_rn_sat(__fmul_rn(v[i], rcp), __fmul_rn(v[i + 1], rcp)) << (8 * ((i >> 1) & 3));
            }
            *reinterpret_cast<uint2 *>(cr + 8 * b) = make_uint2(w[0], w[1]);
            sr[b] = (uint8_t)sc;
        }
        if (lane == 0) glob[pos] = g;
    }
}

cudaError_t launch_quant_nvfp4(const void *src, bool f32_src, int K, const int *sorted_slot, const int *n_pos_dev,
                               int n_pos_static, int n_slots, int top_k, int max_rows, uint8_t *codes,
                               uint8_t *scales, float *glob, cudaStream_t s, int *status)
{
    int blocks = (max_rows + 7) / 8;
    const int bcap = sm_count() * 8;
    if (blocks > bcap) blocks = bcap;
    if (blocks < 1) blocks = 1;
    if (f32_src)
        FT_LAUNCH(quant_nvfp4_rows_kernel<true>, dim3(blocks), dim3(256), 0, s, src, K, sorted_slot, n_pos_dev,
                  n_pos_static, n_slots, top_k, codes, scales, glob, max_rows, status);
    else
        FT_LAUNCH(quant_nvfp4_rows_kernel<false>, dim3(blocks), dim3(256), 0, s, src, K, sorted_slot, n_pos_dev,
                  n_pos_static, n_slots, top_k, codes, scales, glob, max_rows, status);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
