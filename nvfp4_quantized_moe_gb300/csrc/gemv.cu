// Decode-regime grouped GEMV for the NVFP4 experts, on warp-level tensor-core MMAs.
//
// Work unit = (block of 8 expert-sorted slots, group of weight-row tiles). Only the
// experts that own a block are read, so the HBM stream is exactly the touched experts'
// packed codes and scales. A CTA stages the block's 8 activation rows once in shared
// memory as f16, each row scaled by a power of two 2^-e so that its largest magnitude
// lies in [2^14, 2^15) (exact for every bf16 value of normal f16 range; the scale is
// undone on the fp32 accumulator). Each warp then streams a 16-row weight tile with
// 16-byte coalesced loads, prefetched two K steps ahead, dequantises in registers to
// the exact f16 value code*scale (e2m1 and e4m3 values and their products are all
// exact f16 numbers), and feeds m16n8k16 MMAs with fp32 accumulation: weights are
// the M side, the block's tokens the N side. Inside an MMA the K order is permuted
// identically for weights and activations, so each lane reads 32 consecutive elements
// of a row per step.
//
// gate_up (gated): gate rows i and up rows I_l + i of the rank-local bank share a
// warp; the epilogue applies the row globals and SwiGLU h = silu(gate) * up ("[TP=2]
// Quantized MoE expert parallelism ... NVFP4 port", section 4: the MoE output is
// sum_i silu(gate_i) * up_i @ down_i) and stores h in bf16.
// down: the epilogue applies the row global and the routing weight and stores y[slot]
// in fp32; the combine kernel adds the k routed rows of a token in order j = 0..k-1,
// then the shared expert's row.
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "gemv_common.cuh"

#ifndef FTMOE_GEMV_MIN_BLOCKS
#define FTMOE_GEMV_MIN_BLOCKS 2  // resident CTAs per SM the register budget is sized for
#endif

namespace ftmoe {

using namespace gemv;

namespace {

// Codes and scales of one K step for rows g and g+8 of a 16-row tile.
struct Frag {
    uint4 lo, hi;       // 32 codes of row g / row g+8 (16 bytes each)
    uint32_t slo, shi;  // two e4m3 scale bytes (first in the low byte)
};

__device__ __forceinline__ void load_frag(const uint8_t *codes_row_lo, const uint8_t *scales_row_lo, int K, int group,
                                          int kk, int valid, Frag &f)
{
    // valid: elements of the 32-element piece inside K (0, 16 or 32)
    const size_t rs = (size_t)8 * (K / 2);  // 8 rows further
    const size_t ss = (size_t)8 * (K / group);
    if (valid == 32 && (K & 31) == 0) {
        f.lo = ldg_nc_v4(codes_row_lo + kk / 2);
        f.hi = ldg_nc_v4(codes_row_lo + rs + kk / 2);
    } else if (valid > 0) {
        uint2 a = ldg_nc_v2(codes_row_lo + kk / 2), b = ldg_nc_v2(codes_row_lo + rs + kk / 2);
        uint2 a2 = make_uint2(0, 0), b2 = make_uint2(0, 0);
        if (valid == 32) {
            a2 = ldg_nc_v2(codes_row_lo + kk / 2 + 8);
            b2 = ldg_nc_v2(codes_row_lo + rs + kk / 2 + 8);
        }
        f.lo = make_uint4(a.x, a.y, a2.x, a2.y);
        f.hi = make_uint4(b.x, b.y, b2.x, b2.y);
    } else {
        f.lo = f.hi = make_uint4(0, 0, 0, 0);
    }
    if (valid > 0) {
        const int q0 = kk / group, q1 = (kk + 16) / group;
        const uint32_t l0 = __ldg(scales_row_lo + q0), h0 = __ldg(scales_row_lo + ss + q0);
        const uint32_t l1 = (valid == 32) ? (uint32_t)__ldg(scales_row_lo + q1) : l0;
        const uint32_t h1 = (valid == 32) ? (uint32_t)__ldg(scales_row_lo + ss + q1) : h0;
        f.slo = l0 | (l1 << 8);
        f.shi = h0 | (h1 << 8);
    } else {
        f.slo = f.shi = 0x3838;  // 1.0, multiplies zero codes
    }
}

// 8 MMAs of one K step: A from the fragment, B (4 x 16 bytes of f16) from shared memory.
__device__ __forceinline__ void mma_frag(const Frag &f, const uint4 (&b)[4], float (&acc)[4])
{
    mma_step(f.lo, f.hi, f.slo, f.shi, b, acc);
}

}  // namespace

// ---------------------------------------------------------------- gate_up + SwiGLU

// CTA = TPW tile pairs x KS K-splits (TPW * KS = 8 warps). A tile pair is gate rows
// [i0, i0+16) and up rows I_l + [i0, i0+16).
template <int KS>
__global__ void __launch_bounds__(kThreads, FTMOE_GEMV_MIN_BLOCKS) gemv_gated_kernel(const GemvParams p)
{
    pdl_enter();
    constexpr int TPW = 8 / KS;
    extern __shared__ uint4 smem_b[];
    __shared__ float inv[kGemvBlock];
    __shared__ float red[KS > 1 ? 8 : 1][32][8];
    __shared__ int rows[kGemvBlock];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = warp % KS, tp = warp / KS;
    const int g = lane >> 2, c = lane & 3;
    const int Kp = (p.K + kStep - 1) / kStep * kStep;
    const int n_pos = load_n_pos(p);
    const int n_groups = p.n_tiles;  // tile-pair groups per block
    const int n_units = (n_pos / kGemvBlock) * n_groups;
    const int Kw = p.K / KS, k0 = ks * Kw;
    const int n_steps = (Kw + kStep - 1) / kStep;
    const int u_lo = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_hi = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    int staged = -1;
    for (int u = u_lo; u < u_hi; ++u) {
        const int blk = u / n_groups, grp = u - blk * n_groups;
        if (blk != staged) {
            __syncthreads();
            if (threadIdx.x < kGemvBlock) rows[threadIdx.x] = source_row(p, blk * kGemvBlock + threadIdx.x, n_pos, true);
            __syncthreads();
            stage_block(p.act, p.K, Kp, rows, smem_b, inv);
            __syncthreads();
            staged = blk;
        }
        const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + blk) : 0, p.num_experts, p.status);
        const int i0 = (grp * TPW + tp) * 16;
        const bool tile_ok = i0 < p.up_off;
        const uint8_t *gcodes = p.codes + (size_t)e * p.e_codes + (size_t)(i0 + g) * (p.K / 2);
        const uint8_t *gscales = p.scales + (size_t)e * p.e_scales + (size_t)(i0 + g) * (p.K / p.group);
        const uint8_t *ucodes = gcodes + (size_t)p.up_off * (p.K / 2);
        const uint8_t *uscales = gscales + (size_t)p.up_off * (p.K / p.group);
        const uint4 *brow = smem_b + (size_t)g * (Kp / 8);
        float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
        auto piece_k = [&](int s) { return k0 + kStep * s + 32 * c; };
        auto valid = [&](int s) {
            return (tile_ok && s < n_steps) ? max(0, min(32, Kw - (kStep * s + 32 * c))) : 0;
        };
        Frag fg0, fu0, fg1, fu1;
        load_frag(gcodes, gscales, p.K, p.group, piece_k(0), valid(0), fg0);
        load_frag(ucodes, uscales, p.K, p.group, piece_k(0), valid(0), fu0);
        load_frag(gcodes, gscales, p.K, p.group, piece_k(1), valid(1), fg1);
        load_frag(ucodes, uscales, p.K, p.group, piece_k(1), valid(1), fu1);
        for (int s = 0; s < n_steps; s += 2) {
            Frag fg2, fu2, fg3, fu3;
            load_frag(gcodes, gscales, p.K, p.group, piece_k(s + 2), valid(s + 2), fg2);
            load_frag(ucodes, uscales, p.K, p.group, piece_k(s + 2), valid(s + 2), fu2);
            load_frag(gcodes, gscales, p.K, p.group, piece_k(s + 3), valid(s + 3), fg3);
            load_frag(ucodes, uscales, p.K, p.group, piece_k(s + 3), valid(s + 3), fu3);
            uint4 b[4];
            load_b(brow, (k0 + kStep * s) / 8 + 4 * c, g, b);
            mma_frag(fg0, b, accg);
            mma_frag(fu0, b, accu);
            if (s + 1 < n_steps) {
                load_b(brow, (k0 + kStep * (s + 1)) / 8 + 4 * c, g, b);
                mma_frag(fg1, b, accg);
                mma_frag(fu1, b, accu);
            }
            fg0 = fg2; fu0 = fu2; fg1 = fg3; fu1 = fu3;
        }
        if (KS > 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                red[warp][lane][i] = accg[i];
                red[warp][lane][4 + i] = accu[i];
            }
            __syncthreads();
        }
        if (ks == 0 && tile_ok) {
            if (KS > 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float a = 0.f, b2 = 0.f;
                    for (int w = 0; w < KS; ++w) {
                        a += red[tp * KS + w][lane][i];
                        b2 += red[tp * KS + w][lane][4 + i];
                    }
                    accg[i] = a;
                    accu[i] = b2;
                }
            }
            const float *glob_e = p.glob + (size_t)e * p.e_glob;
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int i = i0 + g + 8 * half;
                const float gg = __ldg(glob_e + i), gu = __ldg(glob_e + p.up_off + i);
#pragma unroll
                for (int col = 0; col < 2; ++col) {
                    const int pos = blk * kGemvBlock + 2 * c + col;
                    const float sc = inv[2 * c + col];
                    const float gate = accg[2 * half + col] * sc * gg;
                    const float up = accu[2 * half + col] * sc * gu;
                    __nv_bfloat16 hv = __float2bfloat16_rn(silu(gate) * up);
                    p.h_out[(size_t)pos * p.h_ld + i] = *reinterpret_cast<uint16_t *>(&hv);
                }
            }
        }
        if (KS > 1) __syncthreads();
    }
}

// ---------------------------------------------------------------- down + routing weight

// CTA = TPW row tiles of 16 rows x KS K-splits.
template <int KS>
__global__ void __launch_bounds__(kThreads, FTMOE_GEMV_MIN_BLOCKS) gemv_down_kernel(const GemvParams p)
{
    pdl_enter();
    constexpr int TPW = 8 / KS;
    extern __shared__ uint4 smem_b[];
    __shared__ float inv[kGemvBlock];
    __shared__ float red[KS > 1 ? 8 : 1][32][4];
    __shared__ int rows[kGemvBlock];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = warp % KS, tw = warp / KS;
    const int g = lane >> 2, c = lane & 3;
    const int Kp = (p.K + kStep - 1) / kStep * kStep;
    const int n_pos = load_n_pos(p);
    const int n_groups = p.n_tiles;
    const int n_units = (n_pos / kGemvBlock) * n_groups;
    const int Kw = p.K / KS, k0 = ks * Kw;
    const int n_steps = (Kw + kStep - 1) / kStep;
    const int u_lo = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_hi = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    int staged = -1;
    for (int u = u_lo; u < u_hi; ++u) {
        const int blk = u / n_groups, grp = u - blk * n_groups;
        if (blk != staged) {
            __syncthreads();
            if (threadIdx.x < kGemvBlock) rows[threadIdx.x] = source_row(p, blk * kGemvBlock + threadIdx.x, n_pos, false);
            __syncthreads();
            stage_block(p.act, p.K, Kp, rows, smem_b, inv);
            __syncthreads();
            staged = blk;
        }
        const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + blk) : 0, p.num_experts, p.status);
        const int n0 = (grp * TPW + tw) * 16;
        const bool tile_ok = n0 < p.R;
        const uint8_t *codes = p.codes + (size_t)e * p.e_codes + (size_t)(n0 + g) * (p.K / 2);
        const uint8_t *scales = p.scales + (size_t)e * p.e_scales + (size_t)(n0 + g) * (p.K / p.group);
        const uint4 *brow = smem_b + (size_t)g * (Kp / 8);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        auto piece_k = [&](int s) { return k0 + kStep * s + 32 * c; };
        auto valid = [&](int s) {
            return (tile_ok && s < n_steps) ? max(0, min(32, Kw - (kStep * s + 32 * c))) : 0;
        };
        Frag f0, f1;
        load_frag(codes, scales, p.K, p.group, piece_k(0), valid(0), f0);
        load_frag(codes, scales, p.K, p.group, piece_k(1), valid(1), f1);
        for (int s = 0; s < n_steps; s += 2) {
            Frag f2, f3;
            load_frag(codes, scales, p.K, p.group, piece_k(s + 2), valid(s + 2), f2);
            load_frag(codes, scales, p.K, p.group, piece_k(s + 3), valid(s + 3), f3);
            uint4 b[4];
            load_b(brow, (k0 + kStep * s) / 8 + 4 * c, g, b);
            mma_frag(f0, b, acc);
            if (s + 1 < n_steps) {
                load_b(brow, (k0 + kStep * (s + 1)) / 8 + 4 * c, g, b);
                mma_frag(f1, b, acc);
            }
            f0 = f2; f1 = f3;
        }
        if (KS > 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) red[warp][lane][i] = acc[i];
            __syncthreads();
        }
        if (ks == 0 && tile_ok) {
            if (KS > 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float a = 0.f;
                    for (int w = 0; w < KS; ++w) a += red[tw * KS + w][lane][i];
                    acc[i] = a;
                }
            }
            const float *glob_e = p.glob + (size_t)e * p.e_glob;
#pragma unroll
            for (int col = 0; col < 2; ++col) {
                const int pos = blk * kGemvBlock + 2 * c + col;
                if (pos >= n_pos) continue;
                int dst;
                float wgt = inv[2 * c + col];
                if (p.sorted_slot) {
                    dst = chk_slot(__ldg(p.sorted_slot + pos), p.n_slots, p.status);
                    if (dst >= p.n_slots) continue;
                    if (p.route_w) wgt *= __ldg(p.route_w + dst);
                } else {
                    dst = pos;
                    if (dst >= p.n_pos_static) continue;
                }
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int n = n0 + g + 8 * half;
                    p.y_out[(size_t)dst * p.R + n] = acc[2 * half + col] * __ldg(glob_e + n) * wgt;
                }
            }
        }
        if (KS > 1) __syncthreads();
    }
}

// ---------------------------------------------------------------- combine

// out[t, n] = sum_{j<k} y[t*k + j, n] (+ y_shared[t, n]), in that order.
__global__ void combine_kernel(const float *__restrict__ y, const float *__restrict__ ysh, int T, int k, int H,
                               void *out, int out_dtype)
{
    pdl_enter();
    const int H4 = H / 4;
    size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)T * H4) return;
    const int t = (int)(idx / H4), n4 = (int)(idx % H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    // the shared row first and the routed rows unrolled, so that the loads are in flight
    // together; the additions stay in the order j = 0 .. k-1, then the shared row
    const float4 sh = ysh ? __ldg(reinterpret_cast<const float4 *>(ysh + (size_t)t * H) + n4)
                          : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
    for (int j = 0; j < k; ++j) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(y + ((size_t)t * k + j) * H) + n4);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (ysh) {
        acc.x += sh.x; acc.y += sh.y; acc.z += sh.z; acc.w += sh.w;
    }
    if (out_dtype == FT_DTYPE_F32) {
        reinterpret_cast<float4 *>(static_cast<float *>(out) + (size_t)t * H)[n4] = acc;
    } else {
        __nv_bfloat162 lo = __floats2bfloat162_rn(acc.x, acc.y), hi = __floats2bfloat162_rn(acc.z, acc.w);
        uint2 v;
        v.x = *reinterpret_cast<uint32_t *>(&lo);
        v.y = *reinterpret_cast<uint32_t *>(&hi);
        reinterpret_cast<uint2 *>(static_cast<uint16_t *>(out) + (size_t)t * H)[n4] = v;
    }
}

// ---------------------------------------------------------------- launchers

static size_t stage_bytes(int K) { return (size_t)kGemvBlock * ((K + kStep - 1) / kStep * kStep) * 2; }

template <typename Kern>
static cudaError_t launch_persistent(Kern kern, const GemvParams &p, int max_units, cudaStream_t s)
{
    const size_t smem = stage_bytes(p.K);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int grid = sm_count() * FTMOE_GEMV_MIN_BLOCKS;
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    FT_LAUNCH(kern, dim3(grid), dim3(kThreads), smem, s, p);
    count_launches(1);
    return cudaGetLastError();
}

// K-split so that the unit count covers the GPU: the smallest of 1, 2, 4, 8 with
// enough units, keeping each warp's K range a multiple of the 128-element step.
int gemv_ksplit(int max_blocks, int rows_units_per_block_at_ks1, int K)
{
    const int target = 2 * sm_count();
    int ks = 1;
    while (ks < 8 && max_blocks * rows_units_per_block_at_ks1 * ks < target && (K / (ks * 2)) % kStep == 0 &&
           K / (ks * 2) >= kStep)
        ks *= 2;
    return ks;
}

cudaError_t launch_gemv_gated(const GemvParams &p, int ks, int max_units, cudaStream_t s)
{
    switch (ks) {
    case 1: return launch_persistent(gemv_gated_kernel<1>, p, max_units, s);
    case 2: return launch_persistent(gemv_gated_kernel<2>, p, max_units, s);
    case 4: return launch_persistent(gemv_gated_kernel<4>, p, max_units, s);
    default: return launch_persistent(gemv_gated_kernel<8>, p, max_units, s);
    }
}

cudaError_t launch_gemv_down(const GemvParams &p, int ks, int max_units, cudaStream_t s)
{
    switch (ks) {
    case 1: return launch_persistent(gemv_down_kernel<1>, p, max_units, s);
    case 2: return launch_persistent(gemv_down_kernel<2>, p, max_units, s);
    case 4: return launch_persistent(gemv_down_kernel<4>, p, max_units, s);
    default: return launch_persistent(gemv_down_kernel<8>, p, max_units, s);
    }
}

cudaError_t launch_combine(const float *y, const float *y_shared, int T, int k, int H, void *out, int out_dtype,
                           cudaStream_t s)
{
    const size_t n = (size_t)T * (H / 4);
    const int threads = 256;
    FT_LAUNCH(combine_kernel, dim3((unsigned)((n + threads - 1) / threads)), dim3(threads), 0, s, y, y_shared,
              T, k, H, out, out_dtype);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
