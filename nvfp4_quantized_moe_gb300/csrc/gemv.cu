// Decode-regime grouped GEMV for the NVFP4 experts, on warp-level tensor-core MMAs.
//
// Work unit = (block of 8 expert-sorted slots, tile of 16 weight rows). Only the
// experts that own a block are ever read, so the HBM stream is the touched experts'
// packed codes and scales. Each warp multiplies a 16-row tile against the block's
// activation rows over a K range: the packed codes are loaded with 8-byte
// coalesced loads, dequantised in registers to exact bf16 code*scale values, and fed
// to m16n8k16 MMAs with fp32 accumulation (weights as M, tokens as N). The K order
// inside an MMA is permuted identically for weights and activations so that each
// lane reads 16 consecutive elements (one block scale) per step.
//
// gate_up (gated): rows i and I_l+i of the rank-local gate_up bank share a warp, the
// epilogue applies the per-row globals and SwiGLU h = silu(gate)*up ("[TP=2]
// Quantized MoE expert parallelism ... NVFP4 port", section 4: MoE output =
// sum_i silu(gate_i)*up_i @ down_i) and stores h in bf16.
// down: the epilogue applies the per-row global and the routing weight and stores
// y[slot] in fp32; the combine kernel then adds the k routed rows of a token in
// order j = 0..k-1 and the shared expert's row.
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {

namespace {

struct BlockInfo {
    int expert;
    int n_pos;
};

__device__ __forceinline__ int load_n_pos(const GemvParams &p)
{
    return p.n_pos_dev ? *p.n_pos_dev : (p.n_pos_static + kGemvBlock - 1) / kGemvBlock * kGemvBlock;
}

// Activation row for block position `pos`, or -1 when the position is padding.
__device__ __forceinline__ int act_row_gated(const GemvParams &p, int pos, int n_pos)
{
    if (pos >= n_pos) return -1;
    if (p.sorted_slot) {
        int s = __ldg(p.sorted_slot + pos);
        return (s < p.n_slots) ? s / p.top_k : -1;
    }
    return (pos < p.n_pos_static) ? pos : -1;
}

__device__ __forceinline__ int act_row_down(const GemvParams &p, int pos, int n_pos)
{
    if (pos >= n_pos) return -1;
    if (p.sorted_slot) return (__ldg(p.sorted_slot + pos) < p.n_slots) ? pos : -1;
    return (pos < p.n_pos_static) ? pos : -1;
}

// One K step of a 16-row tile: lane (g = lane/4, c = lane%4) holds rows g and g+8,
// elements [kk, kk+16) of its piece, and the activation row of block column g.
struct TileStep {
    uint2 c_lo, c_hi;  // codes of rows g and g+8 (8 bytes each)
    uint32_t s_lo, s_hi;
};

__device__ __forceinline__ void load_tile_step(const uint8_t *codes_e, const uint8_t *scales_e, int K, int group,
                                               int row, int kk, bool ok, TileStep &st)
{
    if (ok) {
        st.c_lo = ldg_nc_v2(codes_e + (size_t)row * (K / 2) + kk / 2);
        st.c_hi = ldg_nc_v2(codes_e + (size_t)(row + 8) * (K / 2) + kk / 2);
        st.s_lo = __ldg(scales_e + (size_t)row * (K / group) + kk / group);
        st.s_hi = __ldg(scales_e + (size_t)(row + 8) * (K / group) + kk / group);
    } else {
        st.c_lo = make_uint2(0, 0);
        st.c_hi = make_uint2(0, 0);
        st.s_lo = st.s_hi = 0x38;  // 1.0, multiplies zero codes
    }
}

__device__ __forceinline__ void mma_tile_step(const TileStep &st, const uint32_t (&b)[8], float (&acc)[4])
{
    uint32_t sl, sh;
    e4m3x2_to_bf16x2_scaled(st.s_lo | (st.s_hi << 8), sl, sh);
    uint32_t lo[8], hi[8];
    {
        uint32_t t[4];
        dequant8(st.c_lo.x, sl, t);
        lo[0] = t[0]; lo[1] = t[1]; lo[2] = t[2]; lo[3] = t[3];
        dequant8(st.c_lo.y, sl, t);
        lo[4] = t[0]; lo[5] = t[1]; lo[6] = t[2]; lo[7] = t[3];
        dequant8(st.c_hi.x, sh, t);
        hi[0] = t[0]; hi[1] = t[1]; hi[2] = t[2]; hi[3] = t[3];
        dequant8(st.c_hi.y, sh, t);
        hi[4] = t[0]; hi[5] = t[1]; hi[6] = t[2]; hi[7] = t[3];
    }
#pragma unroll
    for (int j = 0; j < 4; ++j)
        mma_bf16_16816(acc, lo[2 * j], hi[2 * j], lo[2 * j + 1], hi[2 * j + 1], b[2 * j], b[2 * j + 1]);
}

__device__ __forceinline__ void load_act(const uint16_t *act, int K, int row, int kk, bool ok, uint32_t (&b)[8])
{
    if (ok && row >= 0) {
        const uint4 *src = reinterpret_cast<const uint4 *>(act + (size_t)row * K + kk);
        uint4 v0 = __ldg(src), v1 = __ldg(src + 1);
        b[0] = v0.x; b[1] = v0.y; b[2] = v0.z; b[3] = v0.w;
        b[4] = v1.x; b[5] = v1.y; b[6] = v1.z; b[7] = v1.w;
    } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) b[i] = 0;
    }
}

constexpr int kUnroll = 4;

}  // namespace

// ---------------------------------------------------------------- gate_up + SwiGLU

// CTA = KSPLIT warps on one tile pair (gate rows [i0, i0+16), up rows I_l + same).
template <int KSPLIT>
__global__ void __launch_bounds__(KSPLIT * 32) gemv_gated_kernel(const GemvParams p)
{
    __shared__ float red[KSPLIT][32][8];
    const int lane = threadIdx.x & 31, ks = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int n_pos = load_n_pos(p);
    const int n_units = (n_pos / kGemvBlock) * p.n_tiles;
    const int Kw = p.K / KSPLIT, k0 = ks * Kw;
    const int n_steps = (Kw + 63) / 64;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int blk = u / p.n_tiles, tile = u - blk * p.n_tiles;
        const int e = p.block_expert ? __ldg(p.block_expert + blk) : 0;
        const int i0 = tile * 16;
        const uint8_t *codes_e = p.codes + (size_t)e * p.e_codes;
        const uint8_t *scales_e = p.scales + (size_t)e * p.e_scales;
        const int arow = act_row_gated(p, blk * kGemvBlock + g, n_pos);
        float accg[4] = {0.f, 0.f, 0.f, 0.f}, accu[4] = {0.f, 0.f, 0.f, 0.f};
        for (int s0 = 0; s0 < n_steps; s0 += kUnroll) {
            TileStep sg[kUnroll], su[kUnroll];
            uint32_t b[kUnroll][8];
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int piece = 4 * (s0 + q) + c;
                const bool ok = (s0 + q) < n_steps && 16 * piece < Kw;
                const int kk = k0 + 16 * piece;
                load_tile_step(codes_e, scales_e, p.K, p.group, i0 + g, kk, ok, sg[q]);
                load_tile_step(codes_e, scales_e, p.K, p.group, p.up_off + i0 + g, kk, ok, su[q]);
                load_act(p.act, p.K, arow, kk, ok, b[q]);
            }
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                mma_tile_step(sg[q], b[q], accg);
                mma_tile_step(su[q], b[q], accu);
            }
        }
        if (KSPLIT > 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                red[ks][lane][i] = accg[i];
                red[ks][lane][4 + i] = accu[i];
            }
            __syncthreads();
        }
        if (ks == 0) {
            if (KSPLIT > 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float a = 0.f, b2 = 0.f;
                    for (int w = 0; w < KSPLIT; ++w) {
                        a += red[w][lane][i];
                        b2 += red[w][lane][4 + i];
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
                    if (pos < n_pos) {
                        const float gate = accg[2 * half + col] * gg;
                        const float up = accu[2 * half + col] * gu;
                        __nv_bfloat16 hv = __float2bfloat16_rn(silu(gate) * up);
                        p.h_out[(size_t)pos * p.h_ld + i] = *reinterpret_cast<uint16_t *>(&hv);
                    }
                }
            }
        }
        if (KSPLIT > 1) __syncthreads();
    }
}

// ---------------------------------------------------------------- down + routing weight

// CTA = (8 / KSPLIT) row tiles x KSPLIT K-splits.
template <int KSPLIT>
__global__ void __launch_bounds__(256) gemv_down_kernel(const GemvParams p)
{
    constexpr int TPC = 8 / KSPLIT;
    __shared__ float red[8][32][4];
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = warp % KSPLIT, tw = warp / KSPLIT;
    const int g = lane >> 2, c = lane & 3;
    const int n_pos = load_n_pos(p);
    const int n_units = (n_pos / kGemvBlock) * p.n_tiles;
    const int Kw = p.K / KSPLIT, k0 = ks * Kw;
    const int n_steps = (Kw + 63) / 64;
    for (int u = blockIdx.x; u < n_units; u += gridDim.x) {
        const int blk = u / p.n_tiles, tile = u - blk * p.n_tiles;
        const int e = p.block_expert ? __ldg(p.block_expert + blk) : 0;
        const int n0 = (tile * TPC + tw) * 16;
        const bool tile_ok = n0 < p.R;
        const uint8_t *codes_e = p.codes + (size_t)e * p.e_codes;
        const uint8_t *scales_e = p.scales + (size_t)e * p.e_scales;
        const int arow = act_row_down(p, blk * kGemvBlock + g, n_pos);
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int s0 = 0; s0 < n_steps; s0 += kUnroll) {
            TileStep st[kUnroll];
            uint32_t b[kUnroll][8];
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) {
                const int piece = 4 * (s0 + q) + c;
                const bool ok = tile_ok && (s0 + q) < n_steps && 16 * piece < Kw;
                const int kk = k0 + 16 * piece;
                load_tile_step(codes_e, scales_e, p.K, p.group, n0 + g, kk, ok, st[q]);
                load_act(p.act, p.K, arow, kk, ok, b[q]);
            }
#pragma unroll
            for (int q = 0; q < kUnroll; ++q) mma_tile_step(st[q], b[q], acc);
        }
        if (KSPLIT > 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) red[warp][lane][i] = acc[i];
            __syncthreads();
        }
        if (ks == 0 && tile_ok) {
            if (KSPLIT > 1) {
#pragma unroll
                for (int i = 0; i < 4; ++i) {
                    float a = 0.f;
                    for (int w = 0; w < KSPLIT; ++w) a += red[tw * KSPLIT + w][lane][i];
                    acc[i] = a;
                }
            }
            const float *glob_e = p.glob + (size_t)e * p.e_glob;
#pragma unroll
            for (int col = 0; col < 2; ++col) {
                const int pos = blk * kGemvBlock + 2 * c + col;
                if (pos >= n_pos) continue;
                int dst;
                float wgt = 1.0f;
                if (p.sorted_slot) {
                    dst = __ldg(p.sorted_slot + pos);
                    if (dst >= p.n_slots) continue;
                    if (p.route_w) wgt = __ldg(p.route_w + dst);
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
        if (KSPLIT > 1) __syncthreads();
    }
}

// ---------------------------------------------------------------- combine

// out[t, n] = sum_{j<k} y[t*k + j, n] (+ y_shared[t, n]), in that order.
__global__ void combine_kernel(const float *__restrict__ y, const float *__restrict__ ysh, int T, int k, int H,
                               void *out, int out_dtype)
{
    const int H4 = H / 4;
    size_t idx = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (idx >= (size_t)T * H4) return;
    const int t = (int)(idx / H4), n4 = (int)(idx % H4);
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    for (int j = 0; j < k; ++j) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(y + ((size_t)t * k + j) * H) + n4);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
    }
    if (ysh) {
        float4 v = __ldg(reinterpret_cast<const float4 *>(ysh + (size_t)t * H) + n4);
        acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
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

static int grid_for(int max_units, int per_sm)
{
    int g = sm_count() * per_sm;
    if (max_units < g) g = max_units;
    return g < 1 ? 1 : g;
}

cudaError_t launch_gemv_gated(const GemvParams &p, int max_units, cudaStream_t s)
{
    gemv_gated_kernel<8><<<grid_for(max_units, 4), 256, 0, s>>>(p);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_gemv_down(const GemvParams &p, int ksplit, int max_units, cudaStream_t s)
{
    const int grid = grid_for(max_units, 4);
    switch (ksplit) {
    case 1: gemv_down_kernel<1><<<grid, 256, 0, s>>>(p); break;
    case 2: gemv_down_kernel<2><<<grid, 256, 0, s>>>(p); break;
    case 4: gemv_down_kernel<4><<<grid, 256, 0, s>>>(p); break;
    default: gemv_down_kernel<8><<<grid, 256, 0, s>>>(p); break;
    }
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_combine(const float *y, const float *y_shared, int T, int k, int H, void *out, int out_dtype,
                           cudaStream_t s)
{
    const size_t n = (size_t)T * (H / 4);
    const int threads = 256;
    combine_kernel<<<(unsigned)((n + threads - 1) / threads), threads, 0, s>>>(y, y_shared, T, k, H, out, out_dtype);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
