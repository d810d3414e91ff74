// Router logits of the replicated router: logits[t][e] = sum_h x[t][h] * W[e][h] over
// bf16 x [T][H] and W [E][H], fp32 accumulation ("[1/3] feat(dsv4): add tensor-parallel
// DeepSeek-V4 runtime", table "Tensor ownership and collectives": the router is
// replicated and every rank computes the same routing). The top-k step then runs on
// these logits exactly as for given logits.
//
// m16n8k16 bf16 MMAs with the router rows as M and tokens as N. A CTA owns 16 rows x
// 8 NJ tokens (NJ = 4, or 1 for small batches so that the grid covers the GPU); its warps
// split K and walk it in 32-element chunks; within a chunk lane
// (g, c) loads the 8 consecutive elements 8c .. 8c+7 of its rows (16 bytes) and of its
// tokens, and the two MMAs of the chunk take elements 8c..8c+3 and 8c+4..8c+7: the same
// K permutation for both operands, so every lane reads contiguous 16-byte pieces.
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {

namespace {

constexpr int kRgWarps = 16;  // warps per CTA, splitting K
constexpr int kGroup = 2;     // 32-element chunks whose loads are issued together

// One CTA = one tile of 16 router rows x 8 NJ tokens; its ks warps (ks a power of two up
// to 16) take equal K ranges, issue the loads of two 32-element chunks at a time, and
// the partial sums are added in warp order.
template <int NJ>
__global__ void __launch_bounds__(32 * kRgWarps) router_gemm_kernel(const uint16_t *__restrict__ x,
                                                                   const uint16_t *__restrict__ w, int T, int H,
                                                                   int E, int ks, float *__restrict__ logits)
{
    pdl_enter();
    constexpr int kRgTok = 8 * NJ;
    __shared__ float red[kRgWarps][4 * NJ][32];
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31, g = lane >> 2, c = lane & 3;
    const int n_rt = (E + 15) / 16;
    const int rt = blockIdx.x % n_rt, tt = blockIdx.x / n_rt;
    const int e0 = rt * 16, t0 = tt * kRgTok;
    float acc[NJ][4] = {};
    {
        const int kw = H / ks, kb = warp * kw;
        // rows past E (last tile of an E not a multiple of 16) read a valid row; not stored
        const int ea = e0 + g < E ? e0 + g : E - 1, eb = e0 + g + 8 < E ? e0 + g + 8 : E - 1;
        const uint16_t *a_lo = w + (size_t)ea * H + kb + 8 * c;
        const uint16_t *a_hi = w + (size_t)eb * H + kb + 8 * c;
        const uint16_t *b[NJ];
#pragma unroll
        for (int j = 0; j < NJ; ++j) {
            int t = t0 + 8 * j + g;
            if (t > T - 1) t = T - 1;  // tail tokens read a valid row; their results are not stored
            b[j] = x + (size_t)t * H + kb + 8 * c;
        }
        // chunks in groups of kGroup: all loads of a group are issued before its MMAs
        for (int kg = 0; kg < kw; kg += kGroup * 32) {
            uint4 lo[kGroup], hi[kGroup], bv[kGroup][NJ];
#pragma unroll
            for (int q = 0; q < kGroup; ++q) {
                const int k0 = kg + 32 * q;
                if (k0 < kw) {
                    lo[q] = ldg_nc_v4(a_lo + k0);
                    hi[q] = ldg_nc_v4(a_hi + k0);
#pragma unroll
                    for (int j = 0; j < NJ; ++j) bv[q][j] = ldg_nc_v4(b[j] + k0);
                }
            }
#pragma unroll
            for (int q = 0; q < kGroup; ++q) {
                if (kg + 32 * q >= kw) break;
#pragma unroll
                for (int j = 0; j < NJ; ++j) {
                    mma_bf16_16816(acc[j], lo[q].x, hi[q].x, lo[q].y, hi[q].y, bv[q][j].x, bv[q][j].y);
                    mma_bf16_16816(acc[j], lo[q].z, hi[q].z, lo[q].w, hi[q].w, bv[q][j].z, bv[q][j].w);
                }
            }
        }
    }
#pragma unroll
    for (int j = 0; j < NJ; ++j)
#pragma unroll
        for (int i = 0; i < 4; ++i) red[warp][4 * j + i][lane] = acc[j][i];
    __syncthreads();
    if (warp != 0) return;
    // D fragment: rows g, g+8 (router rows), columns 2c, 2c+1 (tokens) of each tile
#pragma unroll
    for (int j = 0; j < NJ; ++j) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            float v = 0.f;
            for (int q = 0; q < ks; ++q) v += red[q][4 * j + i][lane];
            const int t = t0 + 8 * j + 2 * c + (i & 1), e = e0 + g + 8 * (i >> 1);
            if (t < T && e < E) logits[(size_t)t * E + e] = v;
        }
    }
}

}  // namespace

cudaError_t launch_router_gemm(const uint16_t *x, const uint16_t *w, int T, int H, int E, float *logits,
                               cudaStream_t s)
{
    // K split: at least 8 warps per tile (their chunk loads overlap), 16 while the grid is
    // small, as long as every K range stays a multiple of 32
    // tokens per tile: 32, or 8 while 32-token tiles would leave most SMs idle
    const int rows = (E + 15) / 16;
    const int nj = rows * ((T + 31) / 32) >= sm_count() ? 4 : 1;
    const int tiles = rows * ((T + 8 * nj - 1) / (8 * nj));
    int ks = 1;
    while (ks < kRgWarps && (ks < 8 || tiles * ks < 4 * sm_count()) && H % (64 * ks) == 0) ks <<= 1;
    if (nj == 4)
        FT_LAUNCH(router_gemm_kernel<4>, dim3(tiles), dim3(32 * ks), 0, s, x, w, T, H, E, ks, logits);
    else
        FT_LAUNCH(router_gemm_kernel<1>, dim3(tiles), dim3(32 * ks), 0, s, x, w, T, H, E, ks, logits);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
