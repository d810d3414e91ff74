// Pieces shared by the two decode-regime GEMV kernels (register-fed and bulk-copy-fed).
#pragma once

#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {
namespace gemv {

constexpr int kThreads = 256;  // 8 warps per CTA
constexpr int kStep = 128;     // K elements per warp step (4 lanes x 32)

__device__ __forceinline__ int load_n_pos(const GemvParams &p)
{
    return p.n_pos_dev ? chk_count(*p.n_pos_dev, kGemvBlock, padded_capacity(p.n_slots, p.num_experts, kGemvBlock),
                                   p.status)
                       : (p.n_pos_static + kGemvBlock - 1) / kGemvBlock * kGemvBlock;
}

// Source row of block position `pos` (x row for gate_up, h row for down), or -1 for padding.
__device__ __forceinline__ int source_row(const GemvParams &p, int pos, int n_pos, bool gated)
{
    if (pos >= n_pos) return -1;
    if (p.sorted_slot) {
        const int s = chk_slot(__ldg(p.sorted_slot + pos), p.n_slots, p.status);
        if (s >= p.n_slots) return -1;
        return gated ? s / p.top_k : pos;
    }
    return (pos < p.n_pos_static) ? pos : -1;
}

// Physical 16-byte chunk of logical chunk q in staged row r. With a row pitch that is a
// multiple of 128 bytes, the 8 lanes of each LDS.128 phase (rows 2m, 2m+1; lanes c = 0..3
// reading chunks base + 4c + j) land in 8 distinct bank quads.
__device__ __forceinline__ int swz(int q, int r) { return q ^ (((q >> 3) & 1) << 1) ^ (r & 1); }

// Stage the block's 8 activation rows (bf16, length K) into shared memory as f16 scaled
// by 2^-e_r; inv[r] = 2^e_r. Warp r handles row r. The row pitch is Kp >= K elements
// (a multiple of kStep) and the tail [K, Kp) is zero.
__device__ __forceinline__ void stage_row(const uint16_t *__restrict__ src, int K, int Kp, const int *rows, uint4 *sm,
                                          float *inv, int r)
{
    const int lane = threadIdx.x & 31;
    const int row = rows[r];
    uint4 *dst = sm + (size_t)r * (Kp / 8);
    if (row < 0) {
        for (int q = lane; q < Kp / 8; q += 32) dst[swz(q, r)] = make_uint4(0, 0, 0, 0);
        if (lane == 0) inv[r] = 0.f;
        return;
    }
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src + (size_t)row * K);
    float m = 0.f;
    for (int q = lane; q < K / 8; q += 32) {
        const uint4 v = __ldg(s4 + q);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            m = fmaxf(m, fabsf(__uint_as_float(w[i] << 16)));
            m = fmaxf(m, fabsf(__uint_as_float(w[i] & 0xFFFF0000u)));
        }
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    const int e = row_scale_exp(m);
    const float down = pow2f(-e);
    for (int q = lane; q < Kp / 8; q += 32) {
        uint4 o = make_uint4(0, 0, 0, 0);
        if (q < K / 8) {
            const uint4 v = __ldg(s4 + q);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half2 hh = __floats2half2_rn(__uint_as_float(w[i] << 16) * down,
                                                     __uint_as_float(w[i] & 0xFFFF0000u) * down);
                h[i] = *reinterpret_cast<const uint32_t *>(&hh);
            }
            o = make_uint4(h[0], h[1], h[2], h[3]);
        }
        dst[swz(q, r)] = o;
    }
    if (lane == 0) inv[r] = pow2f(e);
}

// The same with Kp = K and a single pass over global memory: the raw bf16 pieces go to
// their final shared-memory places while the maximum is taken, then each lane converts
// its own pieces in place. COHERENT: the rows were written by other CTAs of the same
// launch (after an acquire), so they are read through L2 rather than the read-only path.
template <bool COHERENT = false>
__device__ __forceinline__ void stage_row_1pass(const uint16_t *__restrict__ src, int K, const int *rows, uint4 *sm,
                                                float *inv, int r)
{
    const int lane = threadIdx.x & 31;
    const int row = rows[r];
    uint4 *dst = sm + (size_t)r * (K / 8);
    const int nq = K / 8;
    if (row < 0) {
        for (int q = lane; q < nq; q += 32) dst[swz(q, r)] = make_uint4(0, 0, 0, 0);
        if (lane == 0) inv[r] = 0.f;
        return;
    }
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src + (size_t)row * K);
    float m = 0.f;
#pragma unroll 4
    for (int q = lane; q < nq; q += 32) {
        const uint4 v = COHERENT ? __ldcg(s4 + q) : __ldg(s4 + q);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            m = fmaxf(m, fabsf(__uint_as_float(w[j] << 16)));
            m = fmaxf(m, fabsf(__uint_as_float(w[j] & 0xFFFF0000u)));
        }
        dst[swz(q, r)] = v;
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    const int e = row_scale_exp(m);
    const float down = pow2f(-e);
    for (int q = lane; q < nq; q += 32) {
        const uint4 v = dst[swz(q, r)];
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[4];
#pragma unroll
        for (int j = 0; j < 4; ++j) {
            const __half2 hh = __floats2half2_rn(__uint_as_float(w[j] << 16) * down,
                                                 __uint_as_float(w[j] & 0xFFFF0000u) * down);
            h[j] = *reinterpret_cast<const uint32_t *>(&hh);
        }
        dst[swz(q, r)] = make_uint4(h[0], h[1], h[2], h[3]);
    }
    if (lane == 0) inv[r] = pow2f(e);
}

// Stage all 8 rows of the block: warp w handles rows w, w + nwarps, ...
__device__ __forceinline__ void stage_block(const uint16_t *__restrict__ src, int K, int Kp, const int *rows,
                                            uint4 *sm, float *inv)
{
    const int nwarps = blockDim.x >> 5;
    for (int r = threadIdx.x >> 5; r < kGemvBlock; r += nwarps) stage_row(src, K, Kp, rows, sm, inv, r);
}

// One 128-element K step of one 16-row tile for lane (g, c): 32 codes of rows g and
// g+8 (16 bytes each), their two scale bytes (first in the low byte), and the block's
// activations for the same 32 elements (4 x 16 bytes of f16, token g). 8 MMAs.
__device__ __forceinline__ void mma_step(const uint4 &lo, const uint4 &hi, uint32_t slo, uint32_t shi,
                                         const uint4 (&b)[4], float (&acc)[4])
{
    uint32_t s_lo[2], s_hi[2];
    e4m3x2_to_f16x2_bcast(slo, s_lo[0], s_lo[1]);
    e4m3x2_to_f16x2_bcast(shi, s_hi[0], s_hi[1]);
    const uint32_t cl[4] = {lo.x, lo.y, lo.z, lo.w};
    const uint32_t ch[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int w = 0; w < 4; ++w) {  // 8 elements per code word; words 0,1 use scale 0, words 2,3 scale 1
        uint32_t al[4], ah[4];
        dequant8_f16(cl[w], s_lo[w >> 1], al);
        dequant8_f16(ch[w], s_hi[w >> 1], ah);
        const uint32_t bw[4] = {b[w].x, b[w].y, b[w].z, b[w].w};
        mma_f16_16816(acc, al[0], ah[0], al[1], ah[1], bw[0], bw[1]);
        mma_f16_16816(acc, al[2], ah[2], al[3], ah[3], bw[2], bw[3]);
    }
}

// Activations of token g for the 32 elements starting at 16-byte chunk q0.
__device__ __forceinline__ void load_b(const uint4 *sm_row, int q0, int r, uint4 (&b)[4])
{
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = sm_row[swz(q0 + j, r)];
}

}  // namespace gemv
}  // namespace ftmoe
