// Grouped GEMV for fp8_block experts (every batch size): W[n][k] = e4m3(code[n][k]) *
// scale_inv[n/128][k/128], one code byte per weight ("feat(qwen3_5_moe): tensor-parallel
// weight sharding", Implementation notes: an fp8-block weight carries a 128-block
// weight_scale_inv; the dsv4 PR, Checkpoint loading: FP8 128x128 blocks).
//
// Structure of the register-fed NVFP4 decode kernel: weights as M, a block of 8
// expert-sorted positions as N, m16n8k16 f16 MMAs with fp32 accumulation, each warp
// owning two 16-row tiles (gate rows i and up rows I_l + i for gate_up, so SwiGLU fuses;
// rows n and n + 16 for down), loads running two steps ahead through a 4-slot register
// ring, routed and shared expert in one launch; the ordered combine runs as its own launch.
// What differs:
//  * a step is 64 K elements: lane (g, c) loads 16 code bytes of rows g and g + 8 of
//    each tile (K elements 16c .. 16c + 15 of the step); e4m3 converts to f16 exactly
//    (cvt.rn.f16x2.e4m3x2), two codes per instruction, with no scale multiply;
//  * the 16 K elements of a lane are spread over the step's four MMAs (MMA j takes
//    16c + 4j .. 16c + 4j + 3 of every lane c), the same permutation of K for both
//    operands, so the activations are read as two contiguous 16-byte pieces per lane;
//  * a 16-row tile lies inside one 128-row scale block and two steps make one 128-K
//    block, so each tile accumulates a block's MMAs into a fresh fp32 partial that is
//    added to the running sum times the block's scale_inv (exact fp32 arithmetic; no
//    global, and nothing folded into the f16 operands);
//  * activation rows are staged (f16, scaled by a power of two per row, as in the
//    NVFP4 kernels) with a 16-byte row padding that makes the reads conflict-free.
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "gemv_common.cuh"

namespace ftmoe {

using namespace gemv;

namespace {

constexpr int kStep8 = 64;  // K elements per warp step

struct Fp8Frag {
    uint4 a_lo, a_hi, b_lo, b_hi;  // codes: tile 0 rows g / g+8, tile 1 rows g / g+8
};

__device__ __forceinline__ uint32_t e4m3x2_f16x2(uint32_t two_bytes)
{
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}" : "=r"(h2) : "r"(two_bytes));
    return h2;
}

// The four MMAs of one step for one tile: word j of each row's 16 code bytes holds the
// K elements 4j .. 4j + 3 of the lane's range; the activations of token g for the same
// elements are words 2j, 2j + 1 of b.
__device__ __forceinline__ void fp8_tile_step(const uint4 &lo, const uint4 &hi, const uint32_t (&b)[8],
                                              float (&acc)[4])
{
    const uint32_t cl[4] = {lo.x, lo.y, lo.z, lo.w};
    const uint32_t ch[4] = {hi.x, hi.y, hi.z, hi.w};
#pragma unroll
    for (int j = 0; j < 4; ++j) {
        const uint32_t a0 = e4m3x2_f16x2(cl[j]), a2 = e4m3x2_f16x2(cl[j] >> 16);
        const uint32_t a1 = e4m3x2_f16x2(ch[j]), a3 = e4m3x2_f16x2(ch[j] >> 16);
        mma_f16_16816(acc, a0, a1, a2, a3, b[2 * j], b[2 * j + 1]);
    }
}

// Stage the block's 8 activation rows: f16 of x * 2^-e_r (row maximum in [2^14, 2^15)),
// row pitch K + 8 elements; inv[r] = 2^e_r (0 for padding rows, which are zero).
__device__ __forceinline__ void fp8_stage(const GemvParams &p, int blk, int n_pos, bool gated, int *rows,
                                          uint4 *sm, float *inv)
{
    __syncthreads();
    if (threadIdx.x < kGemvBlock) rows[threadIdx.x] = source_row(p, blk * kGemvBlock + threadIdx.x, n_pos, gated);
    __syncthreads();
    const int lane = threadIdx.x & 31, K = p.K, pitch = K / 8 + 1;
    for (int r = threadIdx.x >> 5; r < kGemvBlock; r += blockDim.x >> 5) {
        const int row = rows[r];
        uint4 *dst = sm + (size_t)r * pitch;
        if (row < 0) {
            for (int q = lane; q < K / 8; q += 32) dst[q] = make_uint4(0, 0, 0, 0);
            if (lane == 0) inv[r] = 0.f;
            continue;
        }
        const uint4 *s4 = reinterpret_cast<const uint4 *>(p.act + (size_t)row * K);
        float m = 0.f;
        for (int q = lane; q < K / 8; q += 32) {
            const uint4 v = __ldg(s4 + q);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i)
                m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
        const int e = row_scale_exp(m);
        const float down = pow2f(-e);
        for (int q = lane; q < K / 8; q += 32) {
            const uint4 v = __ldg(s4 + q);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
            uint32_t h[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                const __half2 hh = __floats2half2_rn(__uint_as_float(w[i] << 16) * down,
                                                     __uint_as_float(w[i] & 0xFFFF0000u) * down);
                h[i] = *reinterpret_cast<const uint32_t *>(&hh);
            }
            dst[q] = make_uint4(h[0], h[1], h[2], h[3]);
        }
        if (lane == 0) inv[r] = pow2f(e);
    }
    __syncthreads();
}

// One unit: block `blk` of problem p, pair tiles (group `grp` of TPW per CTA) over the
// warp's K range (K split KS ways across the CTA's warps, partials added in warp order),
// or, with KS = 1, over its 64-K steps [s_lo, s_hi) only (both even: whole scale blocks)
// when the unit is split between CTAs c - 1 and c (piece 1, this CTA is c) or c and c + 1
// (piece 0): the pieces' partial sums meet in split slot c - piece and the second of the
// two CTAs to finish adds the other piece (a sum of two fp32 terms does not depend on
// their order) and runs the epilogue.
template <bool GATED, int KS>
__device__ __forceinline__ void fp8_unit(const GemvParams &p, const FastLaunch &L, int lu, int n_pos,
                                         const uint4 *smem_b, const float *inv,
                                         float (&red)[KS > 1 ? 8 : 1][32][8], int s_lo = 0, int s_hi = -1,
                                         int piece = -1)
{
    constexpr int TPW = 8 / KS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = warp % KS, tp = warp / KS;
    const int g = lane >> 2, c = lane & 3;
    const int K = p.K, kb_n = K / 128;
    const int blk = lu / p.n_tiles, grp = lu - blk * p.n_tiles;
    const int Kw = K / KS, k0 = ks * Kw;
    if (s_hi < 0) s_hi = Kw / kStep8;
    const int nstep = s_hi - s_lo;
    const int pair_rows = GATED ? 16 : 32;
    const int rows_limit = GATED ? p.up_off : p.R;
    const int r0 = (grp * TPW + tp) * pair_rows;
    const bool ok = r0 < rows_limit;
    const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + blk) : 0, p.num_experts, p.status);
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
        const int row_a = r0 + g, row_b = GATED ? p.up_off + r0 + g : r0 + 16 + g;
        const uint8_t *codes_e = p.codes + (size_t)e * p.e_codes;
        const uint8_t *ca = codes_e + (size_t)row_a * K + k0 + 16 * c;
        const uint8_t *cb = codes_e + (size_t)row_b * K + k0 + 16 * c;
        const size_t row8 = (size_t)8 * K;
        // scale_inv rows of the two tiles (each tile lies inside one 128-row block)
        const float *sinv_e = p.sinv + (size_t)e * p.e_sinv;
        const float *sa = sinv_e + (size_t)((r0) / 128) * kb_n + k0 / 128;
        const float *sb = sinv_e + (size_t)((GATED ? p.up_off + r0 : r0 + 16) / 128) * kb_n + k0 / 128;
        const uint4 *bb = smem_b + (size_t)g * (K / 8 + 1) + k0 / 8 + 2 * c;
        auto load = [&](int s, Fp8Frag &f) {
            const int off = (s_lo + s) * kStep8;
            f.a_lo = ldg_nc_v4(ca + off);
            f.a_hi = ldg_nc_v4(ca + row8 + off);
            f.b_lo = ldg_nc_v4(cb + off);
            f.b_hi = ldg_nc_v4(cb + row8 + off);
        };
        float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};  // current 128-K block
        Fp8Frag ring[4];
        load(0, ring[0]);
        if (nstep > 1) load(1, ring[1]);
        for (int s0 = 0; s0 < nstep; s0 += 4) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int s = s0 + q;
                if (s + 2 < nstep) load(s + 2, ring[(q + 2) & 3]);
                if (s < nstep) {
                    const uint4 x0 = bb[8 * (s_lo + s)], x1 = bb[8 * (s_lo + s) + 1];
                    const uint32_t b[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                    fp8_tile_step(ring[q].a_lo, ring[q].a_hi, b, t0);
                    fp8_tile_step(ring[q].b_lo, ring[q].b_hi, b, t1);
                    if (q & 1) {  // end of a 128-K block (steps are 64 K; ranges start on a block)
                        const float fa = __ldg(sa + ((s_lo + s) >> 1)), fb = __ldg(sb + ((s_lo + s) >> 1));
#pragma unroll
                        for (int i = 0; i < 4; ++i) {
                            acc0[i] = fmaf(fa, t0[i], acc0[i]);
                            acc1[i] = fmaf(fb, t1[i], acc1[i]);
                            t0[i] = 0.f;
                            t1[i] = 0.f;
                        }
                    }
                }
            }
        }
    }
    if constexpr (KS == 1) {
        if (piece >= 0) {
            __shared__ int s_flag;
            const int slot = (int)blockIdx.x - piece;
            float *part = L.split_part + (size_t)slot * kSplitPartFloats;
            float4 *mine = reinterpret_cast<float4 *>(part + ((size_t)piece * kThreads + threadIdx.x) * 8);
            __stcg(mine, make_float4(acc0[0], acc0[1], acc0[2], acc0[3]));
            __stcg(mine + 1, make_float4(acc1[0], acc1[1], acc1[2], acc1[3]));
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();  // every thread's partials before the count
                s_flag = atomicAdd(L.split_cnt + slot, 1) == 1;
            }
            __syncthreads();
            if (!s_flag) return;  // the other piece finishes the unit
            __threadfence();
            const float4 *other =
                reinterpret_cast<const float4 *>(part + ((size_t)(1 - piece) * kThreads + threadIdx.x) * 8);
            const float4 o0 = __ldcg(other), o1 = __ldcg(other + 1);
            acc0[0] += o0.x; acc0[1] += o0.y; acc0[2] += o0.z; acc0[3] += o0.w;
            acc1[0] += o1.x; acc1[1] += o1.y; acc1[2] += o1.z; acc1[3] += o1.w;
        }
    }
    if (KS > 1) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            red[warp][lane][i] = acc0[i];
            red[warp][lane][4 + i] = acc1[i];
        }
        __syncthreads();
    }
    if (ks == 0 && ok) {
        if (KS > 1) {
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                float a = 0.f, b2 = 0.f;
                for (int w = 0; w < KS; ++w) {
                    a += red[tp * KS + w][lane][i];
                    b2 += red[tp * KS + w][lane][4 + i];
                }
                acc0[i] = a;
                acc1[i] = b2;
            }
        }
        if (GATED) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int i = r0 + g + 8 * half;
#pragma unroll
                for (int col = 0; col < 2; ++col) {
                    const int pos = blk * kGemvBlock + 2 * c + col;
                    const float scl = inv[2 * c + col];
                    const float gate = acc0[2 * half + col] * scl, up = acc1[2 * half + col] * scl;
                    __nv_bfloat16 hv = __float2bfloat16_rn(silu(gate) * up);
                    p.h_out[(size_t)pos * p.h_ld + i] = *reinterpret_cast<uint16_t *>(&hv);
                }
            }
        } else {
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
                float *yrow = p.y_out + (size_t)dst * p.R;
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int n = r0 + g + 8 * half;
                    yrow[n] = acc0[2 * half + col] * wgt;
                    yrow[n + 16] = acc1[2 * half + col] * wgt;
                }
            }
        }
    }
    if (KS > 1) __syncthreads();
}

// Down stage with KS = 1 and K a multiple of 256 (units of a multiple of 4 steps), whole
// units: the CTA's consecutive units of one block (same expert and staged activations,
// the warp's rows 256 apart, so its scale-block rows two apart) stream through one
// register ring as a single sequence of steps, y written at each unit's last step.
__device__ __forceinline__ void fp8_down_runs(const FastLaunch &L, int units0, int n_pos0, int n_pos1, int u_lo,
                                              int u_hi, uint4 *smem_b, float *inv, int *rows, int *tbl_dst,
                                              float *tbl_w)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    for (int u = u_lo; u < u_hi;) {
        const int pi = u < units0 ? 0 : 1;
        const GemvParams &p = L.prob[pi];
        const int n_pos = pi ? n_pos1 : n_pos0;
        const int lu = pi ? u - units0 : u;
        const int blk = lu / p.n_tiles, grp0 = lu - blk * p.n_tiles;
        const int nu = min(p.n_tiles - grp0, u_hi - u);  // the run: this block's units in range
        u += nu;
        fp8_stage(p, blk, n_pos, false, rows, smem_b, inv);
        if (threadIdx.x < kGemvBlock) {  // per block position: y row (slot) or -1, and its factor
            const int pos = blk * kGemvBlock + threadIdx.x;
            int dst = -1;
            float w = inv[threadIdx.x];
            if (pos < n_pos) {
                if (p.sorted_slot) {
                    const int sl = chk_slot(__ldg(p.sorted_slot + pos), p.n_slots, p.status);
                    if (sl < p.n_slots) {
                        dst = sl;
                        if (p.route_w) w *= __ldg(p.route_w + sl);
                    }
                } else if (pos < p.n_pos_static) {
                    dst = pos;
                }
            }
            tbl_dst[threadIdx.x] = dst;
            tbl_w[threadIdx.x] = w;
        }
        __syncthreads();
        const int K = p.K, kb_n = K / 128, S = K / kStep8;
        const int r0a = (grp0 * 8 + warp) * 32;  // the warp's first row in the run's first unit
        const int nok = r0a < p.R ? min(nu, (p.R - r0a + 255) / 256) : 0;  // units with rows in range
        const int tot = nok * S;
        if (tot == 0) continue;
        const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + blk) : 0, p.num_experts, p.status);
        const uint8_t *ca = p.codes + (size_t)e * p.e_codes + (size_t)(r0a + g) * K + 16 * c;
        const uint8_t *cb = ca + (size_t)16 * K;  // rows r0 + 16 + g
        const size_t row8 = (size_t)8 * K;
        const uint4 *bb = smem_b + (size_t)g * (K / 8 + 1) + 2 * c;
        // scale_inv rows of the warp's two tiles (both inside one 128-row block)
        const float *sa = p.sinv + (size_t)e * p.e_sinv + (size_t)(r0a / 128) * kb_n;
        uint32_t loff = 0;  // load cursor: byte offset from the lane bases
        int ls = 0;         // and the step within its unit
        const uint32_t jump = 256u * (uint32_t)K - (uint32_t)kStep8 * (S - 1);  // to the next unit's first step
        auto load = [&](Fp8Frag &f) {
            f.a_lo = ldg_nc_v4(ca + loff);
            f.a_hi = ldg_nc_v4(ca + row8 + loff);
            f.b_lo = ldg_nc_v4(cb + loff);
            f.b_hi = ldg_nc_v4(cb + row8 + loff);
            if (++ls == S) {
                ls = 0;
                loff += jump;
            } else {
                loff += kStep8;
            }
        };
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        float t0[4] = {0.f, 0.f, 0.f, 0.f}, t1[4] = {0.f, 0.f, 0.f, 0.f};  // current 128-K block
        Fp8Frag ring[4];
        load(ring[0]);
        if (tot > 1) load(ring[1]);
        int cs = 0, r0 = r0a;  // compute cursor: step within the unit, the unit's first row
        for (int t = 0; t < tot; t += 4) {  // S, and so tot, is a multiple of 4
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (t + q + 2 < tot) load(ring[(q + 2) & 3]);
                const uint4 x0 = bb[8 * (cs + q)], x1 = bb[8 * (cs + q) + 1];
                const uint32_t b[8] = {x0.x, x0.y, x0.z, x0.w, x1.x, x1.y, x1.z, x1.w};
                fp8_tile_step(ring[q].a_lo, ring[q].a_hi, b, t0);
                fp8_tile_step(ring[q].b_lo, ring[q].b_hi, b, t1);
                if (q & 1) {  // end of a 128-K block: both tiles share its scale row
                    const float f = __ldg(sa + ((cs + q) >> 1));
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        acc0[i] = fmaf(f, t0[i], acc0[i]);
                        acc1[i] = fmaf(f, t1[i], acc1[i]);
                        t0[i] = 0.f;
                        t1[i] = 0.f;
                    }
                }
            }
            cs += 4;
            if (cs == S) {  // the unit's last step: y rows r0 .. r0 + 31 of its positions
#pragma unroll
                for (int col = 0; col < 2; ++col) {
                    const int dst = tbl_dst[2 * c + col];
                    if (dst < 0) continue;
                    const float w = tbl_w[2 * c + col];
                    float *yrow = p.y_out + (size_t)dst * p.R;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int n = r0 + g + 8 * half;
                        yrow[n] = acc0[2 * half + col] * w;
                        yrow[n + 16] = acc1[2 * half + col] * w;
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) acc0[i] = acc1[i] = 0.f;
                cs = 0;
                r0 += 256;
                sa += 2 * kb_n;  // 256 rows on: two scale-block rows
            }
        }
    }
}

template <bool GATED, int KS>
__global__ void __launch_bounds__(kThreads, 2) gemv_fp8_kernel(const __grid_constant__ FastLaunch L)
{
    pdl_enter();
    extern __shared__ uint4 smem_b[];
    __shared__ float inv[kGemvBlock];
    __shared__ int rows[kGemvBlock];
    __shared__ float red[KS > 1 ? 8 : 1][32][8];
    const int n_pos0 = load_n_pos(L.prob[0]);
    const int n_pos1 = L.nprob > 1 ? load_n_pos(L.prob[1]) : 0;
    const int units0 = (n_pos0 / kGemvBlock) * L.prob[0].n_tiles;
    const int units1 = L.nprob > 1 ? (n_pos1 / kGemvBlock) * L.prob[1].n_tiles : 0;
    const int n_units = units0 + units1;
    int staged = -1;
    auto stage_for = [&](int u) -> int {  // stage the unit's block if needed; returns its local index
        const int pi = u < units0 ? 0 : 1;
        const GemvParams &p = L.prob[pi];
        const int lu = pi ? u - units0 : u;
        const int blk = lu / p.n_tiles;
        const int key = pi * (1 << 30) + blk;
        if (key != staged) {
            fp8_stage(p, blk, pi ? n_pos1 : n_pos0, GATED, rows, smem_b, inv);
            staged = key;
        }
        return lu;
    };
    if constexpr (KS == 1) {
        // Even split of all K, in 128-K scale blocks (two steps): W = units0 * B0 + units1 * B1
        // blocks, CTA c takes [c W / G, (c + 1) W / G). Needs every CTA's share to be at least
        // one unit, so that a unit is cut at most once.
        const int B0 = L.prob[0].K / 128, B1 = L.nprob > 1 ? L.prob[1].K / 128 : B0;
        const int64_t W = (int64_t)units0 * B0 + (int64_t)units1 * B1;
        const int Bmax = B0 > B1 ? B0 : B1;
        if (L.split_part && gridDim.x <= kMaxSplitSlots && W >= (int64_t)gridDim.x * Bmax) {
            const int w_hi = (int)((int64_t)(blockIdx.x + 1) * W / gridDim.x), W0 = units0 * B0;
            for (int w = (int)((int64_t)blockIdx.x * W / gridDim.x); w < w_hi;) {
                int u, q, Bq;
                if (w < W0) {
                    u = w / B0; q = w - u * B0; Bq = B0;
                } else {
                    u = units0 + (w - W0) / B1; q = (w - W0) - (u - units0) * B1; Bq = B1;
                }
                const int q_end = w_hi - w < Bq - q ? q + (w_hi - w) : Bq;
                const int pi = u < units0 ? 0 : 1;
                const int lu = stage_for(u);
                // piece 1: tail of the unit begun by CTA c - 1; piece 0: head of one CTA c + 1 ends
                const int piece = q > 0 ? 1 : (q_end < Bq ? 0 : -1);
                fp8_unit<GATED, KS>(L.prob[pi], L, lu, pi ? n_pos1 : n_pos0, smem_b, inv, red, 2 * q, 2 * q_end,
                                    piece);
                w += q_end - q;
            }
            return;
        }
    }
    const int u_lo = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_hi = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    if constexpr (!GATED && KS == 1) {
        auto runs_ok = [](const GemvParams &q) {  // whole units of 4k steps; 32-bit code offsets
            return q.K % 256 == 0 && (int64_t)q.R * q.K < ((int64_t)1 << 32);
        };
        if (runs_ok(L.prob[0]) && (L.nprob < 2 || runs_ok(L.prob[1]))) {
            __shared__ int tbl_dst[kGemvBlock];
            __shared__ float tbl_w[kGemvBlock];
            fp8_down_runs(L, units0, n_pos0, n_pos1, u_lo, u_hi, smem_b, inv, rows, tbl_dst, tbl_w);
            return;
        }
    }
    for (int u = u_lo; u < u_hi; ++u) {
        const int pi = u < units0 ? 0 : 1;
        const int lu = stage_for(u);
        fp8_unit<GATED, KS>(L.prob[pi], L, lu, pi ? n_pos1 : n_pos0, smem_b, inv, red);
    }
}

template <bool GATED, int KS>
static cudaError_t launch_fp8_t(const FastLaunch &L, int max_units, cudaStream_t s)
{
    auto kern = gemv_fp8_kernel<GATED, KS>;
    const int Kmax = L.nprob > 1 && L.prob[1].K > L.prob[0].K ? L.prob[1].K : L.prob[0].K;
    const size_t smem = (size_t)kGemvBlock * (Kmax + 8) * 2;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int grid = sm_count() * 2;
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    FT_LAUNCH(kern, dim3(grid), dim3(kThreads), smem, s, L);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace

// K a multiple of 128 (one scale block) and each warp's share of K a whole number of blocks.
bool gemv_fp8_ok(int K, int ks) { return K % 128 == 0 && (K / ks) % 128 == 0; }

cudaError_t launch_gemv_fp8(const FastLaunch &L, bool gated, int ks, int max_units, cudaStream_t s)
{
    if (gated) {
        switch (ks) {
        case 1: return launch_fp8_t<true, 1>(L, max_units, s);
        case 2: return launch_fp8_t<true, 2>(L, max_units, s);
        case 4: return launch_fp8_t<true, 4>(L, max_units, s);
        default: return launch_fp8_t<true, 8>(L, max_units, s);
        }
    }
    switch (ks) {
    case 1: return launch_fp8_t<false, 1>(L, max_units, s);
    case 2: return launch_fp8_t<false, 2>(L, max_units, s);
    case 4: return launch_fp8_t<false, 4>(L, max_units, s);
    default: return launch_fp8_t<false, 8>(L, max_units, s);
    }
}

}  // namespace ftmoe
