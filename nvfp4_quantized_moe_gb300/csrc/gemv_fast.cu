// Decode-regime grouped GEMV, lean register-fed variant for the common shapes
// (K a multiple of 32 and each warp's K range a multiple of 128).
//
// Same arithmetic as gemv.cu: exact f16 code*scale weights against f16 activations
// staged per block with a power-of-two row scale, m16n8k16 MMAs with fp32
// accumulation, weights as M and the block's 8 tokens as N. Each warp owns two 16-row
// tiles (gate rows i and up rows I_l + i for gate_up; rows n and n + 16 for down) over
// its K range. Loads run two 128-element steps ahead through a 4-slot register ring;
// every address is a per-lane base plus a step offset; scales arrive as one 16-bit load
// per row and step; the activation swizzle reduces to a per-lane XOR, precomputed.
// gate_up splits all K steps evenly over the CTAs (a unit cut between two CTAs is
// finished by the second); the down stage streams each CTA's consecutive units of one
// block through a single ring (down_runs). The combine is a separate launch.
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "gemv_common.cuh"

namespace ftmoe {

using namespace gemv;

namespace {

struct FastFrag {
    uint4 a_lo, a_hi, b_lo, b_hi;  // codes: tile 0 rows g / g+8, tile 1 rows g / g+8
    uint32_t sa, sb;               // scales: tile 0 (row g low 16 bits, row g+8 high), tile 1
};

struct FastPtrs {
    const uint8_t *ca, *cb, *sa, *sb;  // lane bases for tile 0 / tile 1 codes and scales
    size_t crow8, srow8;               // byte offsets to the row 8 further down
    int group;
};

// The lane's two scale bytes of a row and step (group 16), or its one byte twice (group
// 32). Issued in program order with the code loads (volatile), so that they too run two
// steps ahead of their use.
__device__ __forceinline__ uint32_t scale_pair(const uint8_t *p, int group)
{
    uint32_t v;
    if (group == 16) {
        asm volatile("ld.global.nc.u16 %0, [%1];" : "=r"(v) : "l"(p));
        return v;
    }
    asm volatile("ld.global.nc.u8 %0, [%1];" : "=r"(v) : "l"(p));
    return v | (v << 8);
}

// Step weights at byte offsets co (codes) and so (scales) from the lane bases.
__device__ __forceinline__ void fast_load_at(const FastPtrs &P, uint32_t co, uint32_t so, FastFrag &f)
{
    f.a_lo = ldg_nc_v4(P.ca + co);
    f.a_hi = ldg_nc_v4(P.ca + P.crow8 + co);
    f.b_lo = ldg_nc_v4(P.cb + co);
    f.b_hi = ldg_nc_v4(P.cb + P.crow8 + co);
    f.sa = scale_pair(P.sa + so, P.group) | (scale_pair(P.sa + P.srow8 + so, P.group) << 16);
    f.sb = scale_pair(P.sb + so, P.group) | (scale_pair(P.sb + P.srow8 + so, P.group) << 16);
}

__device__ __forceinline__ void fast_load(const FastPtrs &P, int s, FastFrag &f)
{
    const int co = 64 * s;                     // 128 elements = 64 code bytes per step
    const int so = (P.group == 16) ? 8 * s : 4 * s;
    f.a_lo = ldg_nc_v4(P.ca + co);
    f.a_hi = ldg_nc_v4(P.ca + P.crow8 + co);
    f.b_lo = ldg_nc_v4(P.cb + co);
    f.b_hi = ldg_nc_v4(P.cb + P.crow8 + co);
    f.sa = scale_pair(P.sa + so, P.group) | (scale_pair(P.sa + P.srow8 + so, P.group) << 16);
    f.sb = scale_pair(P.sb + so, P.group) | (scale_pair(P.sb + P.srow8 + so, P.group) << 16);
}

__device__ __forceinline__ void fast_compute(const FastFrag &f, const uint4 *bb, const int (&boff)[4], int s,
                                             float (&acc0)[4], float (&acc1)[4])
{
    uint4 b[4];
#pragma unroll
    for (int j = 0; j < 4; ++j) b[j] = bb[16 * s + boff[j]];
    mma_step(f.a_lo, f.a_hi, f.sa & 0xFFFFu, f.sa >> 16, b, acc0);
    mma_step(f.b_lo, f.b_hi, f.sb & 0xFFFFu, f.sb >> 16, b, acc1);
}

// Lane bases of a warp's pair tile (first row r0) of expert e over the K range from k0.
template <bool GATED>
__device__ __forceinline__ FastPtrs fast_ptrs(const GemvParams &p, int e, int r0, int g, int c, int k0)
{
    const int K = p.K;
    const int row_a = r0 + g, row_b = GATED ? p.up_off + r0 + g : r0 + 16 + g;
    const uint8_t *codes_e = p.codes + (size_t)e * p.e_codes;
    const uint8_t *scales_e = p.scales + (size_t)e * p.e_scales;
    FastPtrs P;
    P.ca = codes_e + (size_t)row_a * (K / 2) + k0 / 2 + 16 * c;
    P.cb = codes_e + (size_t)row_b * (K / 2) + k0 / 2 + 16 * c;
    P.sa = scales_e + (size_t)row_a * (K / p.group) + (k0 + 32 * c) / p.group;
    P.sb = scales_e + (size_t)row_b * (K / p.group) + (k0 + 32 * c) / p.group;
    P.crow8 = (size_t)8 * (K / 2);
    P.srow8 = (size_t)8 * (K / p.group);
    P.group = p.group;
    return P;
}

}  // namespace

// One unit of work: a block of 8 positions of problem `p` and one pair-tile per warp,
// over the warp's 128-element steps [s_lo, s_hi) (all of them unless the unit is split
// between CTAs c - 1 and c (piece 1, this CTA is c) or c and c + 1 (piece 0): the pair's
// partials meet in split slot c - piece and only the second of the two CTAs to finish
// adds the other piece and runs the epilogue; a sum of two fp32 terms does not depend on
// their order).
template <bool GATED, int KS>
__device__ __forceinline__ void fast_unit(const GemvParams &p, const FastLaunch &L, int lu, int n_pos, uint4 *smem_b,
                                          const float *inv, const int *s_e, float (&red)[KS > 1 ? 8 : 1][32][8],
                                          int s_lo = 0, int s_hi = -1, int piece = -1)
{
    constexpr int TPW = 8 / KS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = warp % KS, tp = warp / KS;
    const int g = lane >> 2, c = lane & 3;
    const int K = p.K;
    const int blk = lu / p.n_tiles, grp = lu - blk * p.n_tiles;
    const int Kw = K / KS, k0 = ks * Kw;
    if (s_hi < 0) s_hi = Kw / kStep;
    const int nstep = s_hi - s_lo;
    const int pair_rows = GATED ? 16 : 32;
    const int rows_limit = GATED ? p.up_off : p.R;
    const int m = ((c >> 1) << 1) ^ (g & 1);
    const int boff[4] = {4 * c + (0 ^ m), 4 * c + (1 ^ m), 4 * c + (2 ^ m), 4 * c + (3 ^ m)};
    const int r0 = (grp * TPW + tp) * pair_rows;
    const bool ok = r0 < rows_limit;
    const int e = *s_e;
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    if (ok) {
        const FastPtrs P = fast_ptrs<GATED>(p, e, r0, g, c, k0);
        const uint4 *bb = smem_b + (size_t)g * (K / 8) + k0 / 8;
        FastFrag ring[4];
        fast_load(P, s_lo, ring[0]);
        if (nstep > 1) fast_load(P, s_lo + 1, ring[1]);
        for (int s0 = 0; s0 < nstep; s0 += 4) {
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                const int s = s0 + q;
                if (s + 2 < nstep) fast_load(P, s_lo + s + 2, ring[(q + 2) & 3]);
                if (s < nstep) fast_compute(ring[q], bb, boff, s_lo + s, acc0, acc1);
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
        const float *glob_e = p.glob + (size_t)e * p.e_glob;
        if (GATED) {
#pragma unroll
            for (int half = 0; half < 2; ++half) {
                const int i = r0 + g + 8 * half;
                const float gg = __ldg(glob_e + i), gu = __ldg(glob_e + p.up_off + i);
#pragma unroll
                for (int col = 0; col < 2; ++col) {
                    const int pos = blk * kGemvBlock + 2 * c + col;
                    const float scl = inv[2 * c + col];
                    const float gate = acc0[2 * half + col] * scl * gg;
                    const float up = acc1[2 * half + col] * scl * gu;
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
                    dst = __ldg(p.sorted_slot + pos);
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
                    yrow[n] = acc0[2 * half + col] * __ldg(glob_e + n) * wgt;
                    yrow[n + 16] = acc1[2 * half + col] * __ldg(glob_e + n + 16) * wgt;
                }
            }
        }
    }
    if (KS > 1) __syncthreads();
}

// Stage the activation rows of block `blk` of problem `p` and the block's expert id
// (CTA-wide, with barriers).
template <bool GATED>
__device__ __forceinline__ void fast_stage(const GemvParams &p, int blk, int n_pos, int *rows, uint4 *smem_b,
                                           float *inv, int *s_e)
{
    __syncthreads();
    if (threadIdx.x < kGemvBlock) rows[threadIdx.x] = source_row(p, blk * kGemvBlock + threadIdx.x, n_pos, GATED);
    if (threadIdx.x == kGemvBlock) *s_e = p.block_expert ? __ldg(p.block_expert + blk) : 0;
    __syncthreads();
    for (int r = threadIdx.x >> 5; r < kGemvBlock; r += kThreads / 32) stage_row_1pass(p.act, p.K, rows, smem_b, inv, r);
    __syncthreads();
}

// Down stage over the CTA's unit range [u_lo, u_hi), whole units of a multiple of 4 steps
// (K a multiple of 512). Consecutive units of
// one block share the expert and the staged activations, and warp w's rows in them are
// 256 apart, so each warp streams a run of them through one register ring as a single
// sequence of steps (no refill between units) and writes y at each unit's last step.
__device__ __forceinline__ void down_runs(const FastLaunch &L, int units0, int n_pos0, int n_pos1, int u_lo,
                                          int u_hi, uint4 *smem_b, float *inv, int *rows, int *s_e, float *s_glob,
                                          int *tbl_dst, float *tbl_w)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int m = ((c >> 1) << 1) ^ (g & 1);
    const int boff[4] = {4 * c + (0 ^ m), 4 * c + (1 ^ m), 4 * c + (2 ^ m), 4 * c + (3 ^ m)};
    for (int u = u_lo; u < u_hi;) {
        const int pi = u < units0 ? 0 : 1;
        const GemvParams &p = L.prob[pi];
        const int n_pos = pi ? n_pos1 : n_pos0;
        const int lu = pi ? u - units0 : u;
        const int blk = lu / p.n_tiles, grp0 = lu - blk * p.n_tiles;
        const int nu = min(p.n_tiles - grp0, u_hi - u);  // the run: this block's units in range
        u += nu;
        fast_stage<false>(p, blk, n_pos, rows, smem_b, inv, s_e);
        if (threadIdx.x < kGemvBlock) {  // per block position: y row (slot) or -1, and its factor
            const int pos = blk * kGemvBlock + threadIdx.x;
            int dst = -1;
            float w = inv[threadIdx.x];
            if (pos < n_pos) {
                if (p.sorted_slot) {
                    const int sl = __ldg(p.sorted_slot + pos);
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
        const int r0a = (grp0 * 8 + warp) * 32;  // the warp's first row in the run's first unit
        // units with rows in range form a prefix of the run
        const int nok = r0a < p.R ? min(nu, (p.R - r0a + 255) / 256) : 0;
        const int S = p.K / kStep, tot = nok * S;
        if (tot == 0) continue;
        const int e = *s_e;
        const FastPtrs P = fast_ptrs<false>(p, e, r0a, g, c, 0);
        const uint32_t spb = (p.group == 16) ? 8u : 4u;  // scale bytes per step and row pair
        // from a unit's last step to the next unit's first: 256 rows on, back to K = 0
        const uint32_t jump_c = 256u * (uint32_t)(p.K / 2) - 64u * (uint32_t)(S - 1);
        const uint32_t jump_s = 256u * (uint32_t)(p.K / p.group) - spb * (uint32_t)(S - 1);
        const uint4 *bb = smem_b + (size_t)g * (p.K / 8);
        const float *glob_e = p.glob + (size_t)e * p.e_glob;
        uint32_t lco = 0, lso = 0;
        int ls = 0;  // load cursor: byte offsets and step within its unit
        auto advance_load = [&]() {
            if (++ls == S) {
                ls = 0;
                lco += jump_c;
                lso += jump_s;
            } else {
                lco += 64u;
                lso += spb;
            }
        };
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        FastFrag ring[4];
        fast_load_at(P, lco, lso, ring[0]);
        advance_load();
        if (tot > 1) {
            fast_load_at(P, lco, lso, ring[1]);
            advance_load();
        }
        int cs = 0, r0 = r0a;  // compute cursor: step within the unit, the unit's first row
        float *gs = s_glob + threadIdx.x * 4;
        for (int t0 = 0; t0 < tot; t0 += 4) {  // S, and so tot, is a multiple of 4
            if (cs == 0) {  // a unit's first steps: copy its rows' globals to shared memory
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    cp_async_4(gs + 2 * half, glob_e + r0 + g + 8 * half);
                    cp_async_4(gs + 2 * half + 1, glob_e + r0 + g + 8 * half + 16);
                }
                cp_async_commit();
            }
#pragma unroll
            for (int q = 0; q < 4; ++q) {
                if (t0 + q + 2 < tot) {
                    fast_load_at(P, lco, lso, ring[(q + 2) & 3]);
                    advance_load();
                }
                fast_compute(ring[q], bb, boff, cs + q, acc0, acc1);
            }
            cs += 4;
            if (cs == S) {  // the unit's last step: y rows r0 .. r0 + 31 of its positions
                cp_async_wait<0>();
#pragma unroll
                for (int col = 0; col < 2; ++col) {
                    const int dst = tbl_dst[2 * c + col];
                    if (dst < 0) continue;
                    const float w = tbl_w[2 * c + col];
                    float *yrow = p.y_out + (size_t)dst * p.R;
#pragma unroll
                    for (int half = 0; half < 2; ++half) {
                        const int n = r0 + g + 8 * half;
                        yrow[n] = acc0[2 * half + col] * gs[2 * half] * w;
                        yrow[n + 16] = acc1[2 * half + col] * gs[2 * half + 1] * w;
                    }
                }
#pragma unroll
                for (int i = 0; i < 4; ++i) acc0[i] = acc1[i] = 0.f;
                cs = 0;
                r0 += 256;
            }
        }
    }
}

// Grid-strided over the concatenated unit lists of up to two problems (the routed
// experts and the shared expert); each CTA takes a contiguous range of units.
template <bool GATED, int KS>
__global__ void __launch_bounds__(kThreads, 2) gemv_fast_kernel(const __grid_constant__ FastLaunch L)
{
    pdl_enter();
    extern __shared__ uint4 smem_b[];
    __shared__ float inv[kGemvBlock];
    __shared__ int rows[kGemvBlock];
    __shared__ int s_e;  // expert of the staged block
    __shared__ float s_glob[GATED ? 1 : kThreads * 4];  // down: each thread's row globals of its current unit
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
            fast_stage<GATED>(p, blk, pi ? n_pos1 : n_pos0, rows, smem_b, inv, &s_e);
            staged = key;
        }
        return lu;
    };
    if constexpr (KS == 1) {
        // Even split of all K steps: W = units0 * S0 + units1 * S1 steps, CTA c takes
        // [c W / G, (c + 1) W / G). Needs every CTA's share to be at least one unit, so
        // that a unit is cut at most once.
        const int S0 = L.prob[0].K / kStep, S1 = L.nprob > 1 ? L.prob[1].K / kStep : S0;
        const int64_t W = (int64_t)units0 * S0 + (int64_t)units1 * S1;
        const int Smax = S0 > S1 ? S0 : S1;
        if (L.split_part && gridDim.x <= kMaxSplitSlots && W >= (int64_t)gridDim.x * Smax) {
            const int w_hi = (int)((int64_t)(blockIdx.x + 1) * W / gridDim.x), W0 = units0 * S0;
            for (int w = (int)((int64_t)blockIdx.x * W / gridDim.x); w < w_hi;) {
                int u, s, S;
                if (w < W0) {
                    u = w / S0; s = w - u * S0; S = S0;
                } else {
                    u = units0 + (w - W0) / S1; s = (w - W0) - (u - units0) * S1; S = S1;
                }
                const int s_end = w_hi - w < S - s ? s + (w_hi - w) : S;
                const int pi = u < units0 ? 0 : 1;
                const int lu = stage_for(u);
                // piece 1: tail of the unit begun by CTA c - 1; piece 0: head of one CTA c + 1 ends
                const int piece = s > 0 ? 1 : (s_end < S ? 0 : -1);
                fast_unit<GATED, KS>(L.prob[pi], L, lu, pi ? n_pos1 : n_pos0, smem_b, inv, &s_e, red, s, s_end, piece);
                w += s_end - s;
            }
            return;
        }
    }
    const int u_lo = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_hi = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    if constexpr (!GATED && KS == 1) {  // (the host keeps each expert's bank below 2 GB here)
        if (L.prob[0].K % (4 * kStep) == 0 && (L.nprob < 2 || L.prob[1].K % (4 * kStep) == 0)) {
            __shared__ int tbl_dst[kGemvBlock];
            __shared__ float tbl_w[kGemvBlock];
            down_runs(L, units0, n_pos0, n_pos1, u_lo, u_hi, smem_b, inv, rows, &s_e, s_glob, tbl_dst, tbl_w);
            return;
        }
    }
    for (int u = u_lo; u < u_hi; ++u) {
        const int pi = u < units0 ? 0 : 1;
        const int lu = stage_for(u);
        fast_unit<GATED, KS>(L.prob[pi], L, lu, pi ? n_pos1 : n_pos0, smem_b, inv, &s_e, red);
    }
}

// Usable for this shape and K-split? (R = the matrix's rows: the down path addresses an
// expert's codes with 32-bit offsets.)
bool gemv_fast_ok(int K, int group, int ks, int R)
{
    return K % 32 == 0 && (K / ks) % kStep == 0 && (group == 16 || group == 32) &&
           (int64_t)R * (K / 2) < ((int64_t)1 << 31);
}

template <bool GATED, int KS>
static cudaError_t launch_fast_t(const FastLaunch &L, int max_units, cudaStream_t s)
{
    auto kern = gemv_fast_kernel<GATED, KS>;
    const int Kmax = L.nprob > 1 && L.prob[1].K > L.prob[0].K ? L.prob[1].K : L.prob[0].K;
    const size_t smem = (size_t)kGemvBlock * Kmax * 2;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int grid = sm_count() * 2;
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    FT_LAUNCH(kern, dim3(grid), dim3(kThreads), smem, s, L);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_gemv_fast(const FastLaunch &L, bool gated, int ks, int max_units, cudaStream_t s)
{
    if (gated) {
        switch (ks) {
        case 1: return launch_fast_t<true, 1>(L, max_units, s);
        case 2: return launch_fast_t<true, 2>(L, max_units, s);
        case 4: return launch_fast_t<true, 4>(L, max_units, s);
        default: return launch_fast_t<true, 8>(L, max_units, s);
        }
    }
    switch (ks) {
    case 1: return launch_fast_t<false, 1>(L, max_units, s);
    case 2: return launch_fast_t<false, 2>(L, max_units, s);
    case 4: return launch_fast_t<false, 4>(L, max_units, s);
    default: return launch_fast_t<false, 8>(L, max_units, s);
    }
}

}  // namespace ftmoe
