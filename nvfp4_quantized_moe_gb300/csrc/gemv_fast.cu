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

// Shared-memory scratch of one CTA of the lean kernels (beside the dynamic activation rows).
struct FastShared {
    float inv[kGemvBlock];       // staged rows' power-of-two factors
    int rows[kGemvBlock];        // staged rows' source rows (-1: padding)
    int s_e;                     // expert of the staged block
    int flag;                    // broadcast: split finisher / outcome of a wait
    int dead;                    // fused kernel: a wait of this CTA gave up; later waits return at once
    int tbl_dst[kGemvBlock];     // down runs: y row of each block position (or -1)
    float tbl_w[kGemvBlock];     // down runs: its factor
    float s_glob[kThreads * 4];  // down runs: each thread's row globals of its current unit
};

// The warps' partial sums of an in-CTA K split (declared only by kernels that split K).
typedef float RedBuf[32][8];

__device__ __forceinline__ int ld_acquire(const int *p)
{
    int v;
    asm volatile("ld.acquire.gpu.global.s32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

// Thread 0 waits until *ctr >= want (acquire), sleeping between polls; false after
// limit_ns (FT_ERR_TIMEOUT is recorded) or at once when an earlier wait of the CTA gave up.
// The outcome reaches every thread through sm.flag (the caller synchronises).
__device__ __forceinline__ void wait_counter_t0(const int *ctr, int want, uint64_t limit_ns, int *status,
                                                FastShared &sm)
{
    int ok = !sm.dead;
    if (ok && ld_acquire(ctr) < want) {
        const uint64_t t0 = globaltimer();
        uint32_t ns = 32;
        while (ld_acquire(ctr) < want) {
            __nanosleep(ns);
            if (ns < 256) ns <<= 1;
            if (globaltimer() - t0 > limit_ns) {
                ok = 0;
                raise_status(status, FT_ERR_TIMEOUT);
                break;
            }
        }
    }
    if (!ok) sm.dead = 1;
    sm.flag = ok;
}

}  // namespace

// Cross-CTA ordering inside the fused decode kernel (null for the separate kernels): a
// block's down units start once all of its gate_up CTA units have written h.
struct DecodeSync {
    int *gu_done;     // per block: gate_up CTA units finished (routed blocks, then the shared ones)
    int shared_base;  // index in gu_done of the shared expert's first block
    int target[2];    // count of a complete block of the routed / shared problem (8 per gate_up CTA unit)
    int *status;
    uint64_t wait_ns;
};

__device__ __forceinline__ int *gu_counter(const DecodeSync *S, int pi, int blk)
{
    return S->gu_done + (pi ? S->shared_base + blk : blk);
}

// CTA-wide: wait until block `blk` of problem `pi` has its h rows (fused kernel only).
__device__ __forceinline__ void wait_block_ready(const DecodeSync *S, int pi, int blk, FastShared &sm)
{
    if (!S) return;
    __syncthreads();
    if (threadIdx.x == 0) wait_counter_t0(gu_counter(S, pi, blk), S->target[pi], S->wait_ns, S->status, sm);
    __syncthreads();
}

// One unit of work: a block of 8 positions of problem `p` and one pair-tile per warp,
// over the warp's 128-element steps [s_lo, s_hi) (all of them unless the unit is split
// between CTAs c - 1 and c (piece 1, this CTA is c) or c and c + 1 (piece 0): the pair's
// partials meet in split slot c - piece and only the second of the two CTAs to finish
// adds the other piece and runs the epilogue; a sum of two fp32 terms does not depend on
// their order). done_ctr (fused kernel, gate_up): raised by 8 once the unit's h rows are
// written, with release semantics, by whichever CTA ran the epilogue.
template <bool GATED, int KS>
__device__ __forceinline__ void fast_unit(const GemvParams &p, const FastLaunch &L, int lu, int n_pos, uint4 *smem_b,
                                          FastShared &sm, RedBuf *red, int s_lo = 0, int s_hi = -1, int piece = -1,
                                          int *done_ctr = nullptr)
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
    const int e = sm.s_e;
    const float *inv = sm.inv;
    float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
    // the epilogue's row globals: with the K split inside the CTA (small batches, short
    // loops) loaded while the steps stream, otherwise after them (no registers held)
    const float *glob_e = p.glob + (size_t)e * p.e_glob;
    float gl[4] = {0.f, 0.f, 0.f, 0.f};
    auto load_globals = [&]() {
#pragma unroll
        for (int half = 0; half < 2; ++half) {
            const int i = r0 + g + 8 * half;
            gl[2 * half] = __ldg(glob_e + i);
            gl[2 * half + 1] = __ldg(glob_e + (GATED ? p.up_off + i : i + 16));
        }
    };
    if (KS > 1 && ok && ks == 0) load_globals();
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
            const int slot = (int)blockIdx.x - piece;
            float *part = L.split_part + (size_t)slot * kSplitPartFloats;
            float4 *mine = reinterpret_cast<float4 *>(part + ((size_t)piece * kThreads + threadIdx.x) * 8);
            __stcg(mine, make_float4(acc0[0], acc0[1], acc0[2], acc0[3]));
            __stcg(mine + 1, make_float4(acc1[0], acc1[1], acc1[2], acc1[3]));
            __syncthreads();
            if (threadIdx.x == 0) {
                __threadfence();  // every thread's partials before the count
                sm.flag = atomicAdd(L.split_cnt + slot, 1) == 1;
            }
            __syncthreads();
            if (!sm.flag) return;  // the other piece finishes the unit
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
        if (KS == 1) load_globals();
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
                const float gg = gl[2 * half], gu = gl[2 * half + 1];
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
                    yrow[n] = acc0[2 * half + col] * gl[2 * half] * wgt;
                    yrow[n + 16] = acc1[2 * half + col] * gl[2 * half + 1] * wgt;
                }
            }
        }
    }
    if (KS > 1) __syncthreads();
    if (done_ctr) {
        // publish the unit's h rows: 8 counts per unit, one per warp (each after its own rows,
        // so that no warp waits for the others), or all 8 at once after the K-split barrier
        if (KS > 1) {
            if (threadIdx.x == 0) {
                __threadfence();
                atomicAdd(done_ctr, 8);
            }
        } else {
            __syncwarp();
            if (lane == 0) {
                __threadfence();
                atomicAdd(done_ctr, 1);
            }
        }
    }
}

// Stage the activation rows of block `blk` of problem `p` and the block's expert id
// (CTA-wide, with barriers). COHERENT: rows written earlier in the same launch.
template <bool GATED, bool COHERENT = false>
__device__ __forceinline__ void fast_stage(const GemvParams &p, int blk, int n_pos, uint4 *smem_b, FastShared &sm)
{
    __syncthreads();
    if (threadIdx.x < kGemvBlock)
        sm.rows[threadIdx.x] = source_row(p, blk * kGemvBlock + threadIdx.x, n_pos, GATED);
    if (threadIdx.x == kGemvBlock)
        sm.s_e = chk_expert(p.block_expert ? __ldg(p.block_expert + blk) : 0, p.num_experts, p.status);
    __syncthreads();
    for (int r = threadIdx.x >> 5; r < kGemvBlock; r += kThreads / 32)
        stage_row_1pass<COHERENT>(p.act, p.K, sm.rows, smem_b, sm.inv, r);
    __syncthreads();
}

// Down stage over the CTA's unit range [u_lo, u_hi), whole units of a multiple of 4 steps
// (K a multiple of 512). Consecutive units of one block share the expert and the staged
// activations, and warp w's rows in them are 256 apart, so each warp streams a run of
// them through one register ring as a single sequence of steps (no refill between units)
// and writes y at each unit's last step. S (fused kernel): before a block's h rows are
// staged, its gate_up units must have finished; the run's first weight loads are issued
// before that wait.
template <bool COHERENT>
__device__ __forceinline__ void down_runs(const FastLaunch &L, int units0, int n_pos0, int n_pos1, int u_lo, int u_hi,
                                          uint4 *smem_b, FastShared &sm, const DecodeSync *S)
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
        const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + blk) : 0, p.num_experts, p.status);
        const int r0a = (grp0 * 8 + warp) * 32;  // the warp's first row in the run's first unit
        // units with rows in range form a prefix of the run
        const int nok = r0a < p.R ? min(nu, (p.R - r0a + 255) / 256) : 0;
        const int S_ = p.K / kStep, tot = nok * S_;
        const FastPtrs P = fast_ptrs<false>(p, e, r0a < p.R ? r0a : 0, g, c, 0);
        const uint32_t spb = (p.group == 16) ? 8u : 4u;  // scale bytes per step and row pair
        // from a unit's last step to the next unit's first: 256 rows on, back to K = 0
        const uint32_t jump_c = 256u * (uint32_t)(p.K / 2) - 64u * (uint32_t)(S_ - 1);
        const uint32_t jump_s = 256u * (uint32_t)(p.K / p.group) - spb * (uint32_t)(S_ - 1);
        uint32_t lco = 0, lso = 0;
        int ls = 0;  // load cursor: byte offsets and step within its unit
        auto advance_load = [&]() {
            if (++ls == S_) {
                ls = 0;
                lco += jump_c;
                lso += jump_s;
            } else {
                lco += 64u;
                lso += spb;
            }
        };
        // The first two steps' weights do not depend on h. In the fused kernel they are put in
        // flight before the wait for the block's h rows; in a separate launch h is ready, and the
        // staging and the position table go first (their dependent loads then do not queue
        // behind the weights').
        FastFrag ring[4];
        auto prime = [&]() {
            if (tot > 0) {
                fast_load_at(P, lco, lso, ring[0]);
                advance_load();
            }
            if (tot > 1) {
                fast_load_at(P, lco, lso, ring[1]);
                advance_load();
            }
        };
        if (S) {
            prime();
            wait_block_ready(S, pi, blk, sm);
        }
        fast_stage<false, COHERENT>(p, blk, n_pos, smem_b, sm);
        if (threadIdx.x < kGemvBlock) {  // per block position: y row (slot) or -1, and its factor
            const int pos = blk * kGemvBlock + threadIdx.x;
            int dst = -1;
            float w = sm.inv[threadIdx.x];
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
            sm.tbl_dst[threadIdx.x] = dst;
            sm.tbl_w[threadIdx.x] = w;
        }
        __syncthreads();
        if (!S) prime();
        if (tot == 0) continue;
        const uint4 *bb = smem_b + (size_t)g * (p.K / 8);
        const float *glob_e = p.glob + (size_t)e * p.e_glob;
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        int cs = 0, r0 = r0a;  // compute cursor: step within the unit, the unit's first row
        float *gs = sm.s_glob + threadIdx.x * 4;
        for (int t0 = 0; t0 < tot; t0 += 4) {  // S_, and so tot, is a multiple of 4
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
            if (cs == S_) {  // the unit's last step: y rows r0 .. r0 + 31 of its positions
                cp_async_wait<0>();
#pragma unroll
                for (int col = 0; col < 2; ++col) {
                    const int dst = sm.tbl_dst[2 * c + col];
                    if (dst < 0) continue;
                    const float w = sm.tbl_w[2 * c + col];
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

// gate_up over the CTA's step range [w_lo, w_hi) of the even split (KS = 1, every K a
// multiple of 512, I_l a multiple of 128, range ends on 4-step boundaries): consecutive
// units of one block share the staged activations and warp w's 16 gate (and up) rows in
// them are 128 apart, so each warp streams a run of them through one register ring as a
// single sequence of steps and runs each unit's epilogue (SwiGLU into h, or the split
// exchange of a unit cut between two CTAs) while the next unit's first loads are in flight.
__device__ __forceinline__ void gate_runs(const FastLaunch &L, int units0, int n_pos0, int n_pos1, int64_t w_lo,
                                          int64_t w_hi, uint4 *smem_b, FastShared &sm, const DecodeSync *S)
{
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int g = lane >> 2, c = lane & 3;
    const int m = ((c >> 1) << 1) ^ (g & 1);
    const int boff[4] = {4 * c + (0 ^ m), 4 * c + (1 ^ m), 4 * c + (2 ^ m), 4 * c + (3 ^ m)};
    const int S0 = L.prob[0].K / kStep, S1 = L.nprob > 1 ? L.prob[1].K / kStep : S0;
    const int64_t W0 = (int64_t)units0 * S0;
    for (int64_t w = w_lo; w < w_hi;) {
        int u, s, Sx;
        if (w < W0) {
            u = (int)(w / S0); s = (int)(w - (int64_t)u * S0); Sx = S0;
        } else {
            u = units0 + (int)((w - W0) / S1); s = (int)((w - W0) - (int64_t)(u - units0) * S1); Sx = S1;
        }
        const int pi = u < units0 ? 0 : 1;
        const GemvParams &p = L.prob[pi];
        const int n_pos = pi ? n_pos1 : n_pos0;
        const int lu = pi ? u - units0 : u;
        const int blk = lu / p.n_tiles, grp0 = lu - blk * p.n_tiles;
        // the run: this block's units from grp0 on, as far as the range reaches
        const int64_t avail = w_hi - w;
        const int64_t block_steps = (int64_t)(Sx - s) + (int64_t)(p.n_tiles - grp0 - 1) * Sx;
        const int tot = (int)(avail < block_steps ? avail : block_steps);
        const int last_end = (int)((s + tot - 1) % Sx) + 1;  // the last unit's end step
        const int n_run = (s + tot + Sx - 1) / Sx;             // units in the run
        w += tot;
        fast_stage<true>(p, blk, n_pos, smem_b, sm);
        const int e = sm.s_e;
        const int r0a = (grp0 * 8 + warp) * 16;  // the warp's first gate row in the run's first unit
        const FastPtrs P = fast_ptrs<true>(p, e, r0a, g, c, 0);
        const uint32_t spb = (p.group == 16) ? 8u : 4u;
        const uint32_t jump_c = 128u * (uint32_t)(p.K / 2) - 64u * (uint32_t)(Sx - 1);
        const uint32_t jump_s = 128u * (uint32_t)(p.K / p.group) - spb * (uint32_t)(Sx - 1);
        uint32_t lco = 64u * (uint32_t)s, lso = spb * (uint32_t)s;
        int ls = s;
        auto advance_load = [&]() {
            if (++ls == Sx) {
                ls = 0;
                lco += jump_c;
                lso += jump_s;
            } else {
                lco += 64u;
                lso += spb;
            }
        };
        const uint4 *bb = smem_b + (size_t)g * (p.K / 8);
        const float *glob_e = p.glob + (size_t)e * p.e_glob;
        int *done_ctr = S && S->gu_done ? gu_counter(S, pi, blk) : nullptr;
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        float gl[4] = {0.f, 0.f, 0.f, 0.f};
        FastFrag ring[4];
        fast_load_at(P, lco, lso, ring[0]);
        advance_load();
        if (tot > 1) {
            fast_load_at(P, lco, lso, ring[1]);
            advance_load();
        }
        int j = 0, cs = s, r0 = r0a;  // compute cursor: unit in the run, its step, its first gate row
        for (int t0 = 0; t0 < tot; t0 += 4) {  // every piece is a whole number of 4-step groups
            const int end_j = j == n_run - 1 ? last_end : Sx;
            if (cs + 4 == end_j) {  // the unit's last group: its rows' globals, used by its epilogue
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int i = r0 + g + 8 * half;
                    gl[2 * half] = __ldg(glob_e + i);
                    gl[2 * half + 1] = __ldg(glob_e + p.up_off + i);
                }
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
            if (cs < end_j) continue;
            // the unit's end: a piece of a unit cut between two CTAs meets its other piece
            // first (piece 1: tail of the unit begun by CTA c - 1; piece 0: its head)
            const int piece = (j == 0 && s > 0) ? 1 : (end_j < Sx ? 0 : -1);
            bool finish = true;
            if (piece >= 0) {
                const int slot = (int)blockIdx.x - piece;
                float *part = L.split_part + (size_t)slot * kSplitPartFloats;
                float4 *mine = reinterpret_cast<float4 *>(part + ((size_t)piece * kThreads + threadIdx.x) * 8);
                __stcg(mine, make_float4(acc0[0], acc0[1], acc0[2], acc0[3]));
                __stcg(mine + 1, make_float4(acc1[0], acc1[1], acc1[2], acc1[3]));
                __syncthreads();
                if (threadIdx.x == 0) {
                    __threadfence();  // every thread's partials before the count
                    sm.flag = atomicAdd(L.split_cnt + slot, 1) == 1;
                }
                __syncthreads();
                finish = sm.flag != 0;
                if (finish) {
                    __threadfence();
                    const float4 *other =
                        reinterpret_cast<const float4 *>(part + ((size_t)(1 - piece) * kThreads + threadIdx.x) * 8);
                    const float4 o0 = __ldcg(other), o1 = __ldcg(other + 1);
                    acc0[0] += o0.x; acc0[1] += o0.y; acc0[2] += o0.z; acc0[3] += o0.w;
                    acc1[0] += o1.x; acc1[1] += o1.y; acc1[2] += o1.z; acc1[3] += o1.w;
                }
            }
            if (finish) {
#pragma unroll
                for (int half = 0; half < 2; ++half) {
                    const int i = r0 + g + 8 * half;
#pragma unroll
                    for (int col = 0; col < 2; ++col) {
                        const int pos = blk * kGemvBlock + 2 * c + col;
                        const float scl = sm.inv[2 * c + col];
                        const float gate = acc0[2 * half + col] * scl * gl[2 * half];
                        const float up = acc1[2 * half + col] * scl * gl[2 * half + 1];
                        __nv_bfloat16 hv = __float2bfloat16_rn(silu(gate) * up);
                        p.h_out[(size_t)pos * p.h_ld + i] = *reinterpret_cast<uint16_t *>(&hv);
                    }
                }
                if (done_ctr) {  // publish this warp's rows of the unit
                    __syncwarp();
                    if (lane == 0) {
                        __threadfence();
                        atomicAdd(done_ctr, 1);
                    }
                }
            }
#pragma unroll
            for (int i = 0; i < 4; ++i) acc0[i] = acc1[i] = 0.f;
            ++j;
            cs = 0;
            r0 += 128;
        }
    }
}

// One stage (gate_up or down) of the lean kernels over the concatenated unit lists of up
// to two problems (the routed experts and the shared expert): the even split of all K
// steps (gate_up, KS = 1), block runs (down, KS = 1), or contiguous unit ranges with the K
// split inside the CTA. S: fused kernel (gate_up counts finished units per block; down
// waits for them and reads h through L2).
template <bool GATED, int KS, bool FUSED>
__device__ __forceinline__ void fast_phase(const FastLaunch &L, uint4 *smem_b, FastShared &sm, RedBuf *red,
                                           const DecodeSync *S)
{
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
            if (!GATED) wait_block_ready(S, pi, blk, sm);
            fast_stage<GATED, FUSED && !GATED>(p, blk, pi ? n_pos1 : n_pos0, smem_b, sm);
            staged = key;
        }
        return lu;
    };
    auto counter = [&](int u) -> int * {  // fused gate_up: the unit's block counter
        if (!(FUSED && GATED) || !S->gu_done) return nullptr;
        const int pi = u < units0 ? 0 : 1;
        const int lu = pi ? u - units0 : u;
        return gu_counter(S, pi, lu / L.prob[pi].n_tiles);
    };
    if constexpr (KS == 1 && GATED) {
        // Even split of all K steps: W = units0 * S0 + units1 * S1 steps, CTA c takes
        // [c W / G, (c + 1) W / G). Needs every CTA's share to be at least one unit, so
        // that a unit is cut at most once.
        const int S0 = L.prob[0].K / kStep, S1 = L.nprob > 1 ? L.prob[1].K / kStep : S0;
        const int64_t W = (int64_t)units0 * S0 + (int64_t)units1 * S1;
        const int Smax = S0 > S1 ? S0 : S1;
        if (L.split_part && gridDim.x <= kMaxSplitSlots && W >= (int64_t)gridDim.x * Smax) {
            // runs of units through one ring when every K and every CTA range splits into
            // 4-step groups and every unit's rows are all in range
            const bool runs = S0 % 4 == 0 && S1 % 4 == 0 && L.prob[0].up_off % 128 == 0 &&
                              (L.nprob < 2 || L.prob[1].up_off % 128 == 0);
            if (runs) {
                const int64_t Wq = W / 4;
                gate_runs(L, units0, n_pos0, n_pos1, 4 * ((int64_t)blockIdx.x * Wq / gridDim.x),
                          4 * ((int64_t)(blockIdx.x + 1) * Wq / gridDim.x), smem_b, sm, S);
                return;
            }
            const int w_hi = (int)((int64_t)(blockIdx.x + 1) * W / gridDim.x), W0 = units0 * S0;
            for (int w = (int)((int64_t)blockIdx.x * W / gridDim.x); w < w_hi;) {
                int u, s, Sx;
                if (w < W0) {
                    u = w / S0; s = w - u * S0; Sx = S0;
                } else {
                    u = units0 + (w - W0) / S1; s = (w - W0) - (u - units0) * S1; Sx = S1;
                }
                const int s_end = w_hi - w < Sx - s ? s + (w_hi - w) : Sx;
                const int pi = u < units0 ? 0 : 1;
                const int lu = stage_for(u);
                // piece 1: tail of the unit begun by CTA c - 1; piece 0: head of one CTA c + 1 ends
                const int piece = s > 0 ? 1 : (s_end < Sx ? 0 : -1);
                fast_unit<GATED, KS>(L.prob[pi], L, lu, pi ? n_pos1 : n_pos0, smem_b, sm, red, s, s_end, piece,
                                     counter(u));
                w += s_end - s;
            }
            return;
        }
    }
    const int u_lo = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_hi = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    if constexpr (!GATED && KS == 1) {  // (the host keeps each expert's bank below 2 GB here)
        if (L.prob[0].K % (4 * kStep) == 0 && (L.nprob < 2 || L.prob[1].K % (4 * kStep) == 0)) {
            down_runs<FUSED>(L, units0, n_pos0, n_pos1, u_lo, u_hi, smem_b, sm, S);
            return;
        }
    }
    for (int u = u_lo; u < u_hi; ++u) {
        const int pi = u < units0 ? 0 : 1;
        const int lu = stage_for(u);
        fast_unit<GATED, KS>(L.prob[pi], L, lu, pi ? n_pos1 : n_pos0, smem_b, sm, red, 0, -1, -1, counter(u));
    }
}

// A separate gate_up or down launch (its predecessor's outputs are complete on entry).
template <bool GATED, int KS>
__global__ void __launch_bounds__(kThreads, 2) gemv_fast_kernel(const __grid_constant__ FastLaunch L)
{
    pdl_enter();
    extern __shared__ uint4 smem_b[];
    __shared__ FastShared sm;
    __shared__ RedBuf red[KS > 1 ? 8 : 1];
    if (threadIdx.x == 0) sm.dead = 0;
    fast_phase<GATED, KS, false>(L, smem_b, sm, red, nullptr);
}

// Fused decode forward: gate_up (+ SwiGLU into h) over every touched block, then down
// (+ routing weight and row global into the slot-major y rows), then the ordered combine
// out[t] = sum_{j<k} y[t k + j] (+ y_shared[t]), in one persistent launch. A block's down
// units wait (bounded) for its gate_up units through per-block counters; the combine
// waits (bounded) for every CTA's down units through one grid-wide count. All CTAs are
// resident at once (the host sizes the grid by the occupancy), and the kernel lets the
// next launch of the stream be scheduled only after its last wait, so no CTA can wait on
// one that has no SM to run on.
template <int KSG, int KSD>
__global__ void __launch_bounds__(kThreads, 2) gemv_fused_kernel(const __grid_constant__ FusedLaunch F)
{
    pdl_wait();
    extern __shared__ uint4 smem_b[];
    __shared__ FastShared sm;
    __shared__ RedBuf red[KSG > 1 || KSD > 1 ? 8 : 1];
    if (threadIdx.x == 0) sm.dead = 0;
    __syncthreads();
    DecodeSync S;
    S.gu_done = F.gu_done;
    S.shared_base = F.shared_base;
    S.target[0] = 8 * F.gu.prob[0].n_tiles;  // 8 counts per gate_up CTA unit
    S.target[1] = F.gu.nprob > 1 ? 8 * F.gu.prob[1].n_tiles : 0;
    S.status = F.status;
    S.wait_ns = F.wait_ns ? F.wait_ns : kWaitNs;
    DecodeSync S_gu = S;
    if (F.skip_publish) S_gu.gu_done = nullptr;  // fault injection: nothing is published
    fast_phase<true, KSG, true>(F.gu, smem_b, sm, red, &S_gu);
    fast_phase<false, KSD, true>(F.dn, smem_b, sm, red, &S);
    // every CTA's y rows before any combine
    __syncthreads();
    if (threadIdx.x == 0) {
        __threadfence();
        atomicAdd(F.done, 1);
        wait_counter_t0(F.done, (int)gridDim.x, S.wait_ns, F.status, sm);
    }
    __syncthreads();
    pdl_trigger();  // past the last wait: the next launch may take SM slots now
    const int H4 = F.H / 4, k = F.k;
    const int64_t n = (int64_t)F.T * H4;
    const int64_t lo = (int64_t)blockIdx.x * n / gridDim.x, hi = (int64_t)(blockIdx.x + 1) * n / gridDim.x;
    for (int64_t idx = lo + threadIdx.x; idx < hi; idx += kThreads) {
        const int t = (int)(idx / H4), n4 = (int)(idx % H4);
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
        const float4 sh = F.y_sh ? __ldcg(reinterpret_cast<const float4 *>(F.y_sh + (size_t)t * F.H) + n4)
                                 : make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll 8
        for (int j = 0; j < k; ++j) {  // fixed order: j = 0 .. k - 1, then the shared row
            const float4 v = __ldcg(reinterpret_cast<const float4 *>(F.y + ((size_t)t * k + j) * F.H) + n4);
            acc.x += v.x; acc.y += v.y; acc.z += v.z; acc.w += v.w;
        }
        if (F.y_sh) {
            acc.x += sh.x; acc.y += sh.y; acc.z += sh.z; acc.w += sh.w;
        }
        if (F.out_dtype == FT_DTYPE_F32) {
            reinterpret_cast<float4 *>(static_cast<float *>(F.out) + (size_t)t * F.H)[n4] = acc;
        } else {
            __nv_bfloat162 a = __floats2bfloat162_rn(acc.x, acc.y), b = __floats2bfloat162_rn(acc.z, acc.w);
            uint2 v;
            v.x = *reinterpret_cast<uint32_t *>(&a);
            v.y = *reinterpret_cast<uint32_t *>(&b);
            reinterpret_cast<uint2 *>(static_cast<uint16_t *>(F.out) + (size_t)t * F.H)[n4] = v;
        }
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

template <int KSG, int KSD>
static cudaError_t launch_fused_t(const FusedLaunch &F, int max_units, cudaStream_t s)
{
    auto kern = gemv_fused_kernel<KSG, KSD>;
    int Kmax = 0;
    for (const FastLaunch *L : {&F.gu, &F.dn})
        for (int i = 0; i < L->nprob; ++i) Kmax = L->prob[i].K > Kmax ? L->prob[i].K : Kmax;
    const size_t smem = (size_t)kGemvBlock * Kmax * 2;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    // every CTA must be resident at once: the grid never exceeds what the SMs hold together
    int occ = 0;
    e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, kThreads, smem);
    if (e != cudaSuccess) return e;
    if (occ < 1) return cudaErrorInvalidConfiguration;
    int grid = sm_count() * (occ < 2 ? occ : 2);
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    FT_LAUNCH(kern, dim3(grid), dim3(kThreads), smem, s, F);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_gemv_fused(const FusedLaunch &F, int ks_gu, int ks_dn, int max_units, cudaStream_t s)
{
#define FT_FUSED_DN(KSG)                                             \
    switch (ks_dn) {                                                 \
    case 1: return launch_fused_t<KSG, 1>(F, max_units, s);          \
    case 2: return launch_fused_t<KSG, 2>(F, max_units, s);          \
    default: return launch_fused_t<KSG, 4>(F, max_units, s);         \
    }
    switch (ks_gu) {
    case 1: FT_FUSED_DN(1)
    case 2: FT_FUSED_DN(2)
    case 4: FT_FUSED_DN(4)
    default: FT_FUSED_DN(8)
    }
#undef FT_FUSED_DN
}

}  // namespace ftmoe
