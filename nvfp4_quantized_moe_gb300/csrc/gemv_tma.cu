// Decode-regime grouped GEMV fed by bulk copies (TMA engine) into shared memory.
//
// Same arithmetic as the register-fed kernel in gemv.cu (exact f16 code*scale weights,
// f16 activations staged per block with a power-of-two row scale, m16n8k16 MMAs with
// fp32 accumulation, weights as M and the block's 8 tokens as N), but the weight
// stream moves with cp.async.bulk: every warp owns a ring of R stages in shared memory;
// a stage holds one K chunk (KC elements) of 32 weight rows -- a gate tile and its up
// tile for gate_up, two consecutive 16-row tiles for down -- plus their block scales.
// Each of the 32 lanes copies one row segment into a padded layout (row pitch
// KC/2 + 64 bytes) that keeps the fragment reads free of bank conflicts, and the warp
// keeps copies for its next stages in flight while it computes, across unit
// boundaries. Waits on the stage barriers are bounded: on expiry the kernel records
// FT_ERR_TIMEOUT, stops computing, drains its own copies and returns.
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "gemv_common.cuh"

namespace ftmoe {

using namespace gemv;

namespace {

constexpr int kRing = 2;                 // stages per warp
constexpr uint32_t kWaitLimit = 1u << 22;  // polls before a stage wait gives up

struct TmaLayout {
    int KC, CP, SP, stage_bytes;  // K chunk, code pitch, scale pitch, bytes per stage
};

__device__ __forceinline__ TmaLayout tma_layout(int KC, int group)
{
    TmaLayout L;
    L.KC = KC;
    L.CP = KC / 2 + 64;
    L.SP = KC / group;
    L.stage_bytes = 32 * L.CP + 32 * L.SP;
    return L;
}

}  // namespace

// GATED: a warp pair-tile is gate rows [i0, i0+16) and up rows I_l + [i0, i0+16);
// otherwise rows [n0, n0+32). CTA = NW warps = TPW pair-tiles x KS K-splits.
template <bool GATED, int KS>
__global__ void __launch_bounds__(256, 1) gemv_tma_kernel(const GemvParams p, int KC)
{
    extern __shared__ __align__(128) unsigned char smem[];
    __shared__ float inv[kGemvBlock];
    __shared__ int rows[kGemvBlock];
    __shared__ float red[KS > 1 ? 8 : 1][32][8];
    const int NW = blockDim.x >> 5, TPW = NW / KS;
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    const int ks = warp % KS, tp = warp / KS;
    const int g = lane >> 2, c = lane & 3;
    const int Kp = (p.K + kStep - 1) / kStep * kStep;
    const TmaLayout L = tma_layout(KC, p.group);
    uint4 *sm_b = reinterpret_cast<uint4 *>(smem);
    unsigned char *ring = smem + (size_t)kGemvBlock * Kp * 2 + (size_t)warp * kRing * L.stage_bytes;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + (size_t)kGemvBlock * Kp * 2 +
                                                  (size_t)NW * kRing * L.stage_bytes) + warp * kRing;
    if (lane < kRing) mbar_init(bars + lane, 1);
    fence_mbar_init();
    __syncthreads();

    const int n_pos = load_n_pos(p);
    const int n_groups = p.n_tiles;
    const int n_units = (n_pos / kGemvBlock) * n_groups;
    const int u_lo = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_hi = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    const int Kw = p.K / KS;
    const int NS = Kw / KC;  // stages per unit (host guarantees Kw % KC == 0)
    const int rows_limit = GATED ? p.up_off : p.R;
    const int pair_rows = GATED ? 16 : 32;

    // first weight row of this warp's pair-tile in unit u, or -1 when out of range
    auto pair_row0 = [&](int u) {
        const int grp = u % n_groups;
        const int r0 = (grp * TPW + tp) * pair_rows;
        return r0 < rows_limit ? r0 : -1;
    };
    auto unit_expert = [&](int u) {
        const int blk = u / n_groups;
        return p.block_expert ? __ldg(p.block_expert + blk) : 0;
    };

    // issue cursor over this warp's stages (units with an in-range pair-tile only)
    int iu = u_lo, ich = 0, issued = 0;
    auto skip_invalid = [&]() {
        while (iu < u_hi && pair_row0(iu) < 0) { ++iu; ich = 0; }
    };
    auto issue_next = [&]() {
        skip_invalid();
        if (iu >= u_hi) return false;
        const int slot = issued % kRing;
        unsigned char *st = ring + (size_t)slot * L.stage_bytes;
        const int e = unit_expert(iu), r0 = pair_row0(iu);
        const int kc0 = ks * Kw + ich * KC;
        const int seg = lane;  // 0..31
        int row;
        if (GATED) row = (seg < 16) ? r0 + seg : p.up_off + r0 + (seg - 16);
        else row = r0 + seg;
        const uint8_t *csrc = p.codes + (size_t)e * p.e_codes + (size_t)row * (p.K / 2) + kc0 / 2;
        const uint8_t *ssrc = p.scales + (size_t)e * p.e_scales + (size_t)row * (p.K / p.group) + kc0 / p.group;
        if (lane == 0) mbar_arrive_expect_tx(bars + slot, (uint32_t)(32 * (KC / 2 + L.SP)));
        __syncwarp();
        bulk_g2s(st + seg * L.CP, csrc, KC / 2, bars + slot);
        bulk_g2s(st + 32 * L.CP + seg * L.SP, ssrc, L.SP, bars + slot);
        ++issued;
        if (++ich == NS) { ich = 0; ++iu; }
        return true;
    };
    for (int i = 0; i < kRing; ++i)
        if (!issue_next()) break;

    int consumed = 0;
    bool dead = false;
    int staged = -1;
    for (int u = u_lo; u < u_hi; ++u) {
        const int blk = u / n_groups;
        if (blk != staged) {
            __syncthreads();
            if (threadIdx.x < kGemvBlock)
                rows[threadIdx.x] = source_row(p, blk * kGemvBlock + threadIdx.x, n_pos, GATED);
            __syncthreads();
            stage_block(p.act, p.K, Kp, rows, sm_b, inv);
            __syncthreads();
            staged = blk;
        }
        const int r0 = pair_row0(u);
        float acc0[4] = {0.f, 0.f, 0.f, 0.f}, acc1[4] = {0.f, 0.f, 0.f, 0.f};
        if (r0 >= 0) {
            const uint4 *brow = sm_b + (size_t)g * (Kp / 8);
            for (int ch = 0; ch < NS; ++ch) {
                if (dead) continue;
                const int slot = consumed % kRing;
                const uint32_t parity = (uint32_t)(consumed / kRing) & 1u;
                if (!mbar_wait_bounded(bars + slot, parity, kWaitLimit)) {
                    dead = true;
                    if (lane == 0) raise_status(p.status, FT_ERR_TIMEOUT);
                    continue;
                }
                {
                    const unsigned char *st = ring + (size_t)slot * L.stage_bytes;
                    const unsigned char *sc = st + 32 * L.CP;
                    const int kc0 = ks * Kw + ch * KC;
                    for (int s = 0; s < KC / kStep; ++s) {
                        const int off = 64 * s + 16 * c;
                        const uint4 a0 = *reinterpret_cast<const uint4 *>(st + g * L.CP + off);
                        const uint4 a1 = *reinterpret_cast<const uint4 *>(st + (g + 8) * L.CP + off);
                        const uint4 a2 = *reinterpret_cast<const uint4 *>(st + (g + 16) * L.CP + off);
                        const uint4 a3 = *reinterpret_cast<const uint4 *>(st + (g + 24) * L.CP + off);
                        const int q0 = (kStep * s + 32 * c) / p.group, q1 = (kStep * s + 32 * c + 16) / p.group;
                        const uint32_t s0 = sc[g * L.SP + q0] | (uint32_t)sc[g * L.SP + q1] << 8;
                        const uint32_t s1 = sc[(g + 8) * L.SP + q0] | (uint32_t)sc[(g + 8) * L.SP + q1] << 8;
                        const uint32_t s2 = sc[(g + 16) * L.SP + q0] | (uint32_t)sc[(g + 16) * L.SP + q1] << 8;
                        const uint32_t s3 = sc[(g + 24) * L.SP + q0] | (uint32_t)sc[(g + 24) * L.SP + q1] << 8;
                        uint4 b[4];
                        load_b(brow, (kc0 + kStep * s) / 8 + 4 * c, g, b);
                        mma_step(a0, a1, s0, s1, b, acc0);
                        mma_step(a2, a3, s2, s3, b, acc1);
                    }
                }
                ++consumed;
                __syncwarp();
                fence_proxy_async_smem();
                issue_next();
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
        if (ks == 0 && r0 >= 0 && !dead) {
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
            const int e = unit_expert(u);
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
    // drain: copies still in flight into this warp's ring must land before exit
    while (consumed < issued) {
        const int slot = consumed % kRing;
        mbar_wait_bounded(bars + slot, (uint32_t)(consumed / kRing) & 1u, kWaitLimit);
        ++consumed;
    }
}

// ---------------------------------------------------------------- host side

// Chunk of K moved per stage, or 0 when this shape needs the register-fed kernel:
// segments must be 16-byte multiples on 16-byte boundaries.
int gemv_tma_chunk(int K, int group, int ks)
{
    if (K % (16 * group) || (K / ks) % kStep) return 0;
    const int Kw = K / ks;
    for (int kc : {512, 256}) {
        if (kc < 16 * group) continue;
        if (Kw % kc == 0) return kc;
    }
    return 0;
}

static size_t tma_smem(int K, int group, int kc, int nw)
{
    const int Kp = (K + kStep - 1) / kStep * kStep;
    const size_t stage = 32 * (size_t)(kc / 2 + 64) + 32 * (size_t)(kc / group);
    return (size_t)kGemvBlock * Kp * 2 + (size_t)nw * kRing * stage + (size_t)nw * kRing * 8;
}

// Warps per CTA (8, or 4 when 8 do not fit in shared memory); 0 if neither fits.
int gemv_tma_warps(int K, int group, int kc)
{
    int optin = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    const size_t static_smem = 8 * 32 * 8 * 4 + 128;
    for (int nw : {8, 4})
        if (tma_smem(K, group, kc, nw) + static_smem <= (size_t)optin) return nw;
    return 0;
}

template <bool GATED, int KS>
static cudaError_t launch_tma_t(const GemvParams &p, int kc, int nw, int max_units, cudaStream_t s)
{
    auto kern = gemv_tma_kernel<GATED, KS>;
    const size_t smem = tma_smem(p.K, p.group, kc, nw);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int grid = sm_count();
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    kern<<<grid, nw * 32, smem, s>>>(p, kc);
    count_launches(1);
    return cudaGetLastError();
}

cudaError_t launch_gemv_tma(const GemvParams &p, bool gated, int ks, int kc, int nw, int max_units, cudaStream_t s)
{
    if (gated) {
        switch (ks) {
        case 1: return launch_tma_t<true, 1>(p, kc, nw, max_units, s);
        case 2: return launch_tma_t<true, 2>(p, kc, nw, max_units, s);
        case 4: return launch_tma_t<true, 4>(p, kc, nw, max_units, s);
        default: return launch_tma_t<true, 8>(p, kc, nw, max_units, s);
        }
    }
    switch (ks) {
    case 1: return launch_tma_t<false, 1>(p, kc, nw, max_units, s);
    case 2: return launch_tma_t<false, 2>(p, kc, nw, max_units, s);
    case 4: return launch_tma_t<false, 4>(p, kc, nw, max_units, s);
    default: return launch_tma_t<false, 8>(p, kc, nw, max_units, s);
    }
}

}  // namespace ftmoe
