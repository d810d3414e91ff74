// Decode-regime grouped GEMV fed by a TMA weight stream: one persistent CTA per SM.
//
// Same arithmetic as the register-fed kernels (exact f16 code*scale weights, f16
// activations staged per block of 8 positions with a power-of-two row scale, m16n8k16
// MMAs with fp32 accumulation, weights as M and the block's 8 positions as N), but the
// weights travel as whole slabs: the producer warp streams, for every unit, the unit's
// rows of packed codes and block scales with tiled TMA copies into a ring of stages,
// so tens of kilobytes per SM are in flight independently of what the math warps do.
//
// Geometry. A "line" is 256 K elements of one weight row (128 code bytes). A "pair
// tile" is 32 rows: gate rows [i, i+16) with up rows I_l + [i, i+16) for gate_up, rows
// [n, n+32) for down. A stage holds 8 (pair tile, line) slots -- TPS pair tiles x LPS
// consecutive lines, LPS = min(K/256, 8) -- i.e. 32 KB of codes plus their scales; 16
// math warps take one tile (16 rows) of one slot each. A unit is (problem, block of 8 positions, group of
// TPS pair tiles) over the whole K, i.e. K/(256 LPS) stages. The math warps only
// multiply: at the end of a unit each drops its partial sums into one of 4 buffers;
// 4 epilogue warps add the partials of each pair tile, apply globals, row scales and
// SwiGLU or routing weights, with their global operands fetched before they wait --
// so the weight stream never waits for an epilogue. The combine is its own launch.
//
// Shared-memory layouts (every read is free of bank conflicts):
//   codes    per stage line: TMA boxes of 128 bytes x 16*TPS rows (gate and up boxes)
//            or 32*TPS rows (down), 128-byte swizzled: 16-byte column q of box row r
//            sits at column q ^ (r & 7). Lane (g, c) reads column 2c + j (j = 0, 1) of
//            rows g and g + 8: 32 codes each.
//   scales   per stage: one box (down) or two (gate_up) of LPS*256/group bytes per row.
//   activ.   fragment-native: 16-byte unit ((2L + j) * 4 + q) * 32 + 4t + c holds the 8
//            f16 values of token t at K offset 256L + 32(2c + j) + 8q, so the B operand
//            of lane (g, c) for column j of line L is 4 consecutive-lane reads.
// Every wait on an mbarrier is bounded (about two seconds): on expiry the CTA records
// FT_ERR_TIMEOUT, finishes its loops without computing, lets issued copies land and
// returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "gemv_common.cuh"
#include "tcgen05.cuh"

namespace ftmoe {

using namespace gemv;

namespace {

constexpr int kSlots = 8;                         // (pair tile, line) slots per stage
constexpr int kMath = 2 * kSlots;                 // math warps: one per slot and tile
constexpr int kEpi = 4;                           // epilogue warps
constexpr int kProducer = kMath + kEpi;           // warp index of the producer
constexpr int kStreamThreads = 32 * (kMath + kEpi + 1);
constexpr int kLine = 256;                        // K elements per line
constexpr uint32_t kStageCodes = 32768;           // 8 slots x 32 rows x 128 bytes
constexpr uint32_t kStagePitch = 36864;           // codes + at most 4 KB of scales
constexpr int kMaxStages = 6;
constexpr int kRed = 4;                           // partial-sum buffers between math and epilogue
constexpr int kRedFloats = kMath * 4 * 32;        // one buffer: [math warp][value][lane]
constexpr int kMaxItems = 4;                      // epilogue items per warp and unit (<= 16 / kEpi)
constexpr int kGlob = 8;                          // ring of per-unit row-global slices
constexpr int kGlobFloats = 256;                  // one slice: at most 32 rows x 8 pair tiles
constexpr uint32_t kRedBytes = kRed * (kRedFloats + 8) * 4 + 8 * 4 + kGlob * kGlobFloats * 4;
constexpr uint32_t kMiscBytes = (2 * kMaxStages + 2 * kRed + 2 * kGlob) * 8 + 16;

__device__ __forceinline__ void math_barrier()
{
    asm volatile("bar.sync 1, %0;" ::"n"(32 * kMath) : "memory");
}

// Fragment-native index of 16-byte chunk u (elements 8u .. 8u+7) of token t.
__device__ __forceinline__ int frag_unit(int u, int t)
{
    const int L = u >> 5, c = (u >> 3) & 3, j = (u >> 2) & 1, q = u & 3;
    return (((2 * L + j) << 2) + q) * 32 + 4 * t + c;
}

// Warp t stages token t of the block: f16 of the source row times 2^-e, inv[t] = 2^e.
__device__ __forceinline__ void stage_token(const uint16_t *__restrict__ src, int K, int row, uint4 *act,
                                            float *inv, int t)
{
    const int lane = threadIdx.x & 31;
    if (row < 0) {
        for (int u = lane; u < K / 8; u += 32) act[frag_unit(u, t)] = make_uint4(0, 0, 0, 0);
        if (lane == 0) inv[t] = 0.f;
        return;
    }
    const uint4 *s4 = reinterpret_cast<const uint4 *>(src + (size_t)row * K);
    float m = 0.f;
    for (int u = lane; u < K / 8; u += 32) {
        const uint4 v = __ldg(s4 + u);
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
    for (int u = lane; u < K / 8; u += 32) {
        const uint4 v = __ldg(s4 + u);
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 hh = __floats2half2_rn(__uint_as_float(w[i] << 16) * down,
                                                 __uint_as_float(w[i] & 0xFFFF0000u) * down);
            h[i] = *reinterpret_cast<const uint32_t *>(&hh);
        }
        act[frag_unit(u, t)] = make_uint4(h[0], h[1], h[2], h[3]);
    }
    if (lane == 0) inv[t] = pow2f(e);
}

// Byte offset of scale byte `off` of box row `r` (128-byte swizzled boxes when sw).
__device__ __forceinline__ uint32_t scale_at(uint32_t off, int r, bool sw)
{
    return sw ? ((((off >> 4) ^ (uint32_t)(r & 7)) << 4) | (off & 15u)) : off;
}

struct UnitPos {
    int pi, blk, pt;
};

struct Geo2 {
    int np0, np1, lps0, lps1, tps0, tps1, nst0, nst1, sb0, sb1;
    __device__ __forceinline__ int np(int pi) const { return pi ? np1 : np0; }
    __device__ __forceinline__ int lps(int pi) const { return pi ? lps1 : lps0; }
    __device__ __forceinline__ int tps(int pi) const { return pi ? tps1 : tps0; }
    __device__ __forceinline__ int nst(int pi) const { return pi ? nst1 : nst0; }
    __device__ __forceinline__ int sb(int pi) const { return pi ? sb1 : sb0; }
};

__device__ __forceinline__ UnitPos unit_pos(const Geo2 &geo, int u, int units0)
{
    UnitPos q;
    q.pi = u < units0 ? 0 : 1;
    const int lu = q.pi ? u - units0 : u;
    const int np = geo.np(q.pi);
    q.blk = lu / np;
    q.pt = lu - q.blk * np;
    return q;
}

}  // namespace

template <bool GATED>
__global__ void __launch_bounds__(kStreamThreads, 1) gemv_stream_kernel(const __grid_constant__ StreamLaunch L)
{
    pdl_enter();
    extern __shared__ unsigned char smem_raw[];
    // 1024-byte aligned base by pointer arithmetic on the shared array itself, so that the
    // compiler keeps every access derived from it in the shared state space
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const int ns = L.ns;
    unsigned char *stages = smem;
    uint4 *act = reinterpret_cast<uint4 *>(smem + (size_t)ns * kStagePitch);
    float *red = reinterpret_cast<float *>(smem + (size_t)ns * kStagePitch + L.act_bytes);  // [kRed][warp][value][lane]
    float *red_inv = red + kRed * kRedFloats;  // [kRed][8]: the unit's activation row scales
    float *inv = red_inv + kRed * 8;           // [8]: the staged block's
    float *glob_ring = inv + 8;                // [kGlob][kGlobFloats]: the unit's row globals
    uint64_t *full = reinterpret_cast<uint64_t *>(glob_ring + kGlob * kGlobFloats);
    uint64_t *empty = full + kMaxStages;
    uint64_t *red_full = empty + kMaxStages, *red_empty = red_full + kRed;
    uint64_t *glob_full = red_empty + kRed, *glob_empty = glob_full + kGlob;
    volatile int *abort_flag = reinterpret_cast<volatile int *>(glob_empty + kGlob);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kMaxStages; ++i) {
            mbar_init(full + i, 1);
            mbar_init(empty + i, kMath);
        }
        for (int i = 0; i < kRed; ++i) {
            mbar_init(red_full + i, kMath);
            mbar_init(red_empty + i, kEpi);
        }
        for (int i = 0; i < kGlob; ++i) {
            mbar_init(glob_full + i, 1);
            mbar_init(glob_empty + i, kEpi);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == kProducer && lane == 0) {
        for (int i = 0; i < L.nprob; ++i) {
            tc::prefetch_map(&L.cmap[i]);
            tc::prefetch_map(&L.smap[i]);
        }
    }
    __syncthreads();

    const int n_pos0 = load_n_pos(L.prob[0].p);
    const int n_pos1 = L.nprob > 1 ? load_n_pos(L.prob[1].p) : 0;
    const int units0 = (n_pos0 / kGemvBlock) * L.prob[0].n_ptiles;
    const int units1 = L.nprob > 1 ? (n_pos1 / kGemvBlock) * L.prob[1].n_ptiles : 0;
    const int n_units = units0 + units1;
    // both problems' geometry in registers (selected, never indexed): unit decoding
    // never touches parameter or local memory
    const Geo2 geo{L.prob[0].n_ptiles, L.prob[1].n_ptiles, L.prob[0].lps, L.prob[1].lps, L.prob[0].tps,
                   L.prob[1].tps, L.prob[0].nst, L.prob[1].nst, L.prob[0].sbytes, L.prob[1].sbytes};
    const int u_lo = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_hi = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    constexpr int tile_rows = GATED ? 16 : 32;  // rows of one pair tile per box side
    const int g = lane >> 2, c = lane & 3;
    bool dead = false;

    if (warp == kProducer) {
        // ------------------------------------------------------------ producer
        if (lane != 0) return;
        const uint8_t *codes0 = L.prob[0].p.codes, *codes1 = L.prob[1].p.codes;
        const int K0 = L.prob[0].p.K, K1 = L.prob[1].p.K;
        int it = 0, n_glob = 0;
        for (int u = u_lo; u < u_hi && !dead; ++u) {
            const UnitPos q = unit_pos(geo, u, units0);
            const StreamProb &P = L.prob[q.pi];
            // problem fields in registers (the barrier operations clobber memory)
            const int lps = geo.lps(q.pi), tps = geo.tps(q.pi), nst = geo.nst(q.pi), sbytes = geo.sb(q.pi);
            const int up_off = P.p.up_off;
            const int e = P.p.block_expert ? __ldg(P.p.block_expert + q.blk) : 0;
            const int row0 = e * P.p.R + q.pt * tile_rows * tps;
            {
                // the unit's row globals for the epilogue: gate rows then up rows, or the
                // 32 TPS rows of down
                const int gslot = (u - u_lo) % kGlob;
                const uint32_t guse = (uint32_t)((u - u_lo) / kGlob);
                if (!mbar_wait_timed(glob_empty + gslot, (guse & 1) ^ 1, abort_flag)) { dead = true; break; }
                const uint32_t run = 4u * tile_rows * tps;
                float *gdst = glob_ring + gslot * kGlobFloats;
                mbar_arrive_expect_tx(glob_full + gslot, GATED ? 2 * run : run);
                bulk_g2s(gdst, P.p.glob + row0, run, glob_full + gslot);
                if (GATED) bulk_g2s(gdst + tile_rows * tps, P.p.glob + row0 + up_off, run, glob_full + gslot);
                ++n_glob;
            }
            for (int st = 0; st < nst; ++st, ++it) {
                const int slot = it % ns;
                if (!mbar_wait_timed(empty + slot, ((it / ns) & 1) ^ 1, abort_flag)) { dead = true; break; }
                unsigned char *stg = stages + (size_t)slot * kStagePitch;
                mbar_arrive_expect_tx(full + slot, kStageCodes + 32u * tps * sbytes);
                if (GATED) {
                    // codes as plain bulk copies, row segments of lps*128 bytes packed
                    // back to back: gate rows then up rows (16 KB each)
                    const uint32_t seg = (uint32_t)lps * 128u, rowb = (uint32_t)(q.pi ? K1 : K0) / 2u;
                    const int rows = 16 * tps;
                    const uint8_t *cg = (q.pi ? codes1 : codes0) + (size_t)row0 * rowb + (size_t)st * seg;
                    const uint8_t *cu = cg + (size_t)up_off * rowb;
                    if (seg == rowb) {  // whole rows: one contiguous run per side
                        bulk_g2s(stg, cg, rows * seg, full + slot);
                        bulk_g2s(stg + rows * seg, cu, rows * seg, full + slot);
                    } else {
                        for (int r = 0; r < rows; ++r) {
                            bulk_g2s(stg + r * seg, cg + (size_t)r * rowb, seg, full + slot);
                            bulk_g2s(stg + (rows + r) * seg, cu + (size_t)r * rowb, seg, full + slot);
                        }
                    }
                } else {
                    for (int l = 0; l < lps; ++l) {
                        const int x = (st * lps + l) * 128;
                        tc::tma_load_2d(stg + (size_t)l * 4096 * tps, &L.cmap[q.pi], x, row0, full + slot);
                    }
                }
                unsigned char *sdst = stg + kStageCodes;
                tc::tma_load_2d(sdst, &L.smap[q.pi], st * sbytes, row0, full + slot);
                if (GATED)
                    tc::tma_load_2d(sdst + 16 * tps * sbytes, &L.smap[q.pi], st * sbytes, row0 + up_off, full + slot);
            }
        }
        if (dead) {
            raise_status(L.prob[0].p.status, FT_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        // let every issued copy land before the CTA's shared memory can be released
        for (int i = 0; i < ns && i < it; ++i) {
            const int last = it - 1 - i;
            mbar_wait_timed(full + last % ns, (last / ns) & 1, nullptr);
        }
        for (int i = 0; i < kGlob && i < n_glob; ++i) {
            const int last = n_glob - 1 - i;
            mbar_wait_timed(glob_full + last % kGlob, (last / kGlob) & 1, nullptr);
        }
        return;
    }

    if (warp >= kMath) {
        // ------------------------------------------------------------ epilogue warps
        // Unit by unit: add the math warps' partial sums of each item this warp owns,
        // apply globals, row scales and SwiGLU (gate_up) or routing weights and the fused
        // combine (down). An item is (pair tile, position parity): values i = parity and
        // parity + 2, i.e. all 32 rows of the pair tile for 4 of the block's positions,
        // which is what the combine counts per 32-row group.
        const int ew = warp - kMath;
        int ru = 0, cached = -1;
        int dst_c[2] = {-1, -1};
        float wgt_c[2] = {0.f, 0.f};
        for (int u = u_lo; u < u_hi; ++u, ++ru) {
            const UnitPos q = unit_pos(geo, u, units0);
            const StreamProb &P = L.prob[q.pi];
            const GemvParams &p = P.p;
            const int lps = geo.lps(q.pi), tps = geo.tps(q.pi);
            const int n_pos = q.pi ? n_pos1 : n_pos0;
            const int n_items = 2 * tps;  // <= kEpi * kMaxItems
            const int b = ru % kRed;
            const uint32_t use = (uint32_t)(ru / kRed);
            const int gslot = ru % kGlob;
            const uint32_t guse = (uint32_t)(ru / kGlob);
            const int key = (q.pi << 30) | q.blk;
            if (!GATED && key != cached) {
                // slots and routing weights of positions 2c, 2c+1 of the block
                cached = key;
#pragma unroll
                for (int par = 0; par < 2; ++par) {
                    const int pos = q.blk * kGemvBlock + 2 * c + par;
                    int dst = -1;
                    float w = 1.f;
                    if (pos < n_pos) {
                        if (p.sorted_slot) {
                            dst = __ldg(p.sorted_slot + pos);
                            if (dst >= p.n_slots) dst = -1;
                            else if (p.route_w) w = __ldg(p.route_w + dst);
                        } else if (pos < p.n_pos_static) {
                            dst = pos;
                        }
                    }
                    dst_c[par] = dst;
                    wgt_c[par] = w;
                }
            }
            if (!dead && !mbar_wait_timed(glob_full + gslot, guse & 1, abort_flag)) dead = true;
            const float *gl = glob_ring + gslot * kGlobFloats;
            if (!dead && !mbar_wait_timed(red_full + b, use & 1, abort_flag)) dead = true;
            const float *rb = red + b * kRedFloats;
            const float *rinv = red_inv + b * 8;
#pragma unroll
            for (int k2 = 0; k2 < kMaxItems; ++k2) {
                const int idx = ew + kEpi * k2;
                if (idx >= n_items) break;
                if (GATED) {
                    const int sp = idx >> 1, par = idx & 1;
                    const int t = 2 * c + par;
                    const float scl = rinv[t];
                    uint16_t *hrow = p.h_out + (size_t)(q.blk * kGemvBlock + t) * p.h_ld + (q.pt * tps + sp) * 16;
#pragma unroll
                    for (int h2 = 0; h2 < 2; ++h2) {
                        const int i = par + 2 * h2;
                        float a = 0.f, bb = 0.f;
                        for (int w = sp * lps; w < (sp + 1) * lps; ++w) {
                            a += rb[(w * 4 + i) * 32 + lane];
                            bb += rb[((kSlots + w) * 4 + i) * 32 + lane];
                        }
                        const float gate = a * scl * gl[sp * 16 + g + 8 * h2];
                        const float up = bb * scl * gl[16 * tps + sp * 16 + g + 8 * h2];
                        __nv_bfloat16 hv = __float2bfloat16_rn(silu(gate) * up);
                        hrow[g + 8 * h2] = *reinterpret_cast<uint16_t *>(&hv);
                    }
                } else {
                    const int sp = idx >> 1, par = idx & 1;
                    const int r0 = (q.pt * tps + sp) * 32;
                    const int dst = par ? dst_c[1] : dst_c[0];
                    if (dst >= 0) {
                        const float wgt = (par ? wgt_c[1] : wgt_c[0]) * rinv[2 * c + par];
                        float *yrow = p.y_out + (size_t)dst * p.R;
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const int i = par + 2 * h2;
                            float a = 0.f, bb = 0.f;
                            for (int w = sp * lps; w < (sp + 1) * lps; ++w) {
                                a += rb[(w * 4 + i) * 32 + lane];
                                bb += rb[((kSlots + w) * 4 + i) * 32 + lane];
                            }
                            yrow[r0 + g + 8 * h2] = a * gl[sp * 32 + g + 8 * h2] * wgt;
                            yrow[r0 + 16 + g + 8 * h2] = bb * gl[sp * 32 + 16 + g + 8 * h2] * wgt;
                        }
                    }
                }
            }
            __syncwarp();
            if (lane == 0) {
                mbar_arrive(red_empty + b);
                mbar_arrive(glob_empty + gslot);
            }
        }
        if (dead) {
            raise_status(L.prob[0].p.status, FT_ERR_TIMEOUT);
            *abort_flag = 1;
        }
        return;
    }

    // ---------------------------------------------------------------- math warps
    // warp = tile * kSlots + slot: one tile (gate / first 16 rows, or up / last 16 rows)
    // of one (pair tile, line) slot of every stage
    const int slot_id = warp % kSlots, tile = warp / kSlots;
    const int group = L.prob[0].p.group;  // the same for both problems
    int it = 0, staged = -1, ru = 0;
    for (int u = u_lo; u < u_hi; ++u, ++ru) {
        const UnitPos q = unit_pos(geo, u, units0);
        const int lps = geo.lps(q.pi), tps = geo.tps(q.pi), nst = geo.nst(q.pi), sbytes = geo.sb(q.pi);
        const int key = (q.pi << 30) | q.blk;
        if (key != staged) {
            const GemvParams &p = L.prob[q.pi].p;
            const int n_pos = q.pi ? n_pos1 : n_pos0;
            math_barrier();
            if (warp < kGemvBlock)
                stage_token(p.act, p.K, source_row(p, q.blk * kGemvBlock + warp, n_pos, GATED), act, inv, warp);
            math_barrier();
            staged = key;
        }
        const int sp = slot_id / lps, sl = slot_id - sp * lps;  // this warp's (pair tile, line) slot
        const bool sw = sbytes == 128;
        // box row of this warp's tile, row g: gate / up boxes side by side (gate_up), or
        // rows 0..15 / 16..31 of the pair tile (down)
        const int rt = GATED ? 16 * sp + g : 32 * sp + 16 * tile + g;
        const uint32_t stile_off = GATED ? (uint32_t)tile * 16u * tps * sbytes : 0u;
        const uint32_t soff = group == 16 ? 16u * sl + 4u * c : 8u * sl + 2u * c;
        const uint32_t s_lo = scale_at(soff, rt, sw), s_hi = scale_at(soff, rt + 8, sw);
        // two accumulator chains (columns j = 0, 1), added at the end
        float acc[2][4] = {};
        for (int st = 0; st < nst; ++st, ++it) {
            const int slot = it % ns;
            if (!dead && !mbar_wait_timed(full + slot, (it / ns) & 1, abort_flag)) dead = true;
            if (!dead) {
                const unsigned char *stg = stages + (size_t)slot * kStagePitch;
                // gate_up: linear rows of lps*128 bytes (gate block, then up block);
                // down: 128-byte swizzled TMA boxes, one per line
                const unsigned char *tr = GATED ? stg + (size_t)(tile * 16 * tps + rt) * (lps * 128) + sl * 128
                                                : stg + (size_t)sl * 4096 * tps + rt * 128;
                const unsigned char *sr = stg + kStageCodes + stile_off + rt * sbytes;
                uint32_t s_g, s_g8;  // scale bytes of rows g, g+8 for columns j = 0, 1
                if (group == 16) {
                    s_g = *reinterpret_cast<const uint32_t *>(sr + s_lo);
                    s_g8 = *reinterpret_cast<const uint32_t *>(sr + 8 * sbytes + s_hi);
                } else {
                    // one scale byte per 32-element column: duplicate it for both halves
                    const uint32_t v0 = *reinterpret_cast<const uint16_t *>(sr + s_lo);
                    const uint32_t v1 = *reinterpret_cast<const uint16_t *>(sr + 8 * sbytes + s_hi);
                    s_g = ((v0 & 0xFFu) * 0x0101u) | (((v0 >> 8) * 0x0101u) << 16);
                    s_g8 = ((v1 & 0xFFu) * 0x0101u) | (((v1 >> 8) * 0x0101u) << 16);
                }
                const int Lg = st * lps + sl;  // line index along K
                const int row8 = GATED ? 8 * lps * 128 : 8 * 128;  // bytes to row g + 8
#pragma unroll
                for (int j = 0; j < 2; ++j) {
                    const int col = (GATED ? (2 * c + j) : ((2 * c + j) ^ g)) << 4;
                    const uint4 lo = *reinterpret_cast<const uint4 *>(tr + col);
                    const uint4 hi = *reinterpret_cast<const uint4 *>(tr + row8 + col);
                    uint4 bv[4];
#pragma unroll
                    for (int qq = 0; qq < 4; ++qq) bv[qq] = act[(((2 * Lg + j) << 2) + qq) * 32 + lane];
                    const int sh = 16 * j;
                    mma_step(lo, hi, (s_g >> sh) & 0xFFFFu, (s_g8 >> sh) & 0xFFFFu, bv, acc[j]);
                }
            }
            // every value read from the slot has been consumed: hand it back to the producer
            __syncwarp();
            if (lane == 0) mbar_arrive(empty + slot);
        }
        // partial sums to the epilogue warps
        const int b = ru % kRed;
        const uint32_t use = (uint32_t)(ru / kRed);
        if (!dead && !mbar_wait_timed(red_empty + b, (use & 1) ^ 1, abort_flag)) dead = true;
        float *rb = red + b * kRedFloats;
#pragma unroll
        for (int i = 0; i < 4; ++i) rb[(warp * 4 + i) * 32 + lane] = acc[0][i] + acc[1][i];
        if (warp == 0 && lane < 8) red_inv[b * 8 + lane] = inv[lane];
        __syncwarp();
        if (lane == 0) mbar_arrive(red_full + b);
    }
    if (dead) {
        raise_status(L.prob[0].p.status, FT_ERR_TIMEOUT);
        *abort_flag = 1;
    }
}

// ---------------------------------------------------------------- host side

bool gemv_stream_geom(int K, int group, int rows, bool gated, StreamProb &P)
{
    if (K % kLine || (group != 16 && group != 32)) return false;
    const int nl = K / kLine;
    P.lps = nl < kSlots ? nl : kSlots;
    if (nl % P.lps || kSlots % P.lps) return false;
    P.tps = kSlots / P.lps;
    P.nst = nl / P.lps;
    P.sbytes = P.lps * kLine / group;
    if (P.sbytes % 16 || (K / group) % 16) return false;
    const int pt_rows = (gated ? 16 : 32) * P.tps;
    if (rows % pt_rows) return false;
    P.n_ptiles = rows / pt_rows;
    return true;
}

static int stream_stages(int act_bytes)
{
    int dev = 0, optin = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess) return 0;
    const long room = (long)optin - 1024 - act_bytes - kRedBytes - kMiscBytes;
    long ns = room / (long)kStagePitch;
    if (ns > kMaxStages) ns = kMaxStages;
    return ns < 2 ? 0 : (int)ns;
}

bool gemv_stream_fits(int Kmax) { return stream_stages(kGemvBlock * Kmax * 2) >= 2; }

cudaError_t launch_gemv_stream(StreamLaunch &L, bool gated, int max_units, cudaStream_t s)
{
    int Kmax = 0;
    for (int i = 0; i < L.nprob; ++i) {
        const StreamProb &P = L.prob[i];
        const GemvParams &p = P.p;
        if (p.K > Kmax) Kmax = p.K;
        const uint32_t box_rows = (gated ? 16u : 32u) * P.tps;
        const uint64_t rows_total = (uint64_t)p.num_experts * p.R;
        if (!make_tensor_map_2d(&L.cmap[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.codes, (uint64_t)p.K / 2, rows_total,
                                (uint64_t)p.K / 2, 128, box_rows, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tensor_map_2d(&L.smap[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.scales, (uint64_t)p.K / p.group,
                                rows_total, (uint64_t)p.K / p.group, (uint32_t)P.sbytes, box_rows,
                                P.sbytes == 128 ? CU_TENSOR_MAP_SWIZZLE_128B : CU_TENSOR_MAP_SWIZZLE_NONE))
            return cudaErrorInvalidValue;
    }
    L.act_bytes = kGemvBlock * Kmax * 2;
    L.ns = stream_stages(L.act_bytes);
    if (!L.ns) return cudaErrorInvalidValue;
    const size_t smem = 1024 + (size_t)L.ns * kStagePitch + L.act_bytes + kRedBytes + kMiscBytes;
    auto kern = gated ? gemv_stream_kernel<true> : gemv_stream_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    int grid = sm_count();
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    FT_LAUNCH(kern, dim3(grid), dim3(kStreamThreads), smem, s, L);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
