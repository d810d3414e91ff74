// Decode-regime grouped GEMV on the 5th-generation tensor cores, A operand in tensor memory.
//
// Same arithmetic as the register-fed decode kernels: the exact f16 code*scale weights
// against f16 activation rows staged with a power-of-two row scale, fp32 accumulation,
// weights as M and a block of 8 expert-sorted positions as N (MMA N = 16; columns 8..15
// read the neighbouring rows of the staged block and are never used). A unit is (block,
// two 128-row tiles): gate rows i0.. and the matching up rows I_l + i0.. for gate_up (so
// SwiGLU fuses into the epilogue), rows n0.. and n0 + 128.. for down. The routed experts
// and the shared expert are two problems of one launch. Persistent CTA, one per SM:
//   warp 0      one thread streams the packed codes of both tiles by TMA, 256 K elements
//               (128 bytes per row, 128-byte swizzle) per stage;
//   warps 1, 2  warp 1 allocates tensor memory; one thread of each issues tcgen05.mma
//               (kind::f16, A from tensor memory, B = the staged block in shared memory,
//               M = 128, N = 16, K = 16) for one of the two tiles and its accumulator, and
//               commits to the buffer barriers (each counts both issuers);
//   warps 4..7  stage the block's activation rows into shared memory (f16, K-major,
//               128-byte swizzled) ahead of use, and run the epilogue: one TMEM lane =
//               one weight row per thread, globals, row scales, SwiGLU or routing weight
//               (the combine follows as its own launch);
//   warps 8..23 dequantise: warp (quarter q, operand, half) owns rows 32q .. 32q+31 of its
//               tile; per 128-element sub-stage each thread converts 64 codes of its row
//               (its half) with their block scales (read from global memory, two stages
//               ahead) and writes 32 TMEM columns with tcgen05.st -- no shared-memory round
//               trip for the dequantised operand, no per-warp MMA issue.
// Every wait is bounded; on expiry the CTA records FT_ERR_TIMEOUT and winds down.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "gemv_common.cuh"
#include "tcgen05.cuh"

namespace ftmoe {

using namespace gemv;

namespace {

constexpr int kTM = 128;                      // rows per operand tile (TMEM lanes)
constexpr int kTN = 16;                       // MMA N
constexpr int kSK = 256;                      // K elements per TMA stage
constexpr int kSubK = 128;                    // K elements per tensor-memory A buffer
constexpr int kNA = 3;                        // A buffers (128 columns each: two operands)
constexpr int kNSMax = 4;                     // TMA stages (at most)
constexpr int kStageBytes = 2 * kTM * 128;    // both operand tiles of one stage
// warps 0-3 issue the MMAs (the issue cost of a tcgen05.mma is per issuing thread, so four
// issuers, one per accumulator, quadruple the rate; warp 0 also issues the TMA loads),
// warps 4-7 staging and epilogue (TMEM quarters 0-3), warps 8-23 dequantisation (four per
// TMEM quarter)
constexpr int kNumMma = 4, kWarpEpi0 = 4, kWarpDq0 = 8, kNumDq = 16;
constexpr int kThreadsTg = 32 * (kWarpDq0 + kNumDq);
constexpr uint32_t kColD = kNA * 128;         // first accumulator column: two x (4 x 16)
constexpr uint32_t kTmemCols = 512;

struct TgSmem {
    uint32_t b_off, b_bytes, inv_off, bar_off, total;
    int ns;
};

// Stages first (1024-aligned), then two staged-activation buffers of kmax/64 + 1 atoms
// (8 rows x 128 bytes each; the extra atom is what MMA columns 8..15 of the last K step
// read), four position tables (block kb uses table kb % 4: per position the factor the
// epilogue applies -- row scale, times the routing weight for down -- and the destination
// slot of down, -1 for padding), the barriers.
__host__ __device__ inline TgSmem tg_smem(int kmax, int ns)
{
    TgSmem s;
    s.ns = ns;
    s.b_bytes = (uint32_t)(kmax / 64 + 1) * 1024;
    s.b_off = (uint32_t)ns * kStageBytes;
    s.inv_off = s.b_off + 2 * s.b_bytes;
    s.bar_off = s.inv_off + 2 * 4 * kGemvBlock * 4;
    s.total = s.bar_off + 512;
    return s;
}

__device__ __forceinline__ bool warp_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    const bool ok = mbar_wait_timed(bar, parity, abort_flag);
    return __all_sync(0xFFFFFFFFu, ok);
}

__device__ __forceinline__ void epi_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

struct Unit {
    int pi, blk, rt, e;
};

__device__ __forceinline__ Unit unit_at(const FastLaunch &L, int units0, int u)
{
    Unit I;
    I.pi = u < units0 ? 0 : 1;
    const GemvParams &p = L.prob[I.pi];
    const int lu = I.pi ? u - units0 : u;
    I.blk = lu / p.n_tiles;
    I.rt = lu - I.blk * p.n_tiles;
    I.e = p.block_expert ? __ldg(p.block_expert + I.blk) : 0;
    return I;
}

// First local row of operand `op` (0, 1) of the unit's tiles.
template <bool GATED>
__device__ __forceinline__ int tile_row(const GemvParams &p, int rt, int op)
{
    return GATED ? (op ? p.up_off : 0) + rt * kTM : rt * 2 * kTM + op * kTM;
}

// One activation row (bf16, length K; null = padding) into row r8 of a staged block: f16
// scaled by 2^-e with the row maximum in [2^14, 2^15), 64-element atoms of 8 rows x 128
// bytes, 16-byte chunks swizzled with the row. Returns 2^e (0 for padding). Called by a
// whole warp; a lane issues all loads of a batch before their first use (rows up to 1024
// elements are read once and kept in registers; longer rows are read twice).
__device__ __forceinline__ float stage_row_sw128(const uint16_t *row, int K, unsigned char *bb, int r8)
{
    constexpr int kU = 4;  // 16-byte chunks per lane per batch
    const int lane = threadIdx.x & 31;
    const int nch = K / 8;
    auto put = [&](int c, uint4 o) {
        *reinterpret_cast<uint4 *>(bb + (c >> 3) * 1024 + r8 * 128 + (((c & 7) ^ r8) << 4)) = o;
    };
    if (!row) {
        for (int c = lane; c < nch; c += 32) put(c, make_uint4(0, 0, 0, 0));
        return 0.f;
    }
    const uint4 *s4 = reinterpret_cast<const uint4 *>(row);
    auto rowmax = [&](const uint4 &v, float m) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int i = 0; i < 4; ++i)
            m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)), fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
        return m;
    };
    auto convert = [&](const uint4 &v, float down) {
        const uint32_t w[4] = {v.x, v.y, v.z, v.w};
        uint32_t h[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const __half2 hh = __floats2half2_rn(__uint_as_float(w[i] << 16) * down,
                                                 __uint_as_float(w[i] & 0xFFFF0000u) * down);
            h[i] = *reinterpret_cast<const uint32_t *>(&hh);
        }
        return make_uint4(h[0], h[1], h[2], h[3]);
    };
    uint4 v[kU];
    float m = 0.f;
    for (int base = 0; base < nch; base += 32 * kU) {
#pragma unroll
        for (int i = 0; i < kU; ++i) {
            const int c = base + lane + 32 * i;
            v[i] = c < nch ? __ldg(s4 + c) : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int i = 0; i < kU; ++i) m = rowmax(v[i], m);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xFFFFFFFFu, m, off));
    const int e = row_scale_exp(m);
    const float down = pow2f(-e);
    if (nch <= 32 * kU) {  // the whole row is still in registers
#pragma unroll
        for (int i = 0; i < kU; ++i) {
            const int c = lane + 32 * i;
            if (c < nch) put(c, convert(v[i], down));
        }
    } else {
        for (int base = 0; base < nch; base += 32 * kU) {
#pragma unroll
            for (int i = 0; i < kU; ++i) {
                const int c = base + lane + 32 * i;
                v[i] = c < nch ? __ldg(s4 + c) : make_uint4(0, 0, 0, 0);
            }
#pragma unroll
            for (int i = 0; i < kU; ++i) {
                const int c = base + lane + 32 * i;
                if (c < nch) put(c, convert(v[i], down));
            }
        }
    }
    return pow2f(e);
}

}  // namespace

template <bool GATED>
__global__ void __launch_bounds__(kThreadsTg, 1)
    tc_gemv_kernel(const __grid_constant__ CUtensorMap cmap0, const __grid_constant__ CUtensorMap cmap1,
                   const __grid_constant__ FastLaunch L, int ns, int kmax)
{
    pdl_enter();
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const TgSmem S = tg_smem(kmax, ns);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + S.bar_off);
    uint64_t *full = bars, *empty = bars + kNSMax, *a_full = bars + 2 * kNSMax, *a_empty = a_full + kNA;
    uint64_t *acc_full = a_empty + kNA, *acc_empty = acc_full + 2, *b_full = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(b_full + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    float *inv_tbl = reinterpret_cast<float *>(smem + S.inv_off);            // [4][8]
    int *dst_tbl = reinterpret_cast<int *>(smem + S.inv_off) + 4 * kGemvBlock;  // [4][8]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int i = 0; i < kNSMax; ++i) { mbar_init(full + i, 1); mbar_init(empty + i, kNumDq); }
        // an A buffer is read by the two issuers of its K parity
        for (int i = 0; i < kNA; ++i) { mbar_init(a_full + i, kNumDq); mbar_init(a_empty + i, 2); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full + i, kNumMma);
            mbar_init(acc_empty + i, 4);
            mbar_init(b_full + i, 4);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 0) tc::tmem_alloc(tmem_slot, kTmemCols);
    if (warp == 0 && lane == 0) {
        tc::prefetch_map(&cmap0);
        tc::prefetch_map(&cmap1);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int n_pos0 = load_n_pos(L.prob[0]);
    const int n_pos1 = L.nprob > 1 ? load_n_pos(L.prob[1]) : 0;
    const int units0 = (n_pos0 / kGemvBlock) * L.prob[0].n_tiles;
    const int units1 = L.nprob > 1 ? (n_pos1 / kGemvBlock) * L.prob[1].n_tiles : 0;
    const int n_units = units0 + units1;
    const int u_lo = (int)((int64_t)blockIdx.x * n_units / gridDim.x);
    const int u_hi = (int)((int64_t)(blockIdx.x + 1) * n_units / gridDim.x);
    bool dead = false;

    if (warp < kNumMma) {
        // ------------------------------------------------------------ MMA issuers (+ TMA)
        // Issuer w owns accumulator (tile op = w & 1, K parity par = w >> 1): it issues the
        // MMAs of its tile for the unit's A buffers j = par, par + 2, ... (one per stage).
        // Issuer 0 also streams the codes: after the MMAs of stage g it refills the slot of
        // stage g - 1 (whose codes every dequantising warp has converted by then, since
        // they have converted the first half of stage g) with stage g - 1 + ns.
        if (lane == 0) {
            const int op = warp & 1, par = warp >> 1;
            const uint32_t idesc = tc::idesc_f16_f32(kTM, kTN);
            // producer cursor: next stage to load (global index it_p, unit up, stage sp)
            int it_p = 0, up = u_lo, sp = 0;
            auto produce = [&]() -> bool {
                if (up >= u_hi) return true;
                const Unit I = unit_at(L, units0, up);
                const GemvParams &p = L.prob[I.pi];
                const int slot = it_p % ns;
                if (!mbar_wait_timed(empty + slot, ((it_p / ns) & 1) ^ 1, abort_flag)) return false;
                const CUtensorMap *map = I.pi ? &cmap1 : &cmap0;
                unsigned char *st = smem + slot * kStageBytes;
                mbar_arrive_expect_tx(full + slot, kStageBytes);
                tc::tma_load_2d(st, map, sp * 128, I.e * p.R + tile_row<GATED>(p, I.rt, 0), full + slot);
                tc::tma_load_2d(st + kTM * 128, map, sp * 128, I.e * p.R + tile_row<GATED>(p, I.rt, 1), full + slot);
                ++it_p;
                if (++sp == p.K / kSK) { sp = 0; ++up; }
                return true;
            };
            if (warp == 0)
                for (int i = 0; i < ns && !dead; ++i) dead = !produce();
            int ia = 0, uc = 0, kb = -1, prev = -1;
            for (int u = u_lo; u < u_hi && !dead; ++u, ++uc) {
                const Unit I = unit_at(L, units0, u);
                const GemvParams &p = L.prob[I.pi];
                const int key = I.pi * (1 << 30) + I.blk;
                if (key != prev) {
                    ++kb;
                    prev = key;
                    if (!mbar_wait_timed(b_full + (kb & 1), (kb >> 1) & 1, abort_flag)) { dead = true; break; }
                }
                const int d = uc & 1;
                if (!mbar_wait_timed(acc_empty + d, ((uc >> 1) & 1) ^ 1, abort_flag)) { dead = true; break; }
                tc::fence_after_sync();
                const uint32_t dacc = tmem + kColD + 64u * d + 16u * (2 * op + par);
                const uint32_t bbase = smem_u32(smem + S.b_off + (kb & 1) * S.b_bytes);
                const int nsub = p.K / kSubK;  // even: K is a whole number of stages
                for (int j = par; j < nsub; j += 2) {
                    const int ib = ia + j, buf = ib % kNA;
                    if (!mbar_wait_timed(a_full + buf, (ib / kNA) & 1, abort_flag)) { dead = true; break; }
                    tc::fence_after_sync();
                    const uint32_t a0 = tmem + (uint32_t)buf * 128u + 64u * op;
#pragma unroll
                    for (int kk = 0; kk < kSubK / 16; ++kk) {
                        // K = 128 j + 16 kk: atom 2 j + kk / 4, 32 bytes per 16 elements inside it
                        const uint64_t bd =
                            tc::sw128_desc(bbase + (uint32_t)(2 * j + (kk >> 2)) * 1024u + (kk & 3) * 32u);
                        tc::mma_f16_ts(dacc, a0 + kk * 8u, bd, idesc, (j > par || kk > 0) ? 1u : 0u);
                    }
                    tc::commit(a_empty + buf);
                    if (warp == 0 && (ia + j) > 0 && !produce()) { dead = true; break; }
                }
                if (dead) break;
                ia += nsub;
                tc::commit(acc_full + d);
            }
            if (dead) { raise_status(L.prob[0].status, FT_ERR_TIMEOUT); *abort_flag = 1; }
            if (warp == 0) {
                for (int i = 0; i < ns && i < it_p; ++i) {  // let every issued copy land
                    const int last = it_p - 1 - i;
                    mbar_wait_timed(full + last % ns, (last / ns) & 1, nullptr);
                }
            }
        }
    } else if (warp >= kWarpDq0) {
        // ------------------------------------------------------------ dequantisation
        const int q = warp & 3, role = (warp - kWarpDq0) >> 2, op = role >> 1, half = role & 1;
        const int r = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        const uint32_t col0 = (uint32_t)(op * 64 + half * 32);
        // Scale cursor, two stages ahead of the stage being converted: unit pu, stage ps.
        int pu = u_lo, ps = 0, pnst = 0, pgroup = 16;
        const uint8_t *prow = nullptr;
        auto cursor_unit = [&]() {
            if (pu >= u_hi) return;
            const Unit I = unit_at(L, units0, pu);
            const GemvParams &p = L.prob[I.pi];
            int row = tile_row<GATED>(p, I.rt, op) + r;
            if (row > p.R - 1) row = p.R - 1;  // rows past the matrix: any valid row, never stored
            prow = p.scales + (size_t)I.e * p.e_scales + (size_t)row * (p.K / p.group);
            pnst = p.K / kSK;
            pgroup = p.group;
        };
        auto fetch = [&]() -> uint4 {
            uint4 v = make_uint4(0, 0, 0, 0);
            if (pu >= u_hi) return v;
            if (pgroup == 16) {
                v = __ldg(reinterpret_cast<const uint4 *>(prow + 16 * ps));
            } else {
                const uint2 w = __ldg(reinterpret_cast<const uint2 *>(prow + 8 * ps));
                v.x = w.x;
                v.y = w.y;
            }
            if (++ps == pnst) {
                ++pu;
                ps = 0;
                cursor_unit();
            }
            return v;
        };
        cursor_unit();
        uint4 sc0 = fetch(), sc1 = fetch();
        int it = 0, ia = 0;
        for (int u = u_lo; u < u_hi && !dead; ++u) {
            const Unit I = unit_at(L, units0, u);
            const GemvParams &p = L.prob[I.pi];
            const int nst = p.K / kSK;
            const bool g16 = p.group == 16;
            for (int s = 0; s < nst; ++s, ++it) {
                const uint4 sc = sc0;
                sc0 = sc1;
                sc1 = fetch();
                const int slot = it % ns;
                if (!warp_wait(full + slot, (it / ns) & 1, abort_flag)) { dead = true; break; }
                const unsigned char *rowp = smem + slot * kStageBytes + op * kTM * 128 + r * 128;
                const uint32_t sw[4] = {sc.x, sc.y, sc.z, sc.w};
#pragma unroll
                for (int ss = 0; ss < kSK / kSubK; ++ss, ++ia) {
                    const int c0 = 4 * ss + 2 * half;  // first of this warp's two 32-element chunks
                    const uint4 cw0 = *reinterpret_cast<const uint4 *>(rowp + ((c0 ^ (r & 7)) << 4));
                    const uint4 cw1 = *reinterpret_cast<const uint4 *>(rowp + (((c0 + 1) ^ (r & 7)) << 4));
                    uint32_t four;  // scale bytes of the four 16-element groups of the two chunks
                    if (g16) {
                        four = half ? sw[2 * ss + 1] : sw[2 * ss];  // word c0 / 2 (no dynamic index)
                    } else {
                        const uint32_t b2 = (sw[ss] >> (16 * half)) & 0xFFFFu;  // bytes c0, c0 + 1
                        four = (b2 & 0xFFu) * 0x0101u | ((b2 >> 8) * 0x0101u) << 16;
                    }
                    uint32_t sv[4];
                    e4m3x2_to_f16x2_bcast(four & 0xFFFFu, sv[0], sv[1]);
                    e4m3x2_to_f16x2_bcast(four >> 16, sv[2], sv[3]);
                    const uint32_t words[8] = {cw0.x, cw0.y, cw0.z, cw0.w, cw1.x, cw1.y, cw1.z, cw1.w};
                    uint32_t o[32];
#pragma unroll
                    for (int wv = 0; wv < 8; ++wv) {
                        uint32_t t[4];
                        dequant8_f16(words[wv], sv[wv >> 1], t);
                        o[4 * wv] = t[0]; o[4 * wv + 1] = t[1]; o[4 * wv + 2] = t[2]; o[4 * wv + 3] = t[3];
                    }
                    const int buf = ia % kNA;
                    if (!warp_wait(a_empty + buf, ((ia / kNA) & 1) ^ 1, abort_flag)) { dead = true; break; }
                    tc::st32(tmem + lane_base + (uint32_t)buf * 128u + col0, o);
                    tc::wait_st();
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(a_full + buf);
                }
                if (dead) break;
                // the stage's codes are all in registers and converted: release it
                __syncwarp();
                if (lane == 0) mbar_arrive(empty + slot);
            }
        }
        if (dead && lane == 0) { raise_status(L.prob[0].status, FT_ERR_TIMEOUT); *abort_flag = 1; }
    } else {
        // ------------------------------------------------------------ staging + epilogue
        const int ew = warp - kWarpEpi0;  // 0..3
        const int q = warp & 3;
        const int r = 32 * q + lane;
        const uint32_t lane_base = (uint32_t)(32 * q) << 16;
        // finite contents everywhere the MMAs may read (ignored columns included)
        {
            uint4 *b4 = reinterpret_cast<uint4 *>(smem + S.b_off);
            for (int i = threadIdx.x - 32 * kWarpEpi0; i < (int)(2 * S.b_bytes / 16); i += 128)
                b4[i] = make_uint4(0, 0, 0, 0);
        }
        epi_sync();
        int su = u_lo, kn = 0;  // staging cursor: first unit of the next block to stage; blocks staged
        // Stage the next block into buffer kn & 1 (row scales into table kn & 3): each warp
        // takes 2 rows and arrives on the buffer's barrier. A warp stages block kb + 2 once
        // it has seen the accumulators of block kb's last unit, so the MMAs reading the
        // buffer are done; the table of block kb + 2 is not the one other warps may still
        // read for block kb, and block kb + 4 cannot be staged before every warp staged its
        // rows of kb + 2, which it does after finishing block kb.
        auto stage_next = [&]() {
            if (su >= u_hi) return;
            const Unit I = unit_at(L, units0, su);
            const GemvParams &p = L.prob[I.pi];
            const int n_pos = I.pi ? n_pos1 : n_pos0;
            const int X = kn & 1;
            unsigned char *bb = smem + S.b_off + X * S.b_bytes;
            for (int rr = 0; rr < 2; ++rr) {
                const int r8 = 2 * ew + rr;
                const int src = source_row(p, I.blk * kGemvBlock + r8, n_pos, GATED);
                float sc = stage_row_sw128(src >= 0 ? p.act + (size_t)src * p.K : nullptr, p.K, bb, r8);
                int dst = -1;
                if (!GATED && src >= 0) {  // down: destination slot and routing weight of the position
                    const int pos = I.blk * kGemvBlock + r8;
                    if (p.sorted_slot) {
                        dst = __ldg(p.sorted_slot + pos);  // src >= 0: a real slot
                        if (p.route_w) sc *= __ldg(p.route_w + dst);
                    } else {
                        dst = pos;
                    }
                }
                if (lane == 0) {
                    inv_tbl[(kn & 3) * kGemvBlock + r8] = sc;
                    dst_tbl[(kn & 3) * kGemvBlock + r8] = dst;
                }
            }
            fence_proxy_async_smem();  // the tensor core reads the rows through the async proxy
            __syncwarp();
            if (lane == 0) mbar_arrive(b_full + X);
            ++kn;
            su += p.n_tiles - I.rt;
        };
        stage_next();
        stage_next();
        int uc = 0, kb = -1, prev = -1;
        for (int u = u_lo; u < u_hi && !dead; ++u, ++uc) {
            const Unit I = unit_at(L, units0, u);
            const GemvParams &p = L.prob[I.pi];
            const int n_pos = I.pi ? n_pos1 : n_pos0;
            const int key = I.pi * (1 << 30) + I.blk;
            if (key != prev) {
                ++kb;
                prev = key;
                // acquire the other warps' row scales of this block (the phase is complete
                // already: the MMAs waited for it)
                if (!warp_wait(b_full + (kb & 1), (kb >> 1) & 1, abort_flag)) { dead = true; break; }
            }
            const float *inv = inv_tbl + (kb & 3) * kGemvBlock;
            const int *dsts = dst_tbl + (kb & 3) * kGemvBlock;
            const int d = uc & 1;
            if (!warp_wait(acc_full + d, (uc >> 1) & 1, abort_flag)) { dead = true; break; }
            tc::fence_after_sync();
            // the 8 used columns of the four accumulators; each tile's two K-parity halves are
            // added in a fixed order
            uint32_t a0[8], a1[8], b0[8], b1[8];
            const uint32_t dbase = tmem + lane_base + kColD + 64u * d;
            tc::ld8(dbase, a0);
            tc::ld8(dbase + 16u, a1);
            tc::ld8(dbase + 32u, b0);
            tc::ld8(dbase + 48u, b1);
            tc::wait_ld();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(acc_empty + d);
            float va[8], vb[8];
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                va[j] = __uint_as_float(a0[j]) + __uint_as_float(a1[j]);
                vb[j] = __uint_as_float(b0[j]) + __uint_as_float(b1[j]);
            }
            const float *glob_e = p.glob + (size_t)I.e * p.e_glob;
            if (GATED) {
                const int i = I.rt * kTM + r;
                if (i < p.up_off) {
                    const float gg = __ldg(glob_e + i), gu = __ldg(glob_e + p.up_off + i);
#pragma unroll
                    for (int j = 0; j < kGemvBlock; ++j) {
                        const float s = inv[j];
                        const float gate = va[j] * s * gg;
                        const float up = vb[j] * s * gu;
                        __nv_bfloat16 hv = __float2bfloat16_rn(silu(gate) * up);
                        p.h_out[(size_t)(I.blk * kGemvBlock + j) * p.h_ld + i] = *reinterpret_cast<uint16_t *>(&hv);
                    }
                }
            } else {
#pragma unroll
                for (int opx = 0; opx < 2; ++opx) {
                    const int n0 = I.rt * 2 * kTM + opx * kTM;
                    if (n0 >= p.R) break;  // warp-uniform: the whole tile is past the matrix
                    const int n = n0 + r;
                    const float g = __ldg(glob_e + n);
#pragma unroll
                    for (int j = 0; j < kGemvBlock; ++j) {
                        const int dst = dsts[j];
                        if (dst < 0) continue;
                        p.y_out[(size_t)dst * p.R + n] = (opx ? vb[j] : va[j]) * g * inv[j];
                    }
                }
            }
            // the last unit of a block frees its staging buffer for the block after next
            if (u + 1 == u_hi || I.rt + 1 == p.n_tiles) stage_next();
        }
        if (dead && lane == 0) { raise_status(L.prob[0].status, FT_ERR_TIMEOUT); *abort_flag = 1; }
    }

    // wind down (the producer has let its copies land before reaching this barrier)
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 0) tc::tmem_dealloc(tmem, kTmemCols);
}

// ---------------------------------------------------------------- host side

// Every K (gate_up: H; down: I_l or I_sl) a whole number of 256-element stages.
bool tc_gemv_ok(int K, int group) { return K % kSK == 0 && K >= kSK && (group == 16 || group == 32); }

static int tg_stages(int kmax)
{
    int optin = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    for (int ns = kNSMax; ns >= 2; --ns)
        if (tg_smem(kmax, ns).total + 1024 <= (uint32_t)optin) return ns;
    return 0;
}

bool tc_gemv_fits(int kmax) { return tg_stages(kmax) >= 2; }

cudaError_t launch_tc_gemv(const FastLaunch &L, bool gated, int max_units, cudaStream_t s)
{
    CUtensorMap m[2];
    int kmax = 0;
    for (int i = 0; i < L.nprob; ++i) {
        const GemvParams &p = L.prob[i];
        if (!tc_gemv_ok(p.K, p.group)) return cudaErrorInvalidValue;
        const uint64_t rows = (uint64_t)p.num_experts * p.R;
        if (!make_tensor_map_2d(&m[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, p.codes, (uint64_t)p.K / 2, rows,
                                (uint64_t)p.K / 2, 128, kTM, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
        if (p.K > kmax) kmax = p.K;
    }
    if (L.nprob < 2) m[1] = m[0];
    const int ns = tg_stages(kmax);
    if (ns < 2) return cudaErrorInvalidValue;
    const size_t smem = tg_smem(kmax, ns).total + 1024;
    int grid = sm_count();
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    auto kern = gated ? tc_gemv_kernel<true> : tc_gemv_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    FT_LAUNCH(kern, dim3(grid), dim3(kThreadsTg), smem, s, m[0], m[1], L, ns, kmax);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
