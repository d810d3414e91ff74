// W4A4 grouped GEMM on the block-scaled FP4 tensor cores: the native NVFP4 variant that
// the pages' sm_86/sm_89 cards could not run ("[TP=2] Quantized MoE expert parallelism ...
// NVFP4 port", section 2: without FP4 tensor cores NVFP4 ran there as W4A16).
//
// Both operands stay e2m1 codes: A = the expert's packed weight codes (M = 128 rows per tile),
// B = the NVFP4-quantized activation rows of a block of 128 expert-sorted positions (N), K in
// 256-element stages (one 128-byte swizzled TMA box per row), four tcgen05.mma
// kind::mxf4nvf4 block_scale scale_vec::4X (K = 64) per stage and tile, fp32 accumulators in
// tensor memory. The e4m3 block scales of both operands are the MMA's scale factors (ue4m3,
// one per 16 elements; a 32-element weight scale serves both of its 16-element halves); the
// per-row weight global and the per-position activation row scale multiply the fp32 sum in
// the epilogue. Scale-factor layout in tensor memory (measured on sm_103a): A's scale of row
// m sits in lane m, column sfa + m / 32; B's scale of column n in lane 32 q + n % 32 of every
// lane quadrant q, column sfb + n / 32; the byte is the 16-element block of the K step.
//
// Warp roles (15 warps):
//   0       TMA producer: per stage the two weight tiles' code boxes and the activation
//           codes box (each 128 bytes x 128 rows, 128-byte swizzle);
//   1, 10   MMA issuers, one per weight tile (gate / up rows, or the two down row tiles);
//   2..5    scale writers: per stage each thread (one TMEM lane) stores its weight rows'
//           scale words and the block positions' scale words into a tensor-memory ring;
//   6..9    epilogue group 0, 11..14 epilogue group 1 (alternate 32-position chunks): read
//           the accumulator, apply the row globals and the positions' row scales, then
//           SwiGLU (h, fp32) or the routing weight (y, fp32), each warp transposing 32 x 32
//           blocks through shared memory for 16-byte stores.
// Every barrier wait is bounded (the same limit and fault injection as the W4A16 kernel).
#include <cuda.h>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "tcgen05.cuh"

namespace ftmoe {

namespace {

constexpr int NT = 128;         // positions per unit (MMA N)
constexpr int MT = 128;         // weight rows per tile (MMA M)
constexpr int KS4 = 256;        // K elements per stage (128 code bytes per row)
constexpr int NS4 = 3;          // TMA stages
constexpr int NSF = 4;          // scale-factor slots in tensor memory
constexpr uint32_t kBox = 128u * 128u;     // one code box: 128 rows x 128 bytes
constexpr uint32_t kSfSlotCols = 48;       // per slot: A tile 0 (16 columns), A tile 1 (16), B (16)
constexpr uint32_t kSfCol0 = 2 * NT;       // first scale-factor column (after the accumulator)
constexpr int kThreads4 = 480;
constexpr int kIssuer1 = 10;
constexpr int kEpi0 = 6, kEpi1 = 11;

struct W4Smem {
    uint32_t stage_off, tp_off, tbl_off, bar_off, total;
};

__host__ __device__ inline W4Smem w4_smem()
{
    W4Smem s;
    s.stage_off = 0;                                   // NS4 x (A0, A1, B) boxes, 1024-aligned
    s.tp_off = s.stage_off + NS4 * 3 * kBox;           // 8 epilogue warps x 32 x 32 fp32
    s.tbl_off = s.tp_off + 8 * 32 * 32 * 4;            // two position tables: [NT] slots + [NT] factors
    s.bar_off = s.tbl_off + 2 * NT * 8;
    s.total = s.bar_off + 512;
    return s;
}

// Instruction descriptor of kind::mxf4nvf4 with ue4m3 scales: A and B e2m1 (format 1 at
// bits 7 and 10), both K-major, N / 8 at bit 17, M / 16 at bit 24, scale type 0 (ue4m3) at
// bit 23, scale data ids 0.
constexpr uint32_t idesc_mxf4nvf4(int M, int N)
{
    return (1u << 7) | (1u << 10) | ((uint32_t)(N >> 3) << 17) | ((uint32_t)(M >> 4) << 24);
}

// D[tmem] (+)= A[smem] x B[smem]^T with per-16-element ue4m3 scales of A (sfa) and B (sfb)
// in tensor memory, issued by one thread.
__device__ __forceinline__ void mma_mxf4nvf4(uint32_t d, uint64_t a_desc, uint64_t b_desc, uint32_t idesc,
                                             uint32_t sfa, uint32_t sfb, uint32_t accumulate)
{
    asm volatile(
        "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(d),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void st1(uint32_t taddr, uint32_t v)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}

__device__ __forceinline__ void st4(uint32_t taddr, uint32_t a, uint32_t b, uint32_t c, uint32_t d)
{
    asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(a), "r"(b),
                 "r"(c), "r"(d)
                 : "memory");
}

// 16 scale bytes of a weight row for one stage: group 16 reads them, group 32 reads 8 and
// gives each to both 16-element halves of its block.
__device__ __forceinline__ uint4 weight_scales(const uint8_t *p, int group)
{
    if (group == 16) return __ldg(reinterpret_cast<const uint4 *>(p));
    const uint2 v = __ldg(reinterpret_cast<const uint2 *>(p));
    auto dup = [](uint32_t w) -> uint2 {
        const uint32_t lo = __byte_perm(w, 0, 0x1100), hi = __byte_perm(w, 0, 0x3322);
        return make_uint2(lo, hi);
    };
    const uint2 a = dup(v.x), b = dup(v.y);
    return make_uint4(a.x, a.y, b.x, b.y);
}

// Bounded wait by a whole warp (every lane acquires what the phase publishes); the result is
// the same on all lanes.
__device__ __forceinline__ bool warp_all_wait(uint64_t *bar, uint32_t parity, volatile int *abort_flag, uint64_t limit)
{
    const bool ok = mbar_wait_timed(bar, parity, abort_flag, limit);
    return __all_sync(0xFFFFFFFFu, ok);
}

__device__ __forceinline__ uint32_t word_of(const uint4 &v, int i)
{
    return i == 0 ? v.x : i == 1 ? v.y : i == 2 ? v.z : v.w;
}

}  // namespace

template <bool GATED>
__global__ void __launch_bounds__(kThreads4, 1)
    tc_w4a4_kernel(const __grid_constant__ CUtensorMap wmap0, const __grid_constant__ CUtensorMap amap0,
                   const __grid_constant__ CUtensorMap wmap1, const __grid_constant__ CUtensorMap amap1,
                   const __grid_constant__ W4Launch WL)
{
    pdl_enter();
    const W4Params &p0 = WL.prob[0];
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const W4Smem L = w4_smem();
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *full = bars, *empty = bars + NS4, *sf_full = bars + 2 * NS4, *sf_empty = sf_full + NSF;
    uint64_t *acc_full = sf_empty + NSF, *acc_empty = acc_full + 1, *tbl_bar = acc_empty + 1;  // tbl_bar[2]
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tbl_bar + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t wl = WL.wait_ns ? WL.wait_ns : kWaitNs;
    if (threadIdx.x == 0) {
        for (int i = 0; i < NS4; ++i) { mbar_init(full + i, 1); mbar_init(empty + i, 2); }
        for (int i = 0; i < NSF; ++i) { mbar_init(sf_full + i, 4); mbar_init(sf_empty + i, 2); }
        mbar_init(acc_full, 2);
        mbar_init(acc_empty, 8);  // every epilogue warp, after its last TMEM read
        for (int i = 0; i < 2; ++i) mbar_init(tbl_bar + i, 8);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, 512);
    if (warp == 0 && lane == 0) {
        tc::prefetch_map(&wmap0);
        tc::prefetch_map(&amap0);
        if (WL.nprob > 1) {
            tc::prefetch_map(&wmap1);
            tc::prefetch_map(&amap1);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    auto n_units_of = [&](const W4Params &q) {
        const int n_pos = q.n_pos_dev ? chk_count(*q.n_pos_dev, NT, padded_capacity(q.n_slots, q.num_experts, NT), q.status)
                                      : (q.n_pos_static + NT - 1) / NT * NT;
        return (n_pos / NT) * q.n_mtiles;
    };
    const int units0 = n_units_of(p0);
    const int n_units = units0 + (WL.nprob > 1 ? n_units_of(WL.prob[1]) : 0);
    auto prob_of = [&](int u, int &lu) -> const W4Params & {
        lu = u < units0 ? u : u - units0;
        return WL.prob[u < units0 ? 0 : 1];
    };
    const int tile_rows = GATED ? MT : 2 * MT;  // row stride of the unit index m
    bool dead = false;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        if (lane == 0 && !WL.skip_producer) {
            int it = 0;
            for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x) {
                int lu;
                const W4Params &p = prob_of(u, lu);
                const CUtensorMap *wmap = u < units0 ? &wmap0 : &wmap1;
                const CUtensorMap *amap = u < units0 ? &amap0 : &amap1;
                const int b = lu / p.n_mtiles, m = lu - b * p.n_mtiles;
                const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + b) : 0, p.num_experts, p.status);
                const int row_a = e * p.R + m * tile_rows;
                const int row_b = GATED ? row_a + p.up_off : row_a + MT;
                for (int c = 0; c < p.K / KS4; ++c, ++it) {
                    const int slot = it % NS4;
                    if (!mbar_wait_timed(empty + slot, ((it / NS4) & 1) ^ 1, abort_flag, wl)) { dead = true; break; }
                    unsigned char *st = smem + L.stage_off + slot * 3 * kBox;
                    mbar_arrive_expect_tx(full + slot, 3 * kBox);
                    tc::tma_load_2d(st, wmap, c * 128, row_a, full + slot);
                    tc::tma_load_2d(st + kBox, wmap, c * 128, row_b, full + slot);
                    tc::tma_load_2d(st + 2 * kBox, amap, c * 128, b * NT, full + slot);
                }
            }
            if (dead) { raise_status(p0.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
            for (int i = 0; i < NS4 && i < it; ++i) {  // every issued copy lands before the exit
                const int last = it - 1 - i;
                mbar_wait_timed(full + last % NS4, (last / NS4) & 1, nullptr, wl);
            }
        }
    } else if (warp == 1 || warp == kIssuer1) {
        // ------------------------------------------------------------ MMA issuers
        if (lane == 0) {
            const uint32_t tile = warp == 1 ? 0u : 1u;
            const uint32_t idesc = idesc_mxf4nvf4(MT, NT);
            int it = 0, uc = 0;
            for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x, ++uc) {
                int lu;
                const int nk = prob_of(u, lu).K / KS4;
                if (!mbar_wait_timed(acc_empty, (uc & 1) ^ 1, abort_flag, wl)) { dead = true; break; }
                tc::fence_after_sync();
                const uint32_t acc = tmem + tile * NT;
                for (int c = 0; c < nk; ++c, ++it) {
                    const int slot = it % NS4, ss = it % NSF;
                    if (!mbar_wait_timed(full + slot, (it / NS4) & 1, abort_flag, wl) ||
                        !mbar_wait_timed(sf_full + ss, (it / NSF) & 1, abort_flag, wl)) {
                        dead = true;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t a0 = smem_u32(smem + L.stage_off + slot * 3 * kBox + tile * kBox);
                    const uint32_t b0 = smem_u32(smem + L.stage_off + slot * 3 * kBox + 2 * kBox);
                    const uint32_t sf = tmem + kSfCol0 + (uint32_t)ss * kSfSlotCols;
#pragma unroll
                    for (int s = 0; s < 4; ++s)
                        mma_mxf4nvf4(acc, tc::sw128_desc(a0 + 32 * s), tc::sw128_desc(b0 + 32 * s), idesc,
                                     sf + tile * 16u + 4u * s, sf + 32u + 4u * s, (c | s) != 0);
                    tc::commit(empty + slot);
                    tc::commit(sf_empty + ss);
                }
                if (dead) break;
                tc::commit(acc_full);
            }
            if (dead) { raise_status(p0.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
        }
    } else if (warp < kEpi0) {
        // ------------------------------------------------------------ scale writers
        // warp quadrant q (lanes 32 q .. 32 q + 31), thread j: weight rows 32 q + j of both tiles
        // (column 4 s + q of the tile's 16, lane 32 q + j) and block positions 32 c' + j for
        // c' = 0..3 (columns 4 s .. 4 s + 3 of B's 16, in this quadrant's lanes).
        const int q = warp & 3, r = 32 * q + lane;
        const uint32_t lane_base = tmem + ((uint32_t)(32 * q) << 16);
        // the scales of stage (u, c), loaded one stage ahead of their use (across units), so
        // that the load latency overlaps the previous stage's wait and stores
        struct StageScales {
            uint4 w0, w1, a[4];
        };
        auto load_stage = [&](int u, int c, StageScales &S) {
            int lu;
            const W4Params &p = prob_of(u, lu);
            const int b = lu / p.n_mtiles, m = lu - b * p.n_mtiles;
            const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + b) : 0, p.num_experts, p.status);
            const int wrow0 = e * p.R + m * tile_rows + r;
            const int wrow1 = GATED ? wrow0 + p.up_off : wrow0 + MT;
            const size_t wstride = (size_t)(p.K / p.group);
            const int wbytes = KS4 / p.group;  // weight scale bytes per stage and row
            S.w0 = weight_scales(p.w_scales + (size_t)wrow0 * wstride + c * wbytes, p.group);
            S.w1 = weight_scales(p.w_scales + (size_t)wrow1 * wstride + c * wbytes, p.group);
            const size_t astride = (size_t)(p.K / 16);
            const uint8_t *as = p.a_scales + (size_t)(b * NT + lane) * astride + 16 * c;
#pragma unroll
            for (int cc = 0; cc < 4; ++cc) S.a[cc] = __ldg(reinterpret_cast<const uint4 *>(as + (size_t)32 * cc * astride));
        };
        auto stages_of = [&](int u) {
            int lu;
            return prob_of(u, lu).K / KS4;
        };
        int u = blockIdx.x, c = 0, it = 0;
        StageScales cur, nxt;
        if (u < n_units) load_stage(u, 0, nxt);
        while (u < n_units && !dead) {
            cur = nxt;
            // the stage after (u, c)
            int un = u, cn = c + 1;
            if (cn == stages_of(u)) { un = u + gridDim.x; cn = 0; }
            if (un < n_units) load_stage(un, cn, nxt);
            const int ss = it % NSF;
            if (!warp_all_wait(sf_empty + ss, ((it / NSF) & 1) ^ 1, abort_flag, wl)) {
                dead = true;
                break;
            }
            tc::fence_after_sync();
            const uint32_t sf = lane_base + kSfCol0 + (uint32_t)ss * kSfSlotCols;
#pragma unroll
            for (int s4 = 0; s4 < 4; ++s4) {
                st1(sf + 4u * s4 + q, word_of(cur.w0, s4));
                st1(sf + 16u + 4u * s4 + q, word_of(cur.w1, s4));
                st4(sf + 32u + 4u * s4, word_of(cur.a[0], s4), word_of(cur.a[1], s4), word_of(cur.a[2], s4),
                    word_of(cur.a[3], s4));
            }
            tc::wait_st();
            tc::fence_before_sync();
            __syncwarp();
            if (lane == 0) mbar_arrive(sf_full + ss);
            u = un;
            c = cn;
            ++it;
        }
        if (dead && lane == 0) { raise_status(p0.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
    } else {
        // ------------------------------------------------------------ epilogue
        // thread = TMEM lane = weight row r of both tiles; group eg takes the 32-position
        // chunks eg, eg + 2; group 0 builds the unit's position table (slot and factor).
        const int quarter = warp & 3, r = 32 * quarter + lane;
        const int eg = warp < kIssuer1 ? 0 : 1;
        const int ew = warp - (eg ? kEpi1 : kEpi0);
        float *tb = reinterpret_cast<float *>(smem + L.tp_off) + (size_t)(eg * 4 + ew) * 32 * 32;
        const int jl = lane >> 3, ql = lane & 7;  // read-back: position jb + jl, columns 4 ql ..
        int uc = 0;
        for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x, ++uc) {
            int lu;
            const W4Params &p = prob_of(u, lu);
            const int b = lu / p.n_mtiles, m = lu - b * p.n_mtiles;
            const int X = uc & 1;
            int *tbl_slot = reinterpret_cast<int *>(smem + L.tbl_off) + X * 2 * NT;
            float *tbl_w = reinterpret_cast<float *>(tbl_slot + NT);
            if (eg == 0) {
                const int t = 32 * ew + lane, pos = b * NT + t;
                float w = __ldg(p.a_glob + pos);
                int dst = pos;
                if (!GATED) {
                    if (p.sorted_slot) {
                        dst = chk_slot(__ldg(p.sorted_slot + pos), p.n_slots, p.status);
                        if (dst >= p.n_slots) dst = -1;
                        else if (p.route_w) w *= __ldg(p.route_w + dst);
                    } else if (dst >= p.n_pos_static) {
                        dst = -1;
                    }
                }
                tbl_slot[t] = dst;
                tbl_w[t] = w;
            }
            const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + b) : 0, p.num_experts, p.status);
            const float *glob_e = p.w_glob + (size_t)e * p.R;
            const int row0 = GATED ? m * MT + r : m * 2 * MT + r;
            const float g0 = __ldg(glob_e + row0);
            const float g1 = __ldg(glob_e + (GATED ? p.up_off + row0 : row0 + MT));
            __syncwarp();
            if (lane == 0) mbar_arrive(tbl_bar + X);
            if (!warp_all_wait(tbl_bar + X, (uc >> 1) & 1, abort_flag, wl)) { dead = true; break; }
            if (!warp_all_wait(acc_full, uc & 1, abort_flag, wl)) { dead = true; break; }
            tc::fence_after_sync();
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
            for (int cb = eg; cb < NT / 32; cb += 2) {
                uint32_t v0[32], v1[32];
                tc::ld32(lane_addr + cb * 32, v0);
                tc::ld32(lane_addr + NT + cb * 32, v1);
                tc::wait_ld();
                if (cb + 2 >= NT / 32) {  // this warp's share read out: the next unit's MMAs may start
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) mbar_arrive(acc_empty);
                }
                if (GATED) {
                    // h = silu(gate) * up in fp32, one 32 x 32 (positions x h columns) block per warp
                    __syncwarp();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const float f = tbl_w[cb * 32 + j];
                        const float gate = __uint_as_float(v0[j]) * g0 * f;
                        const float up = __uint_as_float(v1[j]) * g1 * f;
                        tb[j * 32 + lane] = silu(gate) * up;
                    }
                    __syncwarp();
                    const int c0 = m * MT + 32 * quarter + 4 * ql;
#pragma unroll
                    for (int jb = 0; jb < 32; jb += 4) {
                        const int pos = b * NT + cb * 32 + jb + jl;
                        const float4 o = *reinterpret_cast<const float4 *>(tb + (jb + jl) * 32 + 4 * ql);
                        __stcg(reinterpret_cast<float4 *>(p.h_out + (size_t)pos * p.h_ld + c0), o);
                    }
                } else {
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile) {
                        const uint32_t *v = tile ? v1 : v0;
                        const float gr = tile ? g1 : g0;
                        __syncwarp();
                        // the row global (this lane's column) before the transpose, the position's
                        // factor after it (one read per position instead of one per element)
#pragma unroll
                        for (int j = 0; j < 32; ++j) tb[j * 32 + lane] = __uint_as_float(v[j]) * gr;
                        __syncwarp();
                        const int c0 = m * 2 * MT + tile * MT + 32 * quarter + 4 * ql;
#pragma unroll
                        for (int jb = 0; jb < 32; jb += 4) {
                            const int dst = tbl_slot[cb * 32 + jb + jl];
                            const float w = tbl_w[cb * 32 + jb + jl];
                            float4 o = *reinterpret_cast<const float4 *>(tb + (jb + jl) * 32 + 4 * ql);
                            o.x *= w; o.y *= w; o.z *= w; o.w *= w;
                            if (dst >= 0) __stcg(reinterpret_cast<float4 *>(p.y_out + (size_t)dst * p.y_ld + c0), o);
                        }
                    }
                }
            }
        }
        if (dead && lane == 0) { raise_status(p0.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
    }

    // wind down (the producer has let its copies land before reaching this barrier)
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, 512);
}

bool w4a4_shape_ok(int K, int rows_per_expert)
{
    return K % KS4 == 0 && K >= KS4 && rows_per_expert % MT == 0;
}

// Per problem: the bank's packed codes (rows_total rows of K/2 bytes) and the quantized
// activation codes (act_rows rows of K/2 bytes, blocks of 128 consecutive rows).
cudaError_t launch_w4a4_gemm(const W4Params *probs, const W4Operands *ops, int nprob, bool gated, int max_units,
                             cudaStream_t s)
{
    if (nprob < 1 || nprob > 2) return cudaErrorInvalidValue;
    CUtensorMap wmap[2], amap[2];
    W4Launch WL = {};
    WL.nprob = nprob;
    injected_stall(&WL.wait_ns, &WL.skip_producer);
    for (int i = 0; i < nprob; ++i) {
        const W4Params &p = probs[i];
        if (!w4a4_shape_ok(p.K, p.R) || (p.group != 16 && p.group != 32)) return cudaErrorInvalidValue;
        WL.prob[i] = p;
        const uint64_t row_bytes = (uint64_t)p.K / 2;
        if (!make_tensor_map_2d(&wmap[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, ops[i].codes, row_bytes,
                                (uint64_t)ops[i].rows_total, row_bytes, 128, MT, CU_TENSOR_MAP_SWIZZLE_128B) ||
            !make_tensor_map_2d(&amap[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, ops[i].act_codes, row_bytes,
                                (uint64_t)ops[i].act_rows, row_bytes, 128, NT, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (nprob == 1) {  // (never read)
        wmap[1] = wmap[0];
        amap[1] = amap[0];
    }
    const size_t smem = w4_smem().total + 1024;
    int grid = sm_count();
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    auto kern = gated ? tc_w4a4_kernel<true> : tc_w4a4_kernel<false>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    FT_LAUNCH(kern, dim3(grid), dim3(kThreads4), smem, s, wmap[0], amap[0], wmap[1], amap[1], WL);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
