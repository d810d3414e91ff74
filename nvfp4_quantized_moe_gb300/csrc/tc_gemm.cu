// Prefill-regime grouped GEMM for the NVFP4 (and fp8_block) experts on the 5th-generation
// tensor cores.
//
// A work unit is (block of NT = 128 expert-sorted positions, two tiles of 128 weight
// rows): for gate_up the gate rows [i0, i0+128) and the matching up rows I_l + i0 + ..,
// whose accumulators sit side by side in tensor memory so SwiGLU fuses into the
// epilogue; for down the rows [n0, n0+256) as two tiles. One launch covers the routed
// experts' units and then the shared expert's (each role looks up its unit's problem;
// K may differ between the two), strided over persistent CTAs. Warp roles:
//   warp 0      one thread issues every TMA: per stage of 128 K elements (two 64-element
//               sub-chunks, one barrier) the raw packed codes of both tiles (box 32 bytes x
//               128 rows; fp8_block 64 bytes with the 64-byte swizzle) and the block's
//               activations (f16 box 64 x 128, 128-byte swizzled, K-major), per sub-chunk -- gate_up reads them from the expert-sorted f16 copy of
//               x, down from the f16 copy of h; each activation row carries a power-of-two
//               scale (see rows_to_f16_kernel) that the epilogue multiplies back;
//   warps 1, 14 warp 1 allocates tensor memory; one thread of each issues tcgen05.mma
//               (kind::f16, A from tensor memory, B from shared memory, f16 x f16 -> fp32,
//               M = 128, N = 128, K = 16) for one of the two tiles (the issue cost is per
//               issuing thread) and commits to the barriers, which count both issuers;
//   warps 2..9  dequantise the raw codes to the exact f16 code*scale (each thread reads
//               its row's block scales from global memory, 16 bytes a group ahead) and
//               write them straight into tensor memory with tcgen05.st (warp (quarter,
//               half): TMEM lanes of its quarter, tile `half`) -- the A operand makes no
//               round trip through shared memory;
//   warps 10-13 the epilogue (and warps 15-18 as a second group taking the other half
//               of the 32-position chunks): read the accumulator with tcgen05.ld
//               (one TMEM lane = one weight row per thread), apply globals, row scales and
//               SwiGLU (h) or the routing weight (y, fp32: each warp transposes its 32 x 32
//               blocks through shared memory and stores 128 contiguous bytes per position with
//               16-byte stores). Tensor memory: the accumulator (256 columns) and
//               two A buffers of one stage each (256 columns); the accumulator is released once every
//               epilogue warp has loaded its last chunk. A stage of 128 K elements carries
//               the per-chunk synchronisation (two barrier waits per role, a tensor-memory
//               store wait, an arrive, two commits) over twice the work of one 64-element box.
// f16 operands instead of bf16: code*scale is exact in both; a bf16 activation row
// scaled by its power of two (maximum in [2^14, 2^15)) converts to f16 exactly except
// for elements below 2^-31 of the row maximum, which move by less than 2^-38 of it;
// and the f16 dequantisation needs fewer instructions.
// Every wait on an mbarrier is bounded (about two seconds): on expiry the CTA records
// FT_ERR_TIMEOUT, stops, lets its issued copies land, frees its tensor memory and
// returns.
#include <cuda.h>
#include <cuda_runtime.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"
#include "tcgen05.cuh"

namespace ftmoe {

namespace {

constexpr int NT = kTcBlock;  // positions per unit (MMA N)
constexpr int MT = 128;       // weight rows per tile (MMA M)
constexpr int KC = 64;        // K elements per sub-chunk (128 bytes of f16: one TMA box row)
constexpr int NSUB = 2;       // sub-chunks per stage: a stage covers KST = 128 K elements
constexpr int KST = KC * NSUB;
constexpr int NSMAX = 4;      // TMA stages (at most)
constexpr int NA = 2;         // dequantised A buffers (tensor memory), one stage each
// A buffer ab, sub-chunk j, tile t at columns kColA + 128 ab + 64 j + 32 t
constexpr uint32_t kColA = 2 * NT;
// Warps: 0 producer, 1 MMA (tile 0), 2..9 dequantise, 10..13 epilogue, 14 MMA (tile 1),
// 15..18 a second epilogue group: two warps per TMEM quadrant take alternate 32-position
// chunks of the accumulator, so it is read out (and released to the next unit's MMAs) in
// half the time.
__host__ __device__ constexpr int tc_epi_groups(bool gated) { return (void)gated, 2; }
__host__ __device__ constexpr int tc_threads(bool gated) { return (void)gated, 608; }
constexpr int kMmaWarp1 = 14;    // issuer of tile 1: the issue cost of a tcgen05.mma is per
                                 // issuing thread, so one issuer per tile doubles the rate
constexpr int kDq = 256;         // dequantising threads
constexpr int kEpWarp0 = 10;     // first epilogue warp (group 0: 10..13, group 1: 15..18)

__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag, uint64_t limit)
{
    return mbar_wait_timed(bar, parity, abort_flag, limit);
}

// The same, for a whole warp: every lane waits (and so acquires what the phase
// publishes); the result is the same on all lanes, so the warp leaves its loops together.
__device__ __forceinline__ bool warp_wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                              uint64_t limit)
{
    const bool ok = mbar_wait_timed(bar, parity, abort_flag, limit);
    return __all_sync(0xFFFFFFFFu, ok);
}

__device__ __forceinline__ void arrive(uint64_t *bar) { mbar_arrive(bar); }

struct TcSmem {
    uint32_t a_bytes, b_bytes, raw_bytes;
    uint32_t a_off, b_off, raw_off, tp_off, tbl_off, bar_off, total;
    int ns;
};

// Raw code bytes per weight row and 64-element K sub-chunk: 32 (NVFP4, two codes a byte)
// or 64 (fp8_block, one code a byte).
__host__ __device__ constexpr uint32_t raw_row_bytes(bool fp8) { return fp8 ? 64u : 32u; }

__host__ __device__ inline TcSmem tc_smem(int ns, bool fp8, bool gated)
{
    TcSmem s;
    s.a_bytes = 0;  // the dequantised A operand lives in tensor memory
    // a stage: per sub-chunk j, the B box (NT rows x 128 bytes) at b + j NT 128 and the raw
    // code boxes of the two tiles at raw + (2 j + t) MT RB
    s.b_bytes = (uint32_t)NSUB * NT * 128;
    s.raw_bytes = (uint32_t)NSUB * 2u * MT * raw_row_bytes(fp8);
    s.ns = ns;
    s.a_off = 0;
    s.b_off = s.a_off + NA * s.a_bytes;
    s.raw_off = s.b_off + ns * s.b_bytes;
    // down epilogue: a 32 x 32 fp32 transpose block per epilogue warp
    s.tp_off = s.raw_off + ns * s.raw_bytes;
    s.tbl_off = s.tp_off + (gated ? 0 : 4 * tc_epi_groups(false) * 32 * 32 * 4);
    s.bar_off = s.tbl_off + 2 * NT * 8;           // two position tables (unit parity): [NT] slots + [NT] factors
    s.total = s.bar_off + 512;
    return s;
}

}  // namespace

// FP8: fp8_block banks (one e4m3 code byte per weight, an fp32 scale_inv per 128 x 128
// block, no globals). The dequantising warps then convert codes exactly to f16 and
// multiply by f16(scale_inv * 2^-e_t), where 2^e_t is a power of two per 128-row tile
// chosen from the tile's largest scale_inv so that every product stays below 2^15; the
// epilogue multiplies 2^e_t back in place of the row global.
template <bool GATED, bool FP8>
__global__ void __launch_bounds__(tc_threads(GATED), 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap codes_map0, const __grid_constant__ CUtensorMap b_map0,
                   const __grid_constant__ CUtensorMap codes_map1, const __grid_constant__ CUtensorMap b_map1,
                   const __grid_constant__ TcLaunch TL, int ns)
{
    pdl_enter();
    const TcParams &p0 = TL.prob[0];  // what both problems share: group, format, status
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte aligned base by pointer arithmetic on the shared array itself, so that the
    // compiler keeps every access derived from it in the shared state space
    unsigned char *smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
    const TcSmem L = tc_smem(ns, FP8, GATED);
    constexpr int NG = tc_epi_groups(GATED);  // epilogue groups of 4 warps
    constexpr int RB = (int)raw_row_bytes(FP8);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *full = bars, *empty = bars + NSMAX, *a_full = bars + 2 * NSMAX, *a_empty = a_full + NA;
    uint64_t *acc_full = a_empty + NA, *acc_empty = acc_full + 2;  // one accumulator (index 0)
    uint64_t *tbl_bar = acc_empty + 2;  // epilogue: a unit's position table (written by group 0)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(tbl_bar + 2);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const uint64_t wl = TL.wait_ns ? TL.wait_ns : kWaitNs;  // limit of every barrier wait
    // columns [0, 256): the accumulator (two 128-column tiles); [256, 512): NA A buffers
    const uint32_t tmem_cols = 512;

    if (threadIdx.x == 0) {
        // a stage and an A buffer are released by both issuers' commits
        for (int i = 0; i < NSMAX; ++i) { mbar_init(full + i, 1); mbar_init(empty + i, 2); }
        // consumer barriers count warps: each warp arrives once, from lane 0 after __syncwarp
        for (int i = 0; i < NA; ++i) { mbar_init(a_full + i, kDq / 32); mbar_init(a_empty + i, 2); }
        for (int i = 0; i < 2; ++i) {
            mbar_init(acc_full + i, 2);
            mbar_init(acc_empty + i, 4 * NG);  // every epilogue warp, after its last TMEM read
            mbar_init(tbl_bar + i, 4 * NG);
        }
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, tmem_cols);
    if (warp == 0 && lane == 0) {
        tc::prefetch_map(&codes_map0);
        tc::prefetch_map(&b_map0);
        if (TL.nprob > 1) {
            tc::prefetch_map(&codes_map1);
            tc::prefetch_map(&b_map1);
        }
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    // units: problem 0's (blocks x row tiles), then problem 1's
    auto n_units_of = [&](const TcParams &q) {
        const int n_pos = q.n_pos_dev ? chk_count(*q.n_pos_dev, NT, padded_capacity(q.n_slots, q.num_experts, NT), q.status)
                                      : (q.n_pos_static + NT - 1) / NT * NT;
        return (n_pos / NT) * q.n_mtiles;
    };
    const int units0 = n_units_of(p0);
    const int n_units = units0 + (TL.nprob > 1 ? n_units_of(TL.prob[1]) : 0);
    // the problem of unit u and u's index within it
    auto prob_of = [&](int u, int &lu) -> const TcParams & {
        lu = u < units0 ? u : u - units0;
        return TL.prob[u < units0 ? 0 : 1];
    };
    const int tile_rows = GATED ? MT : 2 * MT;  // row stride of the unit index m
    // units are strided over the CTAs: at any moment the GPU works on consecutive units,
    // which share their block's B tiles in L2
    bool dead = false;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // (fault injection: with skip_producer set on the host, no copy is ever issued, so
        // every consumer's bounded wait runs out)
        if (lane == 0 && !TL.skip_producer) {
            int it = 0, slot = 0;  // chunks issued; stage slot = it % ns, with phase ph = (it / ns) & 1
            uint32_t ph = 0;
            for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x) {
                int lu;
                const TcParams &p = prob_of(u, lu);
                const CUtensorMap *codes_map = u < units0 ? &codes_map0 : &codes_map1;
                const CUtensorMap *b_map = u < units0 ? &b_map0 : &b_map1;
                const int b = lu / p.n_mtiles, m = lu - b * p.n_mtiles;
                const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + b) : 0, p.num_experts, p.status);
                const int row_a = e * p.R + m * tile_rows;
                const int row_b = GATED ? row_a + p.up_off : row_a + MT;
                const int nk = p.K / KST;
                for (int c = 0; c < nk; ++c, ++it) {
                    if (!wait_bar(empty + slot, ph ^ 1, abort_flag, wl)) { dead = true; break; }
                    unsigned char *raw = smem + L.raw_off + slot * L.raw_bytes;
                    unsigned char *bt = smem + L.b_off + slot * L.b_bytes;
                    mbar_arrive_expect_tx(full + slot, L.raw_bytes + L.b_bytes);
#pragma unroll
                    for (int j = 0; j < NSUB; ++j) {
                        const int kc = c * NSUB + j;  // 64-element sub-chunk index
                        tc::tma_load_2d(raw + (2 * j) * MT * RB, codes_map, kc * RB, row_a, full + slot);
                        tc::tma_load_2d(raw + (2 * j + 1) * MT * RB, codes_map, kc * RB, row_b, full + slot);
                        tc::tma_load_2d(bt + j * NT * 128, b_map, kc * KC, b * NT, full + slot);
                    }
                    if (++slot == ns) { slot = 0; ph ^= 1; }
                }
            }
            if (dead) { raise_status(p0.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
            // let every issued copy land before the CTA's shared memory can be released:
            // wait for the last issued phase of each stage (already complete unless a
            // consumer gave up)
            for (int i = 0; i < ns && i < it; ++i) {
                const int last = it - 1 - i;
                mbar_wait_timed(full + last % ns, (last / ns) & 1, nullptr, wl);
            }
        }
    } else if (warp == 1 || warp == kMmaWarp1) {
        // ------------------------------------------------------------ MMA issuers
        if (lane == 0) {
            const uint32_t tile = warp == 1 ? 0u : 1u;  // this issuer's tile and accumulator half
            const uint32_t idesc = tc::idesc_f16_f32(MT, NT);
            int ia = 0, uc = 0, slot = 0;  // stage slot and its phase advance incrementally
            uint32_t ph = 0;
            for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x, ++uc) {
                int lu;
                const int nk = prob_of(u, lu).K / KST;
                // one accumulator: the epilogue of the previous unit has read it out
                if (!wait_bar(acc_empty, (uc & 1) ^ 1, abort_flag, wl)) { dead = true; break; }
                tc::fence_after_sync();
                const uint32_t acc = tmem + tile * NT;
                for (int c = 0; c < nk; ++c, ++ia) {
                    const int ab = ia % NA;
                    if (!wait_bar(full + slot, ph, abort_flag, wl) ||
                        !wait_bar(a_full + ab, (ia / NA) & 1, abort_flag, wl)) {
                        dead = true;
                        break;
                    }
                    tc::fence_after_sync();
#pragma unroll
                    for (int j = 0; j < NSUB; ++j) {
                        // A in tensor memory, B from the sub-chunk's swizzled box
                        const uint32_t a0 = tmem + kColA + (uint32_t)ab * 128u + (uint32_t)j * 64u + tile * 32u;
                        const uint32_t b0 = smem_u32(smem + L.b_off + slot * L.b_bytes + j * NT * 128);
#pragma unroll
                        for (int kk = 0; kk < KC / 16; ++kk) {
                            const uint64_t bd = tc::sw128_desc(b0 + kk * 32);
                            tc::mma_f16_ts(acc, a0 + kk * 8u, bd, idesc, (c | j | kk) != 0);
                        }
                    }
                    tc::commit(empty + slot);
                    tc::commit(a_empty + ab);
                    if (++slot == ns) { slot = 0; ph ^= 1; }
                }
                if (dead) break;
                tc::commit(acc_full);
            }
            if (dead) { raise_status(p0.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
        }
    } else if (FP8 && warp < kEpWarp0) {
        // ------------------------------------------------------------ dequantisation (fp8_block)
        // warp (quarter, half): rows 32*quarter .. +32 of tile `half`; per sub-chunk each thread
        // converts the 64 code bytes of its row (read in the 64-byte swizzle of the TMA box:
        // 16-byte piece j of row r sits at j ^ ((r >> 1) & 3), so 8 consecutive rows hit 8
        // different bank quads) and writes 128 bytes of A.
        const int quarter = warp & 3, half = (warp - 2) >> 2;
        const int r = 32 * quarter + lane;
        int ia = 0, slot = 0;  // A buffers used; stage slot and its phase advance incrementally
        uint32_t ph = 0;
        for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x) {
            int lu;
            const TcParams &p = prob_of(u, lu);
            const int kbn = p.K / 128, nk = p.K / KST;
            const int b = lu / p.n_mtiles, m = lu - b * p.n_mtiles;
            const int e = chk_expert(p.block_expert ? __ldg(p.block_expert + b) : 0, p.num_experts, p.status);
            const int nb = GATED ? (half ? p.up_off / MT : 0) + m : 2 * m + half;  // the tile's scale block row
            const float *srow = p.sinv + (size_t)e * p.e_sinv + (size_t)nb * kbn;
            float smax = 0.f;
            for (int q = 0; q < kbn; ++q) smax = fmaxf(smax, __ldg(srow + q));
            const float down = pow2f(-row_scale_exp(448.f * smax));
            for (int c = 0; c < nk; ++c, ++ia) {
                const int ab = ia % NA;
                if (!warp_wait_bar(full + slot, ph, abort_flag, wl) ||
                    !warp_wait_bar(a_empty + ab, ((ia / NA) & 1) ^ 1, abort_flag, wl)) {
                    dead = true;
                    break;
                }
                // a stage is one 128 x 128 scale block along K
                const __half2 s2 = __float2half2_rn(__ldg(srow + c) * down);
                const uint32_t sv = *reinterpret_cast<const uint32_t *>(&s2);
#pragma unroll
                for (int jj = 0; jj < NSUB; ++jj) {
                    const unsigned char *rw = smem + L.raw_off + slot * L.raw_bytes + (2 * jj + half) * MT * RB + r * RB;
                    const int x = (r >> 1) & 3;
                    uint4 q[4];
#pragma unroll
                    for (int j = 0; j < 4; ++j) q[j] = *reinterpret_cast<const uint4 *>(rw + ((j ^ x) << 4));
                    const uint32_t words[16] = {q[0].x, q[0].y, q[0].z, q[0].w, q[1].x, q[1].y, q[1].z, q[1].w,
                                                q[2].x, q[2].y, q[2].z, q[2].w, q[3].x, q[3].y, q[3].z, q[3].w};
                    uint32_t o[32];  // the row's 64 f16 values, TMEM columns in K order
#pragma unroll
                    for (int w = 0; w < 8; ++w) {  // columns 4w .. 4w + 3 = code words 2w, 2w + 1
#pragma unroll
                        for (int h2 = 0; h2 < 2; ++h2) {
                            const uint32_t cw = words[2 * w + h2];
                            uint32_t lo, hi;
                            asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
                                : "=r"(lo) : "r"(cw));
                            asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
                                : "=r"(hi) : "r"(cw >> 16));
                            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[4 * w + 2 * h2]) : "r"(lo), "r"(sv));
                            asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(o[4 * w + 2 * h2 + 1]) : "r"(hi), "r"(sv));
                        }
                    }
                    tc::st32(tmem + ((uint32_t)(32 * quarter) << 16) + kColA + (uint32_t)ab * 128u + (uint32_t)jj * 64u +
                                 (uint32_t)half * 32u,
                             o);
                }
                // every thread's stores complete, then the warp releases the buffer once
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) arrive(a_full + ab);
                if (++slot == ns) { slot = 0; ph ^= 1; }
            }
        }
        if (dead && lane == 0) { raise_status(p0.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
    } else if (warp < kEpWarp0) {
        // ------------------------------------------------------------ dequantisation
        // warp (quarter, half): rows 32*quarter .. +32 of tile `half`.
        // Block scales come straight from global memory: each thread reads its own row's
        // 16- (or 8-) byte groups (one group covers cpl chunks), one group ahead, across units.
        const int quarter = warp & 3, half = (warp - 2) >> 2;
        const int r = 32 * quarter + lane;
        // Scale bytes per load: 16, or 8 when a problem's rows hold K/group = 8 (mod 16)
        // scales (16-byte loads would then cross rows and lose their alignment).
        const int sbytes = TL.scale_load_bytes;
        const int cpl = sbytes * p0.group / KC;  // K chunks covered by one scale load
        auto load_scales = [&](const uint8_t *ptr) -> uint4 {
            if (sbytes == 16) return __ldg(reinterpret_cast<const uint4 *>(ptr));
            const uint2 v = __ldg(reinterpret_cast<const uint2 *>(ptr));
            return make_uint4(v.x, v.y, 0u, 0u);
        };
        auto scale_row = [&](int uu) {
            int lu;
            const TcParams &q = prob_of(uu, lu);
            const int bb = lu / q.n_mtiles, mm = lu - bb * q.n_mtiles;
            const int ee = chk_expert(q.block_expert ? __ldg(q.block_expert + bb) : 0, q.num_experts, q.status);
            const int row = ee * q.R + mm * tile_rows + (half ? (GATED ? q.up_off : MT) : 0) + r;
            return q.scales + (size_t)row * (size_t)(q.K / q.group);
        };
        int ia = 0, slot = 0;  // A buffers used; stage slot and its phase advance incrementally
        uint32_t ph = 0;
        const uint8_t *srow = blockIdx.x < n_units ? scale_row(blockIdx.x) : p0.scales;
        uint4 s_next = blockIdx.x < n_units ? load_scales(srow) : make_uint4(0, 0, 0, 0);
        for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x) {
            int lu;
            const int K = prob_of(u, lu).K;
            const int nk = K / KST, ngroups = (K / KC) / cpl;
            const int u_next = u + gridDim.x;
            const uint8_t *srow_next = u_next < n_units ? scale_row(u_next) : nullptr;
            uint4 s16 = make_uint4(0, 0, 0, 0);
            int ci = 0, q = 0;  // 64-element sub-chunk = q * cpl + ci
            for (int c = 0; c < nk; ++c, ++ia) {
                const int ab = ia % NA;
                if (!warp_wait_bar(full + slot, ph, abort_flag, wl) ||
                    !warp_wait_bar(a_empty + ab, ((ia / NA) & 1) ^ 1, abort_flag, wl)) {
                    dead = true;
                    break;
                }
#pragma unroll
                for (int jj = 0; jj < NSUB; ++jj) {
                    if (ci == 0) {
                        s16 = s_next;
                        if (q + 1 < ngroups) s_next = load_scales(srow + sbytes * (q + 1));
                        else if (srow_next) s_next = load_scales(srow_next);
                    }
                    uint32_t sw;
                    if (p0.group == 16) {
                        sw = ci == 0 ? s16.x : ci == 1 ? s16.y : ci == 2 ? s16.z : s16.w;
                    } else {
                        const int wi = ci >> 1;
                        const uint32_t wv = wi == 0 ? s16.x : wi == 1 ? s16.y : wi == 2 ? s16.z : s16.w;
                        const uint32_t two = (ci & 1) ? (wv >> 16) : (wv & 0xFFFFu);
                        sw = (two & 0xFFu) * 0x0101u | ((two >> 8) * 0x0101u) << 16;
                    }
                    uint32_t sv[4];
                    e4m3x2_to_f16x2_bcast(sw & 0xFFFFu, sv[0], sv[1]);
                    e4m3x2_to_f16x2_bcast(sw >> 16, sv[2], sv[3]);
                    // 32 code bytes of row r; the two 16-byte reads alternate order with row
                    // bit 2 so that 8 consecutive rows hit 8 different bank quads
                    const unsigned char *rw = smem + L.raw_off + slot * L.raw_bytes + (2 * jj + half) * MT * 32 + r * 32;
                    const int j0 = (r >> 2) & 1;
                    const uint4 qa = *reinterpret_cast<const uint4 *>(rw + 16 * j0);
                    const uint4 qb = *reinterpret_cast<const uint4 *>(rw + 16 * (j0 ^ 1));
                    const uint4 q0 = j0 ? qb : qa, q1 = j0 ? qa : qb;
                    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                    uint32_t o[32];  // the row's 64 f16 values, TMEM columns in K order
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        uint32_t t4[4];
                        dequant8_f16(words[w], sv[w >> 1], t4);
                        o[4 * w] = t4[0]; o[4 * w + 1] = t4[1]; o[4 * w + 2] = t4[2]; o[4 * w + 3] = t4[3];
                    }
                    // the row goes to this warp's TMEM lane quarter
                    tc::st32(tmem + ((uint32_t)(32 * quarter) << 16) + kColA + (uint32_t)ab * 128u + (uint32_t)jj * 64u +
                                 (uint32_t)half * 32u,
                             o);
                    if (++ci == cpl) { ci = 0; ++q; }
                }
                // every thread's stores complete, then the warp releases the buffer once
                tc::wait_st();
                tc::fence_before_sync();
                __syncwarp();
                if (lane == 0) arrive(a_full + ab);
                if (++slot == ns) { slot = 0; ph ^= 1; }
            }
            if (dead) break;
            srow = srow_next;
        }
        if (dead && lane == 0) { raise_status(p0.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
    } else {
        // ------------------------------------------------------------ epilogue
        // Thread = TMEM lane = tile row r (warp w may read lanes 32 (w % 4) ..); every
        // thread handles its row in both tiles of the accumulator, for the 32-position
        // chunks cb = eg, eg + NG, ... of its group eg.
        // Per unit the warps first build a table of the block's positions (slot and routing
        // weight x activation row scale, or the row scale alone) in shared memory, and load
        // their rows' globals, while the MMAs of the unit are still running.
        const int quarter = warp & 3;
        const int r = 32 * quarter + lane;
        const int eg = warp < kMmaWarp1 ? 0 : 1;               // epilogue group
        const int ew = warp - (eg ? kMmaWarp1 + 1 : kEpWarp0);  // warp within the group
        // One position table per unit, built by group 0 (lane = position, 32 per warp) and
        // double-buffered by unit parity: a warp writes table X for unit u only after
        // passing the table barrier of unit u - 1, which every epilogue warp reaches after
        // finishing unit u - 2, the last reader of table X.
        int uc = 0;  // units
        for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x, ++uc) {
            int lu;
            const TcParams &p = prob_of(u, lu);
            const int b = lu / p.n_mtiles, m = lu - b * p.n_mtiles;
            const int X = uc & 1;
            int *tbl_slot = reinterpret_cast<int *>(smem + L.tbl_off) + X * 2 * NT;
            float *tbl_w = reinterpret_cast<float *>(tbl_slot + NT);
            if (eg == 0) {
                const int t = 32 * ew + lane, pos = b * NT + t;
                float w = p.act_scale ? __ldg(p.act_scale + pos) : 1.f;
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
            const float *glob_e = p.glob + (size_t)e * p.R;
            const int row0 = GATED ? m * MT + r : m * 2 * MT + r;
            float g0, g1;
            if constexpr (FP8) {
                // 2^e_t of each tile, the inverse of the dequantising warps' factor
                const int kbn = p.K / 128;
                const int nb0 = GATED ? m : 2 * m, nb1 = GATED ? p.up_off / MT + m : 2 * m + 1;
                const float *s0 = p.sinv + (size_t)e * p.e_sinv + (size_t)nb0 * kbn;
                const float *s1 = p.sinv + (size_t)e * p.e_sinv + (size_t)nb1 * kbn;
                float m0 = 0.f, m1 = 0.f;
                for (int q = 0; q < kbn; ++q) {
                    m0 = fmaxf(m0, __ldg(s0 + q));
                    m1 = fmaxf(m1, __ldg(s1 + q));
                }
                g0 = pow2f(row_scale_exp(448.f * m0));
                g1 = pow2f(row_scale_exp(448.f * m1));
            } else {
                g0 = __ldg(glob_e + row0);
                g1 = __ldg(glob_e + (GATED ? p.up_off + row0 : row0 + MT));
            }
            __syncwarp();
            if (lane == 0) arrive(tbl_bar + X);
            if (!warp_wait_bar(tbl_bar + X, (uc >> 1) & 1, abort_flag, wl)) { dead = true; break; }
            if (!warp_wait_bar(acc_full, uc & 1, abort_flag, wl)) { dead = true; break; }
            tc::fence_after_sync();
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
            for (int cb = eg; cb < NT / 32; cb += NG) {
                uint32_t v0[32], v1[32];
                tc::ld32(lane_addr + cb * 32, v0);
                tc::ld32(lane_addr + NT + cb * 32, v1);
                tc::wait_ld();
                if (cb + NG >= NT / 32) {  // this warp's share read out: the next unit's MMAs may start
                    tc::fence_before_sync();
                    __syncwarp();
                    if (lane == 0) arrive(acc_empty);
                }
                if (GATED) {
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int t = cb * 32 + j;
                        const float w = tbl_w[t];
                        const float gate = __uint_as_float(v0[j]) * w * g0;
                        const float up = __uint_as_float(v1[j]) * w * g1;
                        __nv_bfloat16 hv = __float2bfloat16_rn(silu(gate) * up);
                        p.h_out[(size_t)(b * NT + t) * p.h_ld + row0] = *reinterpret_cast<uint16_t *>(&hv);
                    }
                } else {
                    // y rows in fp32 (no rounding of the slot partials before the ordered
                    // combine). The warp holds output columns [c0, c0 + 32) (its TMEM lanes) of 32
                    // positions; it transposes each tile's 32 x 32 block through its own 4 KB of
                    // shared memory so that 8 lanes store one position's 128 contiguous bytes with
                    // 16-byte stores (8 store instructions per block instead of 32).
                    float *tb = reinterpret_cast<float *>(smem + L.tp_off) + (size_t)(eg * 4 + ew) * 32 * 32;
                    const int jl = lane >> 3, ql = lane & 7;  // read-back: position jb + jl, columns 4 ql ..
#pragma unroll
                    for (int tile = 0; tile < 2; ++tile) {
                        const uint32_t *v = tile ? v1 : v0;
                        const float gr = tile ? g1 : g0;
                        __syncwarp();  // the previous block's read-back is done
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
    if (warp == 1) tc::tmem_dealloc(tmem, tmem_cols);
}

// out[pos] = f16(src[row(pos)] * 2^-e_pos), scale[pos] = 2^e_pos with e_pos chosen so that
// the row's largest magnitude lands in [2^14, 2^15); row(pos) = token of the position's
// slot (sorted_slot given) or pos itself; padding positions get zero rows and scale 0.
// One warp per position.
__global__ void rows_to_f16_kernel(const uint16_t *__restrict__ src, int K, const int *__restrict__ sorted_slot,
                                   const int *__restrict__ n_pos_dev, int n_pos_static, int n_slots, int top_k,
                                   uint16_t *__restrict__ out, float *__restrict__ scale, int cap, int *status)
{
    pdl_enter();
    const int n_pos = n_pos_dev ? chk_count(*n_pos_dev, 1, cap, status) : n_pos_static;
    const int lane = threadIdx.x & 31;
    const int warps = (gridDim.x * blockDim.x) >> 5;
    for (int pos = (blockIdx.x * blockDim.x + threadIdx.x) >> 5; pos < n_pos; pos += warps) {
        int row = pos;
        if (sorted_slot) {
            const int sl = chk_slot(__ldg(sorted_slot + pos), n_slots, status);
            row = sl < n_slots ? sl / top_k : -1;
        } else if (pos >= n_slots) {
            row = -1;
        }
        uint4 *o = reinterpret_cast<uint4 *>(out + (size_t)pos * K);
        if (row < 0) {
            for (int q = lane; q < K / 8; q += 32) o[q] = make_uint4(0, 0, 0, 0);
            if (lane == 0) scale[pos] = 0.f;
            continue;
        }
        const uint4 *s4 = reinterpret_cast<const uint4 *>(src + (size_t)row * K);
        float m = 0.f;
        for (int q = lane; q < K / 8; q += 32) {
            const uint4 v = __ldg(s4 + q);
            const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; ++i) m = fmaxf(m, fmaxf(fabsf(__uint_as_float(w[i] << 16)),
                                                           fabsf(__uint_as_float(w[i] & 0xFFFF0000u))));
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
            o[q] = make_uint4(h[0], h[1], h[2], h[3]);
        }
        if (lane == 0) scale[pos] = pow2f(e);
    }
}

// ---------------------------------------------------------------- host side

typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *, const cuuint64_t *,
                                  const cuuint64_t *, const cuuint32_t *, const cuuint32_t *, CUtensorMapInterleave,
                                  CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

static EncodeTiledFn encode_fn()
{
    static EncodeTiledFn fn = nullptr;
    if (!fn) {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<EncodeTiledFn>(ptr);
    }
    return fn;
}

bool make_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t rows,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, const_cast<void *>(base), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_shape_ok_fp8(int K, int rows_per_expert) { return K % 128 == 0 && K >= 128 && rows_per_expert % MT == 0; }

bool tc_shape_ok(int K, int group, int rows_per_expert)
{
    return K % KST == 0 && K >= KST && rows_per_expert % MT == 0 && (K / group) % 8 == 0 && K / group <= 256;
}

// Deepest TMA ring (NSMAX down to 2 stages) that fits the opt-in shared memory.
static int tc_stages(bool fp8, bool gated)
{
    int optin = 0, dev = 0;
    cudaGetDevice(&dev);
    cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev);
    for (int ns = NSMAX; ns >= 2; --ns)
        if (tc_smem(ns, fp8, gated).total + 1024 <= (uint32_t)optin) return ns;
    return 0;
}

cudaError_t launch_rows_to_f16(const uint16_t *src, int K, const int *sorted_slot, const int *n_pos_dev,
                               int n_pos_static, int n_slots, int top_k, int max_rows, uint16_t *out, float *scale,
                               cudaStream_t s, int *status)
{
    int blocks = (max_rows + 7) / 8;
    const int cap = sm_count() * 8;
    if (blocks > cap) blocks = cap;
    if (blocks < 1) blocks = 1;
    FT_LAUNCH(rows_to_f16_kernel, dim3(blocks), dim3(256), 0, s, src, K, sorted_slot, n_pos_dev, n_pos_static,
              n_slots, top_k, out, scale, max_rows, status);
    count_launches(1);
    return cudaGetLastError();
}

// Per problem: codes = the bank's packed codes (rows_total rows of K/2 bytes, or K bytes
// for fp8_block); act = the B operand rows (gate_up: the f16 expert-sorted copy of x or,
// for the shared expert, the f16 copy of x; down: the f16 copy of h), act_rows rows of K
// f16, read in blocks of 128 consecutive rows. The problems share group and format.
cudaError_t launch_tc_gemm(const TcParams *probs, const TcOperands *ops, int nprob, bool gated, int max_units,
                           cudaStream_t s)
{
    if (nprob < 1 || nprob > 2) return cudaErrorInvalidValue;
    if (nprob == 2 && (probs[1].group != probs[0].group || probs[1].fp8 != probs[0].fp8)) return cudaErrorInvalidValue;
    const bool fp8 = probs[0].fp8 != 0;
    const int ns = tc_stages(fp8, gated);
    if (!ns) return cudaErrorInvalidValue;
    CUtensorMap cmap[2], bmap[2];
    TcLaunch TL = {};
    TL.nprob = nprob;
    injected_stall(&TL.wait_ns, &TL.skip_producer);
    TL.scale_load_bytes = 16;
    for (int i = 0; i < nprob; ++i)
        if (!probs[i].fp8 && (probs[i].K / probs[i].group) % 16) TL.scale_load_bytes = 8;
    for (int i = 0; i < nprob; ++i) {
        const TcParams &p = probs[i];
        TL.prob[i] = p;
        // codes: NVFP4 rows of K/2 bytes in boxes of 32 bytes (no swizzle); fp8_block rows of
        // K bytes in boxes of 64 bytes with the 64-byte swizzle the dequantising warps undo
        const uint64_t row_bytes = fp8 ? (uint64_t)p.K : (uint64_t)p.K / 2;
        if (!make_tensor_map_2d(&cmap[i], CU_TENSOR_MAP_DATA_TYPE_UINT8, ops[i].codes, row_bytes,
                                (uint64_t)ops[i].rows_total, row_bytes, raw_row_bytes(fp8), MT,
                                fp8 ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_NONE) ||
            !make_tensor_map_2d(&bmap[i], CU_TENSOR_MAP_DATA_TYPE_FLOAT16, ops[i].act, (uint64_t)p.K,
                                (uint64_t)ops[i].act_rows, (uint64_t)p.K * 2, KC, NT, CU_TENSOR_MAP_SWIZZLE_128B))
            return cudaErrorInvalidValue;
    }
    if (nprob == 1) {  // (never read)
        cmap[1] = cmap[0];
        bmap[1] = bmap[0];
    }
    const size_t smem = tc_smem(ns, fp8, gated).total + 1024;
    int grid = sm_count();
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    auto kern = fp8 ? (gated ? tc_gemm_kernel<true, true> : tc_gemm_kernel<false, true>)
                    : (gated ? tc_gemm_kernel<true, false> : tc_gemm_kernel<false, false>);
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
    FT_LAUNCH(kern, dim3(grid), dim3(tc_threads(gated)), smem, s, cmap[0], bmap[0], cmap[1], bmap[1], TL, ns);
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
