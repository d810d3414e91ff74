// Prefill-regime grouped GEMM for the NVFP4 experts on the 5th-generation tensor cores.
//
// A work unit is (block of NT = 128 expert-sorted positions, tile of MT = 128 weight
// rows). Warp roles in a persistent CTA:
//   warp 0      TMA producer: per 64-element K chunk, the raw packed codes of the weight
//               tile(s) (box 32 bytes x 128 rows) and the block's activation rows
//               (bf16, 128-byte swizzled, K-major); per unit, the tile's block scales
//               (one contiguous bulk copy);
//   warp 1      allocates tensor memory and, from one thread, issues tcgen05.mma
//               (kind::f16, bf16 x bf16 -> fp32, M = 128, N = 128, K = 16 per
//               instruction) and commits to the stage barriers;
//   warps 2..5  dequantise the raw codes to the exact bf16 value code*scale, written in
//               the 128-byte swizzled K-major layout the MMA descriptors describe, and
//               after the last K chunk read the accumulators back with tcgen05.ld for
//               the epilogue: SwiGLU with the row globals for gate_up (gate and up
//               tiles accumulate side by side in tensor memory), routing weight and row
//               global for down.
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

constexpr int NT = kTcBlock;  // tokens (positions) per unit
constexpr int MT = 128;       // weight rows per tile
constexpr int KC = 64;        // K elements per chunk (128 bytes of bf16)
constexpr int NS = 4;         // TMA stages
constexpr int NA = 2;         // dequantised A buffers
constexpr int kThreadsTc = 192;
constexpr uint64_t kWaitNs = 2000000000ull;

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Bounded wait: false after about two seconds (or once another role gave up).
__device__ __forceinline__ bool wait_bar(uint64_t *bar, uint32_t parity, volatile int *abort_flag)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (uint32_t i = 1;; ++i) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((i & 255u) == 0) {
            if (*abort_flag) return false;
            if (globaltimer() - t0 > kWaitNs) return false;
        }
    }
}

struct TcSmem {
    uint32_t a_bytes, b_bytes, raw_bytes, scale_bytes;  // per buffer
    uint32_t a_off, b_off, raw_off, scale_off, bar_off, total;
};

__host__ __device__ inline TcSmem tc_smem(bool gated, int K, int group)
{
    TcSmem s;
    const int ntile = gated ? 2 : 1;
    s.a_bytes = (uint32_t)ntile * MT * 128;
    s.b_bytes = (uint32_t)NT * 128;
    s.raw_bytes = (uint32_t)ntile * MT * 32;
    s.scale_bytes = (uint32_t)MT * (K / group);
    s.a_off = 0;
    s.b_off = s.a_off + NA * s.a_bytes;
    s.raw_off = s.b_off + NS * s.b_bytes;
    s.scale_off = s.raw_off + NS * s.raw_bytes;
    s.bar_off = s.scale_off + (uint32_t)ntile * s.scale_bytes;
    s.total = s.bar_off + 256;
    return s;
}

}  // namespace

template <bool GATED>
__global__ void __launch_bounds__(kThreadsTc, 1)
    tc_gemm_kernel(const __grid_constant__ CUtensorMap codes_map, const __grid_constant__ CUtensorMap b_map,
                   const __grid_constant__ TcParams p)
{
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // 1024-byte alignment for the swizzled tiles
    unsigned char *smem = reinterpret_cast<unsigned char *>(
        (reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~static_cast<uintptr_t>(1023));
    const int K = p.K;
    const TcSmem L = tc_smem(GATED, K, p.group);
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + L.bar_off);
    uint64_t *full = bars, *empty = bars + NS, *a_full = bars + 2 * NS, *a_empty = bars + 2 * NS + NA;
    uint64_t *scale_full = bars + 2 * NS + 2 * NA, *scale_empty = scale_full + 1;
    uint64_t *acc_full = scale_full + 2, *acc_empty = scale_full + 3;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(scale_full + 4);
    volatile int *abort_flag = reinterpret_cast<volatile int *>(tmem_slot + 1);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int ntile = GATED ? 2 : 1;
    const uint32_t tmem_cols = GATED ? 2 * NT : NT;

    if (threadIdx.x == 0) {
        // full: the codes' TMA byte count (+ for gate_up, the producer's arrival once its
        // cp.async gather of the activation rows has landed)
        for (int i = 0; i < NS; ++i) { mbar_init(full + i, GATED ? 2 : 1); mbar_init(empty + i, 1); }
        for (int i = 0; i < NA; ++i) { mbar_init(a_full + i, 128); mbar_init(a_empty + i, 1); }
        mbar_init(scale_full, 1);
        mbar_init(scale_empty, 128);
        mbar_init(acc_full, 1);
        mbar_init(acc_empty, 128);
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tc::tmem_alloc(tmem_slot, tmem_cols);
    if (warp == 0 && lane == 0) {
        tc::prefetch_map(&codes_map);
        tc::prefetch_map(&b_map);
    }
    tc::fence_before_sync();
    __syncthreads();
    tc::fence_after_sync();
    const uint32_t tmem = *tmem_slot;

    const int n_pos = p.n_pos_dev ? *p.n_pos_dev : (p.n_pos_static + NT - 1) / NT * NT;
    const int n_units = (n_pos / NT) * p.n_mtiles;
    const int nk = K / KC;
    const uint32_t sbytes = (uint32_t)(MT * (K / p.group));
    bool dead = false;

    if (warp == 0) {
        // ------------------------------------------------------------ producer
        // gate_up gathers activation rows with cp.async (16 bytes per copy) straight into
        // the 128-byte swizzled K-major layout; it waits for its own copies LAG chunks
        // later, makes them visible to the tensor core (async proxy) and arrives.
        constexpr int LAG = 2;
        int it = 0, uc = 0;
        for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x, ++uc) {
            const int b = u / p.n_mtiles, m = u - b * p.n_mtiles;
            const int e = p.block_expert ? __ldg(p.block_expert + b) : 0;
            const int row_a = e * p.R + m * MT;
            const int row_b = row_a + p.up_off;  // gated: the matching up rows
            if (lane == 0) {
                if (!wait_bar(scale_empty, (uc & 1) ^ 1, abort_flag)) dead = true;
                if (!dead) {
                    mbar_arrive_expect_tx(scale_full, ntile * sbytes);
                    bulk_g2s(smem + L.scale_off, p.scales + (size_t)row_a * (K / p.group), sbytes, scale_full);
                    if (GATED)
                        bulk_g2s(smem + L.scale_off + L.scale_bytes, p.scales + (size_t)row_b * (K / p.group), sbytes,
                                 scale_full);
                }
            }
            dead = __shfl_sync(0xFFFFFFFFu, dead, 0);
            // lane l copies chunk l % 8 of rows l / 8 + 4 i (i = 0..31) of each K chunk
            const int jc = lane & 7;
            const uint16_t *src_row[NT / 4];
            if (GATED) {
#pragma unroll
                for (int i = 0; i < NT / 4; ++i) {
                    const int pos = b * NT + (lane >> 3) + 4 * i;
                    int r = 0;
                    if (p.sorted_slot) {
                        const int sl = __ldg(p.sorted_slot + pos);
                        r = sl < p.n_slots ? sl / p.top_k : 0;
                    } else {
                        r = pos < p.n_pos_static ? pos : 0;
                    }
                    src_row[i] = p.act + (size_t)r * K + jc * 8;
                }
            }
            for (int c = 0; c < nk && !dead; ++c, ++it) {
                const int slot = it % NS;
                if (lane == 0 && !wait_bar(empty + slot, ((it / NS) & 1) ^ 1, abort_flag)) dead = true;
                dead = __shfl_sync(0xFFFFFFFFu, dead, 0);
                if (dead) break;
                unsigned char *raw = smem + L.raw_off + slot * L.raw_bytes;
                unsigned char *bt = smem + L.b_off + slot * L.b_bytes;
                if (lane == 0) {
                    mbar_arrive_expect_tx(full + slot, ntile * MT * 32 + (GATED ? 0u : (uint32_t)NT * 128));
                    tc::tma_load_2d(raw, &codes_map, c * 32, row_a, full + slot);
                    if (GATED) tc::tma_load_2d(raw + MT * 32, &codes_map, c * 32, row_b, full + slot);
                    else tc::tma_load_2d(bt, &b_map, c * KC, b * NT, full + slot);
                }
                if (GATED) {
#pragma unroll
                    for (int i = 0; i < NT / 4; ++i) {
                        const int t = (lane >> 3) + 4 * i;
                        cp_async_16(bt + t * 128 + ((jc ^ (t & 7)) << 4), src_row[i] + c * KC);
                    }
                    cp_async_commit();
                    if (c >= LAG) {
                        cp_async_wait<LAG>();
                        fence_proxy_async_smem();
                        __syncwarp();
                        if (lane == 0)
                            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(full + (it - LAG) % NS))
                                         : "memory");
                    }
                }
            }
            if (GATED && !dead) {
                // this unit's last chunks: their gathers must land before the next unit
                // waits on the scale buffer, which needs this unit fully consumed
                cp_async_wait<0>();
                fence_proxy_async_smem();
                __syncwarp();
                if (lane == 0)
                    for (int j = it - (nk < LAG ? nk : LAG); j < it; ++j)
                        asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(full + j % NS))
                                     : "memory");
            }
        }
        if (dead && lane == 0) { raise_status(p.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
    } else if (warp == 1) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            const uint32_t idesc = tc::idesc_bf16_f32(MT, NT);
            int it = 0, ia = 0, uc = 0;
            for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x, ++uc) {
                if (!wait_bar(acc_empty, (uc & 1) ^ 1, abort_flag)) { dead = true; break; }
                tc::fence_after_sync();
                for (int c = 0; c < nk; ++c, ++it, ++ia) {
                    const int slot = it % NS, ab = ia % NA;
                    if (!wait_bar(full + slot, (it / NS) & 1, abort_flag) ||
                        !wait_bar(a_full + ab, (ia / NA) & 1, abort_flag)) {
                        dead = true;
                        break;
                    }
                    tc::fence_after_sync();
                    const uint32_t a0 = smem_u32(smem + L.a_off + ab * L.a_bytes);
                    const uint32_t b0 = smem_u32(smem + L.b_off + slot * L.b_bytes);
#pragma unroll
                    for (int kk = 0; kk < KC / 16; ++kk) {
                        const uint64_t bd = tc::sw128_desc(b0 + kk * 32);
                        tc::mma_bf16(tmem, tc::sw128_desc(a0 + kk * 32), bd, idesc, (c | kk) != 0);
                        if (GATED)
                            tc::mma_bf16(tmem + NT, tc::sw128_desc(a0 + MT * 128 + kk * 32), bd, idesc,
                                         (c | kk) != 0);
                    }
                    tc::commit(empty + slot);
                    tc::commit(a_empty + ab);
                }
                if (dead) break;
                tc::commit(acc_full);
            }
            if (dead) { raise_status(p.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
        }
    } else {
        // ------------------------------------------------------------ dequant + epilogue
        const int quarter = warp & 3;
        const int r = 32 * quarter + lane;  // weight row in the tile == TMEM lane
        int it = 0, ia = 0, uc = 0;
        for (int u = blockIdx.x; u < n_units && !dead; u += gridDim.x, ++uc) {
            const int b = u / p.n_mtiles, m = u - b * p.n_mtiles;
            if (!wait_bar(scale_full, uc & 1, abort_flag)) { dead = true; break; }
            const unsigned char *sc0 = smem + L.scale_off + r * (K / p.group);
            for (int c = 0; c < nk; ++c, ++it, ++ia) {
                const int slot = it % NS, ab = ia % NA;
                if (!wait_bar(full + slot, (it / NS) & 1, abort_flag) ||
                    !wait_bar(a_empty + ab, ((ia / NA) & 1) ^ 1, abort_flag)) {
                    dead = true;
                    break;
                }
                const unsigned char *raw = smem + L.raw_off + slot * L.raw_bytes;
                unsigned char *at = smem + L.a_off + ab * L.a_bytes;
#pragma unroll
                for (int t = 0; t < (GATED ? 2 : 1); ++t) {
                    const uint4 *rw = reinterpret_cast<const uint4 *>(raw + t * MT * 32 + r * 32);
                    const uint4 q0 = rw[0], q1 = rw[1];
                    const uint32_t words[8] = {q0.x, q0.y, q0.z, q0.w, q1.x, q1.y, q1.z, q1.w};
                    const unsigned char *sc = sc0 + t * L.scale_bytes;
                    uint32_t sv[4];
                    if (p.group == 16) {
                        const uint32_t s4 = *reinterpret_cast<const uint32_t *>(sc + c * 4);
                        e4m3x2_to_bf16x2_scaled(s4 & 0xFFFFu, sv[0], sv[1]);
                        e4m3x2_to_bf16x2_scaled(s4 >> 16, sv[2], sv[3]);
                    } else {
                        const uint32_t s2 = *reinterpret_cast<const uint16_t *>(sc + c * 2);
                        e4m3x2_to_bf16x2_scaled(s2, sv[0], sv[2]);
                        sv[1] = sv[0];
                        sv[3] = sv[2];
                    }
                    unsigned char *arow = at + t * MT * 128 + r * 128;
#pragma unroll
                    for (int w = 0; w < 8; ++w) {
                        uint32_t o[4];
                        dequant8(words[w], sv[w >> 1], o);
                        *reinterpret_cast<uint4 *>(arow + ((w ^ (r & 7)) << 4)) = make_uint4(o[0], o[1], o[2], o[3]);
                    }
                }
                fence_proxy_async_smem();
                asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(a_full + ab)) : "memory");
            }
            if (dead) break;
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(scale_empty)) : "memory");

            // epilogue
            if (!wait_bar(acc_full, uc & 1, abort_flag)) { dead = true; break; }
            tc::fence_after_sync();
            const int e = p.block_expert ? __ldg(p.block_expert + b) : 0;
            const float *glob_e = p.glob + (size_t)e * p.R;
            const uint32_t lane_addr = tmem + ((uint32_t)(32 * quarter) << 16);
            const int row = m * MT + r;
            if (GATED) {
                const float gg = __ldg(glob_e + row), gu = __ldg(glob_e + p.up_off + row);
                for (int cb = 0; cb < NT / 32; ++cb) {
                    uint32_t dg[32], du[32];
                    tc::ld32(lane_addr + cb * 32, dg);
                    tc::ld32(lane_addr + NT + cb * 32, du);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int pos = b * NT + cb * 32 + j;
                        const float gate = __uint_as_float(dg[j]) * gg, up = __uint_as_float(du[j]) * gu;
                        __nv_bfloat16 hv = __float2bfloat16_rn(silu(gate) * up);
                        p.h_out[(size_t)pos * p.h_ld + row] = *reinterpret_cast<uint16_t *>(&hv);
                    }
                }
            } else {
                const float dg = __ldg(glob_e + row);
                for (int cb = 0; cb < NT / 32; ++cb) {
                    uint32_t d[32];
                    tc::ld32(lane_addr + cb * 32, d);
                    tc::wait_ld();
#pragma unroll
                    for (int j = 0; j < 32; ++j) {
                        const int pos = b * NT + cb * 32 + j;
                        int dst;
                        float wgt = 1.f;
                        if (p.sorted_slot) {
                            dst = __ldg(p.sorted_slot + pos);
                            if (dst >= p.n_slots) continue;
                            if (p.route_w) wgt = __ldg(p.route_w + dst);
                        } else {
                            dst = pos;
                            if (dst >= p.n_pos_static) continue;
                        }
                        __nv_bfloat16 yv = __float2bfloat16_rn(__uint_as_float(d[j]) * dg * wgt);
                        p.y_out[(size_t)dst * p.y_ld + row] = *reinterpret_cast<uint16_t *>(&yv);
                    }
                }
            }
            tc::fence_before_sync();
            asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(acc_empty)) : "memory");
        }
        if (dead && lane == 0) { raise_status(p.status, FT_ERR_TIMEOUT); *abort_flag = 1; }
    }

    // wind down: every issued stage has landed or been consumed once all roles are here
    tc::fence_before_sync();
    __syncthreads();
    if (*abort_flag && threadIdx.x == 0) {
        // let copies still in flight land before the CTA's shared memory is released
        for (int i = 0; i < NS; ++i) {
            const uint64_t t0 = globaltimer();
            while (!mbar_try_wait(full + i, 0) && !mbar_try_wait(full + i, 1) && globaltimer() - t0 < kWaitNs) {
            }
        }
    }
    __syncthreads();
    tc::fence_after_sync();
    if (warp == 1) tc::tmem_dealloc(tmem, tmem_cols);
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

static bool make_map(CUtensorMap *map, CUtensorMapDataType dt, void *base, uint64_t inner, uint64_t rows,
                     uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz)
{
    EncodeTiledFn fn = encode_fn();
    if (!fn) return false;
    const cuuint64_t dims[2] = {inner, rows};
    const cuuint64_t strides[1] = {row_bytes};
    const cuuint32_t box[2] = {box_inner, box_rows};
    const cuuint32_t estr[2] = {1, 1};
    return fn(map, dt, 2, base, dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
              CU_TENSOR_MAP_L2_PROMOTION_L2_128B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

bool tc_shape_ok(int K, int group, int rows_per_expert) { return K % KC == 0 && K >= KC && rows_per_expert % MT == 0 && (K / group) % 4 == 0; }

size_t tc_smem_bytes(bool gated, int K, int group) { return tc_smem(gated, K, group).total + 1024; }

// codes: raw code bank (rows_total x K/2 bytes); act: gate_up -> x [T, K] bf16 (rows
// gathered per position), down -> h [act_rows, K] bf16 (consecutive positions).
cudaError_t launch_tc_gemm(const TcParams &p, bool gated, const void *codes, int64_t rows_total, const void *act,
                           int64_t act_rows, int max_units, cudaStream_t s)
{
    CUtensorMap cmap, bmap;
    if (!make_map(&cmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, const_cast<void *>(codes), (uint64_t)p.K / 2,
                  (uint64_t)rows_total, (uint64_t)p.K / 2, 32, MT, CU_TENSOR_MAP_SWIZZLE_NONE))
        return cudaErrorInvalidValue;
    if (!make_map(&bmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, const_cast<void *>(act), (uint64_t)p.K,
                  (uint64_t)act_rows, (uint64_t)p.K * 2, KC, gated ? 1 : NT, CU_TENSOR_MAP_SWIZZLE_128B))
        return cudaErrorInvalidValue;
    const size_t smem = tc_smem_bytes(gated, p.K, p.group);
    int grid = sm_count();
    if (max_units < grid) grid = max_units;
    if (grid < 1) grid = 1;
    cudaError_t e;
    if (gated) {
        e = cudaFuncSetAttribute(tc_gemm_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        tc_gemm_kernel<true><<<grid, kThreadsTc, smem, s>>>(cmap, bmap, p);
    } else {
        e = cudaFuncSetAttribute(tc_gemm_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        tc_gemm_kernel<false><<<grid, kThreadsTc, smem, s>>>(cmap, bmap, p);
    }
    count_launches(1);
    return cudaGetLastError();
}

}  // namespace ftmoe
