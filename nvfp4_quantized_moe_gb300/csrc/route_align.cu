// Router (softmax / top-k / renormalise) and moe_align (expert-sorted, tile-padded
// slot order) kernels.
//
// Routing follows norm_topk_prob with a replicated router ("Offloaded MoE ignores
// tensor parallelism", follow-up comment): every rank selects the same experts.
// moe_align is the sort/pad step the "feat(qwen3_5_moe): tensor-parallel weight
// sharding" Notes name for the MoE paths.
#include <cuda_runtime.h>
#include <float.h>
#include <math.h>

#include "ftmoe_device.cuh"
#include "ftmoe_internal.h"

namespace ftmoe {

// ---------------------------------------------------------------- router

// One warp per token. Lane l holds logits l, l+32, ...; k rounds of a warp-wide
// arg-max over the unselected experts (larger logit first, then the lower index).
// Softmax is monotone, so this selects exactly the top-k probabilities. The kept
// weights are exp(l_j - l_max) / sum over kept exp(l_i - l_max): the softmax
// normaliser cancels in the renormalisation.
template <int VPL>
__global__ void __launch_bounds__(256) route_kernel(const float *__restrict__ logits, int T, int E, int k,
                                                    int32_t *__restrict__ ids, float *__restrict__ w)
{
    pdl_enter();
    const int lane = threadIdx.x & 31;
    const int t = blockIdx.x * (blockDim.x >> 5) + (threadIdx.x >> 5);
    if (t >= T) return;
    const float *row = logits + (size_t)t * E;
    float v[VPL];
    uint32_t taken = 0;
#pragma unroll
    for (int i = 0; i < VPL; ++i) {
        int e = lane + 32 * i;
        v[i] = (e < E) ? __ldg(row + e) : 0.0f;
        if (e >= E) taken |= 1u << i;
    }
    float top = 0.0f, sum = 0.0f, my_w = 0.0f;
    int my_id = 0;
    for (int r = 0; r < k; ++r) {
        float bv = -INFINITY;
        int bi = 0x7FFFFFFF;
#pragma unroll
        for (int i = 0; i < VPL; ++i) {
            if (!((taken >> i) & 1u)) {
                int e = lane + 32 * i;
                if (bi == 0x7FFFFFFF || v[i] > bv) { bv = v[i]; bi = e; }  // ascending e: ties keep the lower
            }
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            float ov = __shfl_xor_sync(0xFFFFFFFFu, bv, off);
            int oi = __shfl_xor_sync(0xFFFFFFFFu, bi, off);
            bool better = (oi != 0x7FFFFFFF) && (bi == 0x7FFFFFFF || ov > bv || (ov == bv && oi < bi));
            if (better) { bv = ov; bi = oi; }
        }
        if ((bi & 31) == lane) taken |= 1u << (bi >> 5);
        if (r == 0) top = bv;
        float ex = expf(bv - top);
        sum += ex;
        if (lane == r) { my_id = bi; my_w = ex; }
    }
    if (lane < k) {
        ids[(size_t)t * k + lane] = my_id;
        w[(size_t)t * k + lane] = my_w / sum;
    }
}

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w, cudaStream_t s)
{
    const int warps = 8;
    dim3 grid((T + warps - 1) / warps), block(warps * 32);
    int vpl = (E + 31) / 32;
    if (vpl <= 1) FT_LAUNCH(route_kernel<1>, dim3(grid), dim3(block), 0, s, logits, T, E, k, ids, w);
    else if (vpl <= 2) FT_LAUNCH(route_kernel<2>, dim3(grid), dim3(block), 0, s, logits, T, E, k, ids, w);
    else if (vpl <= 4) FT_LAUNCH(route_kernel<4>, dim3(grid), dim3(block), 0, s, logits, T, E, k, ids, w);
    else if (vpl <= 8) FT_LAUNCH(route_kernel<8>, dim3(grid), dim3(block), 0, s, logits, T, E, k, ids, w);
    else if (vpl <= 16) FT_LAUNCH(route_kernel<16>, dim3(grid), dim3(block), 0, s, logits, T, E, k, ids, w);
    else FT_LAUNCH(route_kernel<32>, dim3(grid), dim3(block), 0, s, logits, T, E, k, ids, w);
    count_launches(1);
    return cudaGetLastError();
}

// ---------------------------------------------------------------- align

// Rank of each slot among the slots of the same expert inside a warp's contiguous
// range [lo, hi), in slot order; per-warp expert counts accumulate in cnt[E]. An id
// out of range is flagged and the slot skipped; an id repeated inside a token's row is
// flagged but still placed. The row's earlier slots inside the warp's 32-slot window
// are compared through shuffles, the rest (a row that began before the window) loaded.
__device__ __forceinline__ void warp_rank_range(const int32_t *ids, int lo, int hi, int k, int E, int *cnt,
                                                int *rank_out, int rank_base, int *status, int *e_out = nullptr)
{
    const int lane = threadIdx.x & 31;
    constexpr int kAhead = 8;  // windows of 32 slots whose ids are loaded together
    for (int s00 = lo; s00 < hi; s00 += 32 * kAhead) {
    int raws[kAhead];
#pragma unroll
    for (int i = 0; i < kAhead; ++i) {
        const int s = s00 + 32 * i + lane;
        raws[i] = (s < hi) ? __ldg(ids + s) : -1;
    }
#pragma unroll
    for (int i = 0; i < kAhead; ++i) {
        const int s0 = s00 + 32 * i;
        if (s0 >= hi) continue;  // (uniform over the warp)
        const int s = s0 + lane;
        const int raw = raws[i];
        int e = raw;
        if (s < hi && (raw < 0 || raw >= E)) {
            raise_status(status, FT_ERR_INVALID_ROUTING);
            e = -1;
        }
        const int base = s - s % k;  // first slot of the token's row
        bool dup = false;
        for (int d = 1; d < k && d < 32; ++d) {
            const int v = __shfl_up_sync(0xFFFFFFFFu, raw, d);
            if (e >= 0 && lane >= d && s - d >= base && v == e) dup = true;
        }
        if (e >= 0)
            for (int j = base; j < s0; ++j)
                if (__ldg(ids + j) == e) dup = true;
        if (dup) raise_status(status, FT_ERR_INVALID_ROUTING);
        uint32_t peers = __match_any_sync(0xFFFFFFFFu, e);
        int rank = __popc(peers & lanemask_lt());
        int leader = __ffs(peers) - 1;
        int before = (e >= 0) ? cnt[e] : 0;
        if (e >= 0) rank_out[s - rank_base] = before + rank;
        if (e_out && s < hi) e_out[s - rank_base] = e;  // the slot's expert, or -1
        __syncwarp();
        if (e >= 0 && lane == leader) cnt[e] = before + __popc(peers);
        __syncwarp();
    }
    }
}

// Exclusive scan of vals[0..n) in place (n <= blockDim.x <= 1024), returns the total.
__device__ int block_exclusive_scan(int *vals, int n, int *warp_tot)
{
    const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
    int v = (tid < n) ? vals[tid] : 0;
    int incl = v;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
        int o = __shfl_up_sync(0xFFFFFFFFu, incl, off);
        if (lane >= off) incl += o;
    }
    if (lane == 31) warp_tot[wid] = incl;
    __syncthreads();
    if (wid == 0) {
        int nw = (blockDim.x + 31) >> 5;
        int x = (lane < nw) ? warp_tot[lane] : 0;
        int xi = x;
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
            int o = __shfl_up_sync(0xFFFFFFFFu, xi, off);
            if (lane >= off) xi += o;
        }
        warp_tot[lane] = xi - x;  // exclusive warp offsets
        if (lane == 31) warp_tot[32] = xi;
    }
    __syncthreads();
    if (tid < n) vals[tid] = incl - v + warp_tot[wid];
    int total = warp_tot[32];
    __syncthreads();
    return total;
}

// Fill padding positions with the sentinel and give every block its expert: one thread per
// block for small blocks, one warp per block (its lanes filling the positions together) for
// blocks of 64 positions or more.
__device__ void fill_blocks(const int *off, const int *count, int E, int B, int n_slots, int total,
                            int32_t *sorted_slot, int32_t *block_expert)
{
    const bool per_warp = B >= 64;
    const int lane = per_warp ? (threadIdx.x & 31) : 0, step = per_warp ? 32 : 1;
    const int nworkers = per_warp ? (int)(blockDim.x >> 5) : (int)blockDim.x;
    for (int b = per_warp ? (int)(threadIdx.x >> 5) : (int)threadIdx.x; b < total / B; b += nworkers) {
        int pos = b * B;
        int lo = 0, hi = E;  // largest e with off[e] <= pos and a non-empty run
        while (hi - lo > 1) {
            int mid = (lo + hi) >> 1;
            if (off[mid] <= pos) lo = mid; else hi = mid;
        }
        while (lo + 1 < E && off[lo + 1] <= pos) ++lo;
        if (lane == 0) block_expert[b] = lo;
        int run_end_real = off[lo] + count[lo];
        for (int q = pos + lane; q < pos + B; q += step)
            if (q >= run_end_real) sorted_slot[q] = n_slots;
    }
}

// One CTA sorts up to kAlignFusedMax slots (shared memory permitting): 32 warps each rank a contiguous range,
// then per-expert prefixes over warps, padded offsets, placement.
__global__ void __launch_bounds__(1024) align_fused_kernel(const int32_t *__restrict__ ids, int n, int k, int E,
                                                           int B, int32_t *sorted_slot, int32_t *block_expert,
                                                           int32_t *expert_off, int32_t *n_padded, int *status,
                                                           int *zero, int zero_words)
{
    pdl_enter();
    // the forward's status word and split counts start at zero (cleared here instead
    // of by a separate memset); the __syncthreads below orders this before any error report
    for (int i = threadIdx.x; i < zero_words; i += blockDim.x) zero[i] = 0;
    extern __shared__ int smem[];
    int *cnt = smem;                    // [32][E]
    int *rank = cnt + 32 * E;           // [n]
    int *off = rank + n;                // [E+1]
    int *count = off + E + 1;           // [E]
    int *wt = count + E;                // [33]
    int *ex = wt + 33;                  // [n] expert of each slot (-1: out of range)
    const int tid = threadIdx.x, wid = tid >> 5;
    for (int i = tid; i < 32 * E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int per = (n + 31) / 32;
    int lo = min(n, wid * per), hi = min(n, lo + per);
    warp_rank_range(ids, lo, hi, k, E, cnt + wid * E, rank, 0, status, ex);
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 32; ++w) {
            int c = cnt[w * E + e];
            cnt[w * E + e] = run;
            run += c;
        }
        count[e] = run;
        off[e] = (run + B - 1) / B * B;
    }
    __syncthreads();
    int total = 0;
    // E may exceed blockDim only if E > 1024, which the host rejects.
    total = block_exclusive_scan(off, E, wt);
    if (tid == 0) off[E] = total;
    __syncthreads();
    for (int s = tid; s < n; s += blockDim.x) {
        const int e = ex[s];
        if (e < 0) continue;
        int w = s / per;
        sorted_slot[off[e] + cnt[w * E + e] + rank[s]] = s;
    }
    fill_blocks(off, count, E, B, n, total, sorted_slot, block_expert);
    for (int e = tid; e <= E; e += blockDim.x) expert_off[e] = off[e];
    if (tid == 0) *n_padded = total;
}

// Pass 1 of the large align: chunk c = slots [c*kAlignChunk, ...) handled by one
// CTA of 8 warps; ranks within the chunk and per-chunk expert counts.
__global__ void __launch_bounds__(256) align_count_kernel(const int32_t *__restrict__ ids, int n, int k, int E,
                                                          int *chunk_cnt, int *rank, int *status)
{
    pdl_enter();
    extern __shared__ int smem[];
    int *cnt = smem;  // [8][E]
    const int tid = threadIdx.x, wid = tid >> 5;
    for (int i = tid; i < 8 * E; i += blockDim.x) cnt[i] = 0;
    __syncthreads();
    const int c0 = blockIdx.x * kAlignChunk;
    const int per = kAlignChunk / 8;
    int lo = min(n, c0 + wid * per), hi = min(n, lo + per);
    warp_rank_range(ids, lo, hi, k, E, cnt + wid * E, rank, 0, status);
    __syncthreads();
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int w = 0; w < 8; ++w) {
            int c = cnt[w * E + e];
            cnt[w * E + e] = run;
            run += c;
        }
        chunk_cnt[(size_t)blockIdx.x * E + e] = run;
    }
    __syncthreads();
    for (int s = lo + (tid & 31); s < hi; s += 32) {
        int e = __ldg(ids + s);
        if (e >= 0 && e < E) rank[s] += cnt[wid * E + e];
    }
}

// Pass 2: per-expert prefix over chunks, padded offsets, sentinel/block fill.
__global__ void __launch_bounds__(1024) align_scan_kernel(int *chunk_cnt, int n_chunks, int E, int B, int n,
                                                          int32_t *sorted_slot, int32_t *block_expert,
                                                          int32_t *expert_off, int32_t *n_padded)
{
    pdl_enter();
    extern __shared__ int smem[];
    int *off = smem;          // [E+1]
    int *count = off + E + 1; // [E]
    int *wt = count + E;      // [33]
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int c0 = 0; c0 < n_chunks; c0 += 8) {  // 8 chunks' counts loaded together
            int v[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) v[i] = c0 + i < n_chunks ? chunk_cnt[(size_t)(c0 + i) * E + e] : 0;
#pragma unroll
            for (int i = 0; i < 8; ++i) {
                if (c0 + i < n_chunks) chunk_cnt[(size_t)(c0 + i) * E + e] = run;
                run += v[i];
            }
        }
        count[e] = run;
        off[e] = (run + B - 1) / B * B;
    }
    __syncthreads();
    int total = block_exclusive_scan(off, E, wt);
    if (tid == 0) off[E] = total;
    __syncthreads();
    fill_blocks(off, count, E, B, n, total, sorted_slot, block_expert);
    for (int e = tid; e <= E; e += blockDim.x) expert_off[e] = off[e];
    if (tid == 0) *n_padded = total;
}

// Pass 3: every slot to its place.
__global__ void align_place_kernel(const int32_t *__restrict__ ids, int n, int E, const int *chunk_base,
                                   const int *rank, const int32_t *expert_off, int32_t *sorted_slot)
{
    pdl_enter();
    int s = blockIdx.x * blockDim.x + threadIdx.x;
    if (s >= n) return;
    int e = __ldg(ids + s);
    if (e < 0 || e >= E) return;
    int c = s / kAlignChunk;
    sorted_slot[expert_off[e] + chunk_base[(size_t)c * E + e] + rank[s]] = s;
}

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Shared memory of the one-CTA align, and whether it fits the per-block opt-in limit.
static size_t align_fused_smem(int n, int E) { return sizeof(int) * ((size_t)32 * E + n + (E + 1) + E + 33 + n); }
static bool align_fused_ok(int n, int E) { return n <= kAlignFusedMax && align_fused_smem(n, E) <= 227 * 1024; }

size_t align_scratch_bytes(int n_slots, int E)
{
    if (align_fused_ok(n_slots, E)) return 0;
    size_t chunks = (size_t)(n_slots + kAlignChunk - 1) / kAlignChunk;
    return round_up(chunks * E * sizeof(int), 256) + round_up((size_t)n_slots * sizeof(int), 256);
}

cudaError_t launch_align(const int32_t *ids, int T, int k, int E, int B, int32_t *sorted_slot,
                         int32_t *block_expert, int32_t *expert_off, int32_t *n_padded, int *status,
                         void *scratch, cudaStream_t s, int *zero, size_t zero_bytes)
{
    const int n = T * k;
    if (align_fused_ok(n, E)) {
        const size_t smem = align_fused_smem(n, E);
        cudaError_t err = cudaFuncSetAttribute(align_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                               (int)smem);
        if (err != cudaSuccess) return err;
        FT_LAUNCH(align_fused_kernel, dim3(1), dim3(1024), smem, s, ids, n, k, E, B, sorted_slot, block_expert,
                  expert_off, n_padded, status, zero, (int)(zero_bytes / sizeof(int)));
        count_launches(1);
        return cudaGetLastError();
    }
    if (zero_bytes) {
        cudaError_t err = cudaMemsetAsync(zero, 0, zero_bytes, s);
        if (err != cudaSuccess) return err;
    }
    const int chunks = (n + kAlignChunk - 1) / kAlignChunk;
    int *chunk_cnt = static_cast<int *>(scratch);
    int *rank = reinterpret_cast<int *>(static_cast<char *>(scratch) + round_up((size_t)chunks * E * sizeof(int), 256));
    size_t smem1 = sizeof(int) * 8 * (size_t)E;
    cudaError_t err = cudaFuncSetAttribute(align_count_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem1);
    if (err != cudaSuccess) return err;
    FT_LAUNCH(align_count_kernel, dim3(chunks), dim3(256), smem1, s, ids, n, k, E, chunk_cnt, rank, status);
    size_t smem2 = sizeof(int) * ((size_t)(E + 1) + E + 33);
    FT_LAUNCH(align_scan_kernel, dim3(1), dim3(1024), smem2, s, chunk_cnt, chunks, E, B, n, sorted_slot,
              block_expert, expert_off, n_padded);
    FT_LAUNCH(align_place_kernel, dim3((n + 255) / 256), dim3(256), 0, s, ids, n, E, chunk_cnt, rank,
              expert_off, sorted_slot);
    count_launches(3);
    return cudaGetLastError();
}

}  // namespace ftmoe
