// Host-side declarations shared by the libftmoe translation units.
#pragma once

#include <cuda.h>
#include <nvtx3/nvToolsExt.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "ft_moe.h"

namespace ftmoe {

// Slots are grouped into blocks of this many rows for the warp-MMA (decode) path:
// one block is the N=8 side of an m16n8k16 MMA.
constexpr int kGemvBlock = 8;
// Align: slot counts up to this size are sorted by one CTA when its shared memory
// (32 E + 2 n + 2 E + 34 ints) fits; larger ones by three grid-wide passes over chunks of
// kAlignChunk slots.
constexpr int kAlignFusedMax = 8192;
constexpr int kAlignChunk = 2048;

// Everything one grouped warp-MMA launch needs. Rows of an expert matrix are the
// MMA M side (16 per warp tile); up to eight activation rows (slots of one block)
// are the N side; K is split across KSPLIT warps of the CTA.
struct GemvParams {
    const uint8_t *codes;    // [E][R][K/2]
    const uint8_t *scales;   // [E][R][K/group]
    const float *glob;       // [E][R]
    int64_t e_codes, e_scales, e_glob;  // per-expert strides (elements)
    int R, K, group;
    int up_off;              // gated: row offset of the up half (I_l)
    const uint16_t *act;     // bf16 rows of length K
    const int *n_pos_dev;    // routed: device count of padded positions
    int n_pos_static;        // shared: number of positions (tokens)
    const int *sorted_slot;  // routed: position -> slot (>= n_slots: padding)
    const int *block_expert; // routed: block -> expert
    int n_slots;             // routed: T*k; shared: T
    int top_k;               // routed: k (slot -> token); shared: 1
    int n_tiles;             // CTA tiles per block
    int num_experts;
    uint16_t *h_out;         // gated: bf16 [positions][h_ld]
    int h_ld;
    float *y_out;            // down: f32 [n_slots][R]
    const float *route_w;    // down, routed: [T*k]; nullptr = weight 1
    int *status;
    const float *sinv;       // fp8_block: scale_inv [E][R/128][K/128] (codes are then [E][R][K])
    int64_t e_sinv;          // fp8_block: per-expert stride of sinv (elements)
};

// Positions per block (the MMA N side) of the tensor-core prefill path.
constexpr int kTcBlock = 128;

// One grouped GEMM launch of the tensor-core path. Rows of expert e's matrix are
// e * R .. e * R + R - 1 of the bank; a unit is (block of kTcBlock positions, tile of
// 128 rows); gate_up units pair gate rows with the up rows up_off further down.
struct TcParams {
    const uint8_t *scales;   // [E][R][K/group]
    const float *glob;       // [E][R]
    int R, K, group, up_off, n_mtiles;
    const int *n_pos_dev;    // routed: device count of padded positions
    int n_pos_static;        // shared: number of tokens
    const int *sorted_slot;  // routed: position -> slot
    const int *block_expert; // routed: block -> expert
    int n_slots, top_k;
    int num_experts;         // routed: E (block_expert values index the banks); shared: 1
    uint16_t *h_out;         // gate_up: bf16 [positions][h_ld]
    int h_ld;
    float *y_out;            // down: fp32 [slots][y_ld]
    int y_ld;
    const float *route_w;    // down, routed: [T*k]
    const float *act_scale;  // per position: factor that undoes the B rows' f16 scaling (or null)
    int *status;
    int fp8;                 // fp8_block banks: codes [E][R][K] bytes, sinv below, no globals
    const float *sinv;       // fp8_block: scale_inv [E][R/128][K/128]
    int64_t e_sinv;          // fp8_block: per-expert stride of sinv (elements)
};
// One tensor-core grouped GEMM launch over up to two problems of the same stage, format
// and group (the routed experts, then the shared expert): units of problem 0, then of
// problem 1; K may differ between them.
struct TcLaunch {
    TcParams prob[2];
    int nprob;
    uint64_t wait_ns;   // limit of every barrier wait (0: the default, about two seconds)
    int skip_producer;  // fault injection: issue no copies, so the consumers' waits run out
    int scale_load_bytes;  // NVFP4 block scales read 16 (or 8, when some K/group is 8 mod 16) bytes at a time
};
// Fault injection armed by ft_moe_debug_inject_stall for the current ft_moe_forward call
// on this thread: the wait limit (0 = default) and whether the pipelined kernels skip
// their producer role.
void injected_stall(uint64_t *wait_ns, int *skip_producer);
// The operands of one problem: its bank's packed codes (rows_total rows) and the f16
// matrix its B operand comes from (act_rows rows of K).
struct TcOperands {
    const void *codes;
    int64_t rows_total;
    const void *act;
    int64_t act_rows;
};
bool tc_shape_ok(int K, int group, int rows_per_expert);
bool tc_shape_ok_fp8(int K, int rows_per_expert);
// nprob (1 or 2) problems in one launch; max_units bounds their total unit count.
cudaError_t launch_tc_gemm(const TcParams *probs, const TcOperands *ops, int nprob, bool gated, int max_units,
                           cudaStream_t s);
// B rows for the f16 tensor-core path: out[pos] = f16(src[row] * 2^-e), scale[pos] = 2^e,
// row = token of sorted_slot[pos] (or pos when sorted_slot is null; rows >= n_slots and
// padding slots give zero rows). pos < *n_pos_dev, or < n_pos_static when that is null.
cudaError_t launch_rows_to_f16(const uint16_t *src, int K, const int *sorted_slot, const int *n_pos_dev,
                               int n_pos_static, int n_slots, int top_k, int max_rows, uint16_t *out, float *scale,
                               cudaStream_t s, int *status);
// One W4A4 (native FP4) grouped GEMM problem: NVFP4 weight banks against NVFP4-quantized
// activation rows (codes, e4m3 scales per 16 elements, fp32 row scale per position).
struct W4Params {
    const uint8_t *w_scales;  // [E][R][K/group] e4m3
    const float *w_glob;      // [E][R]
    const uint8_t *a_scales;  // [positions][K/16] e4m3
    const float *a_glob;      // [positions]
    int R, K, group, up_off, n_mtiles;
    const int *n_pos_dev;     // routed: device count of padded positions
    int n_pos_static;         // shared: number of tokens
    const int *sorted_slot;   // routed: position -> slot
    const int *block_expert;  // routed: block -> expert
    int n_slots, top_k;
    int num_experts;          // routed: E; shared: 1
    float *h_out;             // gate_up: fp32 [positions][h_ld]
    int h_ld;
    float *y_out;             // down: fp32 [slots][y_ld]
    int y_ld;
    const float *route_w;     // down, routed: [T*k]
    int *status;
};
struct W4Launch {
    W4Params prob[2];
    int nprob;
    uint64_t wait_ns;
    int skip_producer;
};
struct W4Operands {
    const void *codes;        // the bank's packed weight codes
    int64_t rows_total;
    const void *act_codes;    // quantized activation codes, [act_rows][K/2]
    int64_t act_rows;
};
bool w4a4_shape_ok(int K, int rows_per_expert);
cudaError_t launch_w4a4_gemm(const W4Params *probs, const W4Operands *ops, int nprob, bool gated, int max_units,
                             cudaStream_t s);
// NVFP4 quantization of position rows (the token of sorted_slot[pos], or pos itself; bf16 or
// fp32 source rows of K elements, K a multiple of 16): codes [pos][K/2], e4m3 scales
// [pos][K/16], fp32 row scales [pos]; padding positions get zeros.
cudaError_t launch_quant_nvfp4(const void *src, bool f32_src, int K, const int *sorted_slot, const int *n_pos_dev,
                               int n_pos_static, int n_slots, int top_k, int max_rows, uint8_t *codes,
                               uint8_t *scales, float *glob, cudaStream_t s, int *status);

// 2D tiled tensor map (rows of `row_bytes` bytes, `inner` elements used per row) through
// the driver's cuTensorMapEncodeTiled; false when the driver refuses the shape.
bool make_tensor_map_2d(CUtensorMap *map, CUtensorMapDataType dt, const void *base, uint64_t inner, uint64_t rows,
                        uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows, CUtensorMapSwizzle swz);

int sm_count();

// Launch with programmatic stream serialization: the kernel may be scheduled before its
// predecessor in the stream finishes; it waits for it in pdl_wait() before touching
// memory (every kernel of the library starts with pdl_enter()).
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kern)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t s, Args... args)
{
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kern, static_cast<KArgs>(args)...);
}
// launch_pdl inside a function returning cudaError_t: return the launch error, if any.
#define FT_LAUNCH(...)                                                                                         \
    do {                                                                                                       \
        const cudaError_t le_ = launch_pdl(__VA_ARGS__);                                                       \
        if (le_ != cudaSuccess) return le_;                                                                    \
    } while (0)
// An NVTX range named after the ABI call for the scope of the call (header-only NVTX 3:
// nothing is loaded unless a profiler is attached), so that profiles group each call's
// launches.
struct NvtxScope {
    explicit NvtxScope(const char *name) { nvtxRangePushA(name); }
    ~NvtxScope() { nvtxRangePop(); }
    NvtxScope(const NvtxScope &) = delete;
    NvtxScope &operator=(const NvtxScope &) = delete;
};
#define FT_NVTX_RANGE(name) const NvtxScope ft_nvtx_scope_(name)

// Sets the thread-local error message (cleared for FT_OK) and returns `code`.
ft_status report_error(ft_status code, const char *message);
// Adds n to the calling thread's launch counter (ft_moe_launch_count).
void count_launches(int n);

cudaError_t launch_route(const float *logits, int T, int E, int k, int32_t *ids, float *w, cudaStream_t s);
// logits [T][E] (fp32) = x [T][H] . w [E][H]^T over bf16; H % 32 == 0.
cudaError_t launch_router_gemm(const uint16_t *x, const uint16_t *w, int T, int H, int E, float *logits,
                               cudaStream_t s);

// Align into caller buffers; `scratch` holds kAlignChunk-sized chunk counts and
// per-slot ranks (align_scratch_bytes). The zero_bytes at `zero` (a multiple of 4, the
// status word among them) are cleared first, in the align launch itself when it is a
// single CTA.
size_t align_scratch_bytes(int n_slots, int E);
cudaError_t launch_align(const int32_t *ids, int T, int k, int E, int B, int32_t *sorted_slot,
                         int32_t *block_expert, int32_t *expert_off, int32_t *n_padded, int *status,
                         void *scratch, cudaStream_t s, int *zero = nullptr, size_t zero_bytes = 0);

// K-split (1, 2, 4 or 8 warps per row tile) for a launch whose CTA-unit count at
// K-split 1 is max_blocks * units_per_block_ks1.
int gemv_ksplit(int max_blocks, int units_per_block_ks1, int K);
// p.n_tiles = CTA units per block: ceil(rows / (16 * 8 / ks)) with rows = I_l (gated) or H.
cudaError_t launch_gemv_gated(const GemvParams &p, int ks, int max_units, cudaStream_t s);
cudaError_t launch_gemv_down(const GemvParams &p, int ks, int max_units, cudaStream_t s);
// Lean register-fed GEMV (two 16-row tiles per warp): usable when K % 32 == 0 and
// (K / ks) % 128 == 0 and one expert's R x K codes take under 2 GB. p.n_tiles =
// ceil(rows / (pair_rows * 8 / ks)).
bool gemv_fast_ok(int K, int group, int ks, int R);

// One lean-GEMV launch over up to two problems (routed experts, shared expert); the
// down stage writes the slot-major y rows, and the combine runs as its own launch.
struct FastLaunch {
    GemvParams prob[2];
    int nprob;
    // Even split of the K steps over the CTAs (register-fed kernel, no in-CTA K split): a
    // unit shared by CTAs c and c + 1 leaves each piece's partial sums in
    // split_part[c][piece] and the second arrival on split_cnt[c] finishes it. Null: each
    // CTA takes whole units. split_cnt is zero at launch; at most kMaxSplitSlots CTAs.
    float *split_part;
    int *split_cnt;
};
constexpr int kMaxSplitSlots = 512;
constexpr size_t kSplitPartFloats = 2 * 256 * 8;  // two pieces x 256 threads x 8 partial sums
cudaError_t launch_gemv_fast(const FastLaunch &L, bool gated, int ks, int max_units, cudaStream_t s);

// The fused decode launch: the gate_up stage (gu, as for launch_gemv_fast with gated =
// true, its split buffers included), the down stage (dn) and the ordered combine in one
// persistent kernel. gu_done (one counter per block: the routed expert's blocks, then the
// shared expert's from shared_base) and done are zero at launch.
struct FusedLaunch {
    FastLaunch gu, dn;
    int *gu_done;
    int shared_base;
    int *done;
    const float *y, *y_sh;  // the down stage's outputs (dn.prob[0/1].y_out), combined in order
    void *out;
    int out_dtype, T, k, H;
    int *status;
    uint64_t wait_ns;       // limit of every cross-CTA wait (0: the default, about two seconds)
    int skip_publish;       // fault injection: gate_up publishes no finished units, so down's waits run out
};
// ks_gu in {1, 2, 4, 8}, ks_dn in {1, 2, 4}; max_units bounds the larger stage's unit count.
cudaError_t launch_gemv_fused(const FusedLaunch &F, int ks_gu, int ks_dn, int max_units, cudaStream_t s);

// fp8_block grouped GEMV (register-fed, any batch size): K a whole number of 128-element
// scale blocks per warp's share.
bool gemv_fp8_ok(int K, int ks);
cudaError_t launch_gemv_fp8(const FastLaunch &L, bool gated, int ks, int max_units, cudaStream_t s);

cudaError_t launch_combine(const float *y, const float *y_shared, int T, int k, int H, void *out, int out_dtype,
                           cudaStream_t s);

cudaError_t launch_pack_copy2d(const uint8_t *src, size_t src_pitch, uint8_t *dst, size_t dst_pitch,
                               size_t width, size_t height, cudaStream_t s);
cudaError_t launch_dequant(const uint8_t *codes, const uint8_t *scales, int rows, int K, int group,
                           uint16_t *out, cudaStream_t s);

}  // namespace ftmoe
