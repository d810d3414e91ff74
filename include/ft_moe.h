/*
 * ft_moe.h -- C ABI of libftmoe, the sm_103a NVFP4 (W4A16) routed-MoE expert forward.
 *
 * The layer (sources: "[TP=2] Quantized MoE expert parallelism on heterogeneous
 * consumer CUDA GPUs -- a working NVFP4 port", sections 2 and 4 with the diffs of
 * nvfp4.py and nvfp4_banks.py; "Offloaded MoE ignores tensor parallelism", sections
 * "The fix that fits" and "What it touches", and its follow-up comment;
 * "feat(qwen3_5_moe): tensor-parallel weight sharding", Implementation notes;
 * "[1/3] feat(dsv4): add tensor-parallel DeepSeek-V4 runtime", table "Tensor
 * ownership and collectives"):
 *
 *   route:    p = softmax(logits_t); keep the top-k (descending, ties to the lower
 *             expert index); w_j = p_j / sum of kept p              (norm_topk_prob)
 *   gate_up:  G[s, n] = sum_k x[t, k] * W_gu[e][n][k],  n < 2*I_l    (gate rows first)
 *   SwiGLU:   h[s, i] = silu(G[s, i]) * G[s, I_l + i]
 *   down:     y[s, n] = sum_i h[s, i] * W_dn[e][n][i],  n < H
 *   combine:  out[t, :] = sum_{j<k} w[t, j] * y[t*k + j, :] + shared(x_t)
 *
 * with W[n][k] = e2m1(code[n][k]) * e4m3(scale[n][k / group]) * global[n]. At
 * tp_size > 1 every bank holds rank tp_rank's slice of the intermediate axis and
 * the result is that rank's hidden-width partial sum; the sum over ranks equals
 * the tp_size = 1 output (the linearity argument of the NVFP4 port, section 4).
 * No collective is issued by this library.
 *
 * Storage conventions
 *   - Packed codes: two e2m1 codes per byte, element 2m in the LOW nibble of byte m,
 *     element 2m+1 in the high nibble; nibble bit 3 is the sign.
 *   - Block scales: OCP FP8 E4M3 ("fn") bytes, one per `group` consecutive elements
 *     along K (the packed axis).
 *   - Globals: fp32, one per output row (the checkpoint's per-tensor weight_scale_2
 *     expanded to rows, as the pages' fused_global/global_rows do).
 *   - Activations: bf16, row-major [T, H]. Outputs: bf16 or fp32, row-major [T, H].
 *
 * Memory and threading
 *   - All device memory is owned by the caller. The library allocates nothing on
 *     the device and keeps no per-call state; sizes come from ft_moe_layout and
 *     ft_moe_workspace_size.
 *   - Every call that takes a stream is asynchronous on that stream (cudaStream_t,
 *     passed as void*; NULL is the legacy default stream). Argument and geometry
 *     errors are detected on the host and returned before anything is launched.
 *   - Errors detected by kernels (invalid routing ids, bounded waits that ran out)
 *     are recorded in a status word inside the workspace and read back with
 *     ft_moe_read_status.
 *   - A failing call sets a thread-local message readable with ft_last_error().
 *
 * Limits: 1 <= top_k <= 32, top_k <= num_experts <= 1024, group in {16, 32},
 * hidden a multiple of 128, T <= 2^20.
 */
#ifndef FT_MOE_H
#define FT_MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    FT_OK = 0,
    FT_ERR_INVALID_ARG = 1,      /* null/misaligned pointer, bad size or enum */
    FT_ERR_INDIVISIBLE = 2,      /* tp split or quantisation block does not divide */
    FT_ERR_UNSUPPORTED = 3,      /* shape outside the limits above */
    FT_ERR_WORKSPACE = 4,        /* workspace smaller than ft_moe_workspace_size */
    FT_ERR_CUDA = 5,             /* a CUDA runtime call or launch failed */
    FT_ERR_INVALID_ROUTING = 6,  /* device: an expert id out of range or repeated in a row */
    FT_ERR_TIMEOUT = 7,          /* device: a bounded wait gave up */
    FT_ERR_BOUNDS = 8            /* device, bounds-checking builds only: an index derived from the
                                    routing (expert id, slot, padded count) was out of range */
} ft_status;

/* Geometry of one MoE layer as seen by one tp rank. `intermediate` and
 * `shared_intermediate` are the FULL (unsliced) sizes; the rank-local sizes are
 * I_l = intermediate / tp_size and I_sl = shared_intermediate / tp_size (the rank's
 * share of the intermediate axis that the NVFP4 port's MoE config derives from the full
 * size and tp_size, NVFP4 port section 3a), or the explicit shard sizes below. shared_intermediate = 0 means the
 * layer has no shared expert. A shard range that is negative, empty, not a multiple
 * of group or past the full size is FT_ERR_INDIVISIBLE. */
typedef struct {
    int32_t hidden;               /* H */
    int32_t intermediate;         /* I (full) */
    int32_t num_experts;          /* E */
    int32_t top_k;                /* k */
    int32_t group;                /* elements per e4m3 block scale: 16 (NVFP4) or 32 */
    int32_t shared_intermediate;  /* I_s (full), 0 = none */
    int32_t tp_rank;              /* r in [0, tp_size) */
    int32_t tp_size;              /* >= 1 */
    /* Asymmetric split (optional): with shard_size > 0 this rank owns the explicit
     * intermediate range [shard_begin, shard_begin + shard_size) instead of the even
     * share [r*I/tp, (r+1)*I/tp). The pages leave such a ratio open ("[TP=2] Quantized
     * MoE expert parallelism ... NVFP4 port", section 8: a split weighted toward the
     * faster card was not attempted); the slicing rule and the exact sum of partials
     * over any partition of [0, I) carry over from the even split (section 4). Both
     * values must be multiples of group; 0 = even split. The shared expert likewise
     * with shared_shard_begin / shared_shard_size (0 = its even share). */
    int32_t shard_begin;
    int32_t shard_size;
    int32_t shared_shard_begin;
    int32_t shared_shard_size;
    /* Expert weight format (FT_FORMAT_*). FT_FORMAT_FP8_BLOCK is the fp8-block expert
     * format the sharding pages carry beside NVFP4 ("feat(qwen3_5_moe): tensor-parallel
     * weight sharding", Summary and Implementation notes; the dsv4 PR, Checkpoint
     * loading: FP8 128x128 blocks): one e4m3 code byte per weight and an fp32
     * weight_scale_inv per 128 x 128 block, W = code * scale_inv, no per-row global.
     * It needs group = 128, and H, the rank's intermediate share (and any explicit
     * range) multiples of 128 (the same issue's item 2: "128 for fp8_block"). */
    int32_t format;
} ft_moe_config;

enum { FT_FORMAT_NVFP4 = 0, FT_FORMAT_FP8_BLOCK = 1 };

enum { FT_DTYPE_U8 = 0, FT_DTYPE_E4M3 = 1, FT_DTYPE_F32 = 2, FT_DTYPE_BF16 = 3 };

/* Bank indices, in the order of the pages' BankSpec layout. */
enum { FT_GU = 0, FT_GU_SCALE, FT_GU_GLOBAL, FT_DN, FT_DN_SCALE, FT_DN_GLOBAL, FT_NBANKS };

typedef struct {
    int64_t shape[3];
    int32_t ndim;
    int32_t dtype;   /* FT_DTYPE_* */
    int64_t bytes;
} ft_bank_spec;

/* Rank-local banks of one expert set, expert-major (routed: E experts; shared: 1):
 *   p[FT_GU]        u8   [E, 2*I_l, H/2]   gate rows [0, I_l), up rows [I_l, 2*I_l)
 *   p[FT_GU_SCALE]  e4m3 [E, 2*I_l, H/group]
 *   p[FT_GU_GLOBAL] f32  [E, 2*I_l]
 *   p[FT_DN]        u8   [E, H, I_l/2]
 *   p[FT_DN_SCALE]  e4m3 [E, H, I_l/group]
 *   p[FT_DN_GLOBAL] f32  [E, H]
 * FT_FORMAT_FP8_BLOCK instead:
 *   p[FT_GU]        u8 (e4m3 codes) [E, 2*I_l, H]
 *   p[FT_GU_SCALE]  f32 [E, 2*I_l/128, H/128]   scale_inv, gate block rows first
 *   p[FT_DN]        u8 (e4m3 codes) [E, H, I_l]
 *   p[FT_DN_SCALE]  f32 [E, H/128, I_l/128]
 *   p[FT_GU_GLOBAL], p[FT_DN_GLOBAL]: none (0 bytes; the pointers may be NULL).
 * Device pointers, caller-owned, each 16-byte aligned. */
typedef struct { void *p[FT_NBANKS]; } ft_moe_banks;

/* Checkpoint-shaped expert tensors at FULL intermediate size, expert-major (the
 * nine tensors per expert the NVFP4 port's loader yields: weight, _scale, _global
 * of gate, up and down):
 *   gate, up          u8 [E, I, H/2];  gate_scale, up_scale  e4m3 [E, I, H/group];
 *   gate_global, up_global f32 [E, I]
 *   down u8 [E, H, I/2];  down_scale e4m3 [E, H, I/group];  down_global f32 [E, H]
 * FT_FORMAT_FP8_BLOCK: gate, up u8 [E, I, H] with gate_scale, up_scale f32 scale_inv
 * [E, I/128, H/128]; down u8 [E, H, I] with down_scale f32 [E, H/128, I/128]; the
 * three _global pointers are ignored (may be NULL).
 * on_device = 1: all are device pointers; 0: all are host pointers. */
typedef struct {
    const void *gate, *gate_scale, *gate_global;
    const void *up, *up_scale, *up_global;
    const void *down, *down_scale, *down_global;
    int32_t on_device;
} ft_moe_pieces;

/* Shapes and byte sizes of the six rank-local banks.
 * Follows the NVFP4 kernel's layout() sized by cfg.local_intermediate (NVFP4 port,
 * section 4 and the nvfp4.py diff). shared = 0: routed banks (E experts, I_l);
 * shared = 1: shared-expert banks (1 expert, I_sl).
 * Errors: FT_ERR_INVALID_ARG for null pointers or bad fields; FT_ERR_INDIVISIBLE
 * when I % tp, (I/tp) % group, H % group, I_s % tp or (I_s/tp) % group is nonzero
 * ("I/tp must stay a multiple of each format's block size", issue "Offloaded MoE
 * ignores tensor parallelism", What it touches item 2 -- never padded);
 * FT_ERR_UNSUPPORTED outside the limits above, or shared = 1 without a shared
 * expert. Host-only, no CUDA call. */
ft_status ft_moe_layout(const ft_moe_config *cfg, int32_t shared, ft_bank_spec out[FT_NBANKS]);

/* Fill rank tp_rank's banks from full checkpoint-shaped pieces:
 * gate_up rows [0, I_l) = gate rows [r*I_l, (r+1)*I_l), rows [I_l, 2*I_l) = up rows
 * [r*I_l, (r+1)*I_l) (in the fused [2I, .] view the two disjoint ranges of the
 * issue's What it touches item 1); their scales and globals follow the rows. down
 * keeps all H rows and takes code columns [r*I_l/2, (r+1)*I_l/2) and scale columns
 * [r*I_l/group, ...) (_shard_expert_tensor: gate/up dim 0, down the last dim);
 * down_global is copied whole. tp_size = 1 is the identity (byte-identical
 * concatenation). The destination banks are separate storage, never views of
 * the source (".clone()" rule of the dsv4 PR). Asynchronous on `stream`; with host
 * pieces the host buffers must stay valid until the stream reaches this point.
 * Errors: as ft_moe_layout, plus FT_ERR_INVALID_ARG for null/misaligned pointers
 * or overlapping source and destination, FT_ERR_CUDA. */
ft_status ft_moe_pack(const ft_moe_config *cfg, int32_t shared, const ft_moe_pieces *src,
                      const ft_moe_banks *dst, void *stream);

/* Router: for each of T tokens, softmax over E fp32 logits, the k largest in
 * descending order (ties to the lower expert index), weights renormalised to sum
 * to 1 ("Offloaded MoE ignores tensor parallelism", follow-up comment:
 * norm_topk_prob, replicated router). Selection compares the fp32 logits
 * themselves, which orders experts exactly as the probabilities do.
 *   logits    device f32 [T, E], row-major, finite values
 *   topk_ids  device i32 [T, k] (out)
 *   topk_w    device f32 [T, k] (out)
 * T = 0 is a no-op. Errors: FT_ERR_INVALID_ARG, FT_ERR_UNSUPPORTED (E > 1024,
 * k > 32, k > E), FT_ERR_CUDA. */
ft_status ft_moe_route(const float *logits, int32_t T, int32_t E, int32_t k,
                       int32_t *topk_ids, float *topk_w, void *stream);

/* Router with its logit GEMM: logits[t, e] = sum_h x[t, h] * w_router[e, h] over the
 * bf16 values, accumulated in fp32 (the router is replicated on every rank and every
 * rank computes the same routing: "[1/3] feat(dsv4): add tensor-parallel DeepSeek-V4
 * runtime", table "Tensor ownership and collectives"), then exactly ft_moe_route on
 * those logits.
 *   x         device bf16 [T, H], row-major, 16-byte aligned
 *   w_router  device bf16 [E, H], row-major, 16-byte aligned (caller-owned)
 *   logits    device f32 [T, E] (out, also the router's input), 4-byte aligned
 *   topk_ids  device i32 [T, k] (out); topk_w device f32 [T, k] (out)
 * H must be a multiple of 32. T = 0 is a no-op. Errors:
 * FT_ERR_INVALID_ARG (NULL or misaligned pointer, H not a positive multiple of 32),
 * FT_ERR_UNSUPPORTED (E > 1024, k > 32, k > E), FT_ERR_CUDA. */
ft_status ft_moe_route_gemm(const void *x, int32_t T, int32_t H, const void *w_router, int32_t E, int32_t k,
                            float *logits, int32_t *topk_ids, float *topk_w, void *stream);

/* Bytes of workspace ft_moe_forward needs for this config and token count
 * (256-byte aligned buffer). Host-only. The pages keep the layer's intermediates
 * (sorted token order, the SwiGLU activations h, the per-slot down outputs) as
 * framework-owned buffers ("feat(qwen3_5_moe): tensor-parallel weight sharding", Notes:
 * the moe_align step feeding the grouped GEMMs); here the caller owns them, sized by
 * this call, since the library allocates nothing. Errors: as ft_moe_layout, plus
 * FT_ERR_INVALID_ARG (bytes NULL) and FT_ERR_UNSUPPORTED (T outside [0, 2^20]). */
ft_status ft_moe_workspace_size(const ft_moe_config *cfg, int32_t T, size_t *bytes);

/* Rank-local MoE partial for T tokens:
 *   out[t, :] = sum_{j<k} topk_w[t, j] * expert_{topk_ids[t, j]}(x_t) + shared(x_t)
 * (routed and shared partials are added locally before any reduction, dsv4 PR
 * ownership table). Terms are accumulated in a fixed order, so repeated calls give
 * bitwise-identical results.
 *   routed    banks of all E experts (required)
 *   shared    banks of the shared expert, or NULL (required iff shared_intermediate > 0)
 *   x         device bf16 [T, H]
 *   topk_ids  device i32 [T, k]; topk_w device f32 [T, k]
 *   out       device [T, H], dtype FT_DTYPE_BF16 or FT_DTYPE_F32
 *   workspace device, >= ft_moe_workspace_size bytes, 256-byte aligned; its first
 *             bytes hold the status word read by ft_moe_read_status
 * T = 0 returns FT_OK without launching. Ids outside [0, E) or repeated within a
 * row set FT_ERR_INVALID_ROUTING in the status word (those slots are skipped).
 * Errors: FT_ERR_INVALID_ARG, FT_ERR_INDIVISIBLE, FT_ERR_UNSUPPORTED,
 * FT_ERR_WORKSPACE, FT_ERR_CUDA. */
ft_status ft_moe_forward(const ft_moe_config *cfg, const ft_moe_banks *routed, const ft_moe_banks *shared,
                         const void *x, int32_t T, const int32_t *topk_ids, const float *topk_w,
                         void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes,
                         void *stream);

/* ---- W4A4: the native block-scaled FP4 variant ------------------------------ */

/* The same rank-local partial with the activations in NVFP4 as well (W4A4): the path the
 * pages' sm_86/sm_89 cards could not take ("[TP=2] Quantized MoE expert parallelism ...
 * NVFP4 port", section 2: without FP4 tensor cores NVFP4 ran there as W4A16). Each token's
 * x (per expert-sorted position) and each expert's h (fp32, per position) are quantized with
 * ft_moe_quantize_nvfp4's rule, and both GEMMs run on tcgen05 kind::mxf4nvf4 with the e4m3
 * block scales of weights and activations as the MMA's scale factors; row globals and the
 * activations' row scales multiply the fp32 sums. The quantization changes the numbers: the
 * result equals the W4A16 forward only up to activation quantization error. Banks are the
 * NVFP4 banks of ft_moe_pack (group 16 or 32). Needs hidden and the rank's intermediate
 * sizes (routed and shared) to be multiples of 256, else FT_ERR_UNSUPPORTED. At tp_size > 1
 * each rank quantizes its own h slice, so the sum of partials matches the tp = 1 output only
 * up to that quantization. Arguments, errors and the status word as ft_moe_forward; the
 * workspace size comes from ft_moe_workspace_size_w4a4. */
ft_status ft_moe_workspace_size_w4a4(const ft_moe_config *cfg, int32_t T, size_t *bytes);
ft_status ft_moe_forward_w4a4(const ft_moe_config *cfg, const ft_moe_banks *routed, const ft_moe_banks *shared,
                              const void *x, int32_t T, const int32_t *topk_ids, const float *topk_w,
                              void *out, int32_t out_dtype, void *workspace, size_t workspace_bytes,
                              void *stream);

/* NVFP4 quantization of `rows` activation rows of K elements (K a multiple of 16), the rule
 * of the W4A4 path (the pages name the format but give no activation recipe; this is NVFP4's
 * own two-level scaling applied per row): row scale glob = amax / (6 * 448); per 16 elements
 * the e4m3 scale s = e4m3(block max / (6 * glob)); codes q = e2m1(x * r) with the block's
 * reciprocal r = 1 / (s * glob); every step one correctly rounded fp32 operation, both
 * conversions to nearest with ties to even, saturating. Value of an element:
 * e2m1(q) * e4m3(s) * glob.
 *   src     device rows, bf16 or fp32 (src_dtype FT_DTYPE_BF16 / FT_DTYPE_F32), [rows, K],
 *           16-byte aligned
 *   codes   device u8 [rows, K/2] (out), element 2m in the low nibble; 8-byte aligned
 *   scales  device u8 [rows, K/16] (out, e4m3); glob device f32 [rows] (out)
 * Errors: FT_ERR_INVALID_ARG, FT_ERR_CUDA. */
ft_status ft_moe_quantize_nvfp4(const void *src, int32_t src_dtype, int32_t rows, int32_t K, uint8_t *codes,
                                uint8_t *scales, float *glob, void *stream);

/* ---- test and debug exports ------------------------------------------------ */

/* Expert-sorted, tile-padded slot order (the moe_align step named in "feat(qwen3_5_moe):
 * tensor-parallel weight sharding", Notes). Slot s = t*k + j. Slots are grouped by
 * expert in increasing expert order, in increasing slot order within an expert;
 * each expert's run is padded with the sentinel T*k to a multiple of `block`;
 * experts without slots get no blocks.
 *   sorted_slot  device i32, capacity T*k + min(E, T*k)*(block-1)   (out)
 *   block_expert device i32, capacity (that capacity)/block          (out)
 *   expert_off   device i32 [E+1] start of each expert's padded run (out)
 *   n_padded     device i32 [1]                                      (out)
 *   workspace    device scratch of ft_moe_align_workspace_size bytes (256-aligned)
 * Ids outside [0, E) are skipped and flagged FT_ERR_INVALID_ROUTING in the status
 * word at the start of `workspace`. block in [1, 1024]. */
ft_status ft_moe_align_workspace_size(int32_t T, int32_t k, int32_t E, size_t *bytes);
ft_status ft_moe_align(const int32_t *topk_ids, int32_t T, int32_t k, int32_t E, int32_t block,
                       int32_t *sorted_slot, int32_t *block_expert, int32_t *expert_off,
                       int32_t *n_padded, void *workspace, size_t workspace_bytes, void *stream);

/* ft_moe_align without a workspace, for callers that cannot allocate device memory:
 * an engine that fixes every device allocation at start-up and may not allocate
 * afterwards, or a caller that only owns the buffers handed to it. The pages have no
 * counterpart: it is the same sort as ft_moe_align, with the scratch and the status
 * word in a static array of 393,472 bytes that the library holds on every GPU that
 * loads it, until the process exits. It still issues CUDA calls on `stream` (a memset,
 * kernel launches, a device-to-device copy of the status), so it must not be called
 * from a stream host callback or anywhere else the CUDA API may not be used.
 *   Limits: T*k <= 65536 slots, E <= 1024, k <= 32; larger inputs return
 *   FT_ERR_UNSUPPORTED (use ft_moe_align with a workspace).
 *   status  device i32 [1] (out, may be NULL): FT_OK or FT_ERR_INVALID_ROUTING.
 * Other arguments as ft_moe_align. The first call on each device (and again after a
 * cudaDeviceReset, in the new context) looks up the array's device address with that
 * device current; make that first call before any stream capture on that device.
 * All calls share the one array: calls that overlap on the GPU (other streams, other
 * threads) race and must be ordered by the caller. Allocates nothing. */
ft_status ft_moe_align_static(const int32_t *topk_ids, int32_t T, int32_t k, int32_t E, int32_t block,
                              int32_t *sorted_slot, int32_t *block_expert, int32_t *expert_off,
                              int32_t *n_padded, int32_t *status, void *stream);

/* Dequantised weights of one expert without the per-row global:
 * out[n, k] = bf16(e2m1(code[n][k]) * e4m3(scale[n][k/group])), exact in bf16 -- the
 * weight value the NVFP4 port's dequantiser produces before its fp16 matmul, less the
 * per-row global that this library applies to each row's fp32 sum instead ("[TP=2]
 * Quantized MoE expert parallelism ... NVFP4 port", section 4, the _dequant_nvfp4
 * routine of the weight.py diff, packed NVFP4 to bf16).
 * which = FT_GU (rows 2*I_l, K = H) or FT_DN (rows H, K = I_l); `banks` are
 * routed banks when shared = 0, else the shared expert's. out: device bf16 [rows, K].
 * It runs the same device routine the fused kernels use. */
ft_status ft_moe_dequant(const ft_moe_config *cfg, int32_t shared, const ft_moe_banks *banks,
                         int32_t which, int32_t expert, void *out_bf16, void *stream);

/* Synchronise `stream` and return the status word at the start of `workspace`
 * (FT_OK, FT_ERR_INVALID_ROUTING, FT_ERR_TIMEOUT, or FT_ERR_BOUNDS from a library built
 * with FTMOE_BOUNDS_CHECK). Returns FT_ERR_CUDA if the
 * stream itself failed. The pages want bad geometry to fail with an error rather
 * than run ("[1/3] feat(dsv4): add tensor-parallel DeepSeek-V4 runtime", Checkpoint
 * loading and memory correctness: incompatible sizes fail before any layer is built)
 * and count a stage that hangs instead of erroring as a defect ("Offloaded MoE ignores
 * tensor parallelism", follow-up comment: the rank-0 relay race that wedges the
 * server); kernels cannot return an error code, so they record the first one here for
 * the host to read. */
ft_status ft_moe_read_status(const void *workspace, void *stream);

/* Thread-local description of the last error returned on this thread ("" if none). */
const char *ft_last_error(void);

/* ---- measurement hooks ------------------------------------------------------ */

/* Stages of one ft_moe_forward call, in launch order. */
enum { FT_STAGE_ALIGN = 0, FT_STAGE_GATE_UP, FT_STAGE_SHARED_GATE_UP, FT_STAGE_DOWN, FT_STAGE_SHARED_DOWN,
       FT_STAGE_COMBINE, FT_NSTAGES };

/* Arm per-stage timing for the next ft_moe_forward call on this thread: `events`
 * points to FT_NSTAGES + 1 cudaEvent_t handles (created by the caller); the call
 * records events[i] on its stream just before stage i and events[FT_NSTAGES] after
 * the last stage (stages absent for this layer record back-to-back events). Inside
 * a stream capture the records become event-record graph nodes. The hook disarms
 * itself after one forward call; events = NULL disarms it explicitly. */
ft_status ft_moe_set_stage_events(void *const *events);

/* Fault injection for tests of the error path, armed for the next ft_moe_forward call
 * on this thread that launches kernels (then disarmed). wait_limit_ns replaces the
 * pipelined kernels' limit on every barrier wait (0 = the default, about two seconds;
 * otherwise 1 ms to 2 s); skip_producer = 1 makes the tensor-core (prefill) kernels issue
 * no copies, so that their consumers' bounded waits run out: each CTA then records
 * FT_ERR_TIMEOUT in the status word, stops, frees its tensor memory and returns, and
 * the stream and the context stay usable. In the fused decode kernel skip_producer = 1
 * makes the gate_up stage publish no finished block, so that every down unit's bounded
 * wait for its block runs out, with the same outcome. The pages count a distributed stage that wedges instead of failing as a
 * defect ("Offloaded MoE ignores tensor parallelism", follow-up comment: the rank-0
 * relay race); this hook shows that a stalled pipeline here ends with an error status.
 * Errors: FT_ERR_INVALID_ARG (skip_producer not 0/1, limit out of range). Host-only. */
ft_status ft_moe_debug_inject_stall(uint64_t wait_limit_ns, int32_t skip_producer);

/* Number of kernels this library has launched (or captured into a graph) from the
 * calling thread since it was loaded. */
int64_t ft_moe_launch_count(void);

#ifdef __cplusplus
}
#endif

#endif /* FT_MOE_H */
