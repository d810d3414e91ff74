// extern "C" entry points of libftmoe: argument validation, workspace layout and
// kernel orchestration. See include/ft_moe.h for the contract of every call.
#include <cuda_runtime.h>
#include <stdarg.h>
#include <stdio.h>
#include <string.h>

#include "ft_moe.h"
#include "ftmoe_internal.h"

namespace ftmoe {

static thread_local char g_err[512];
static thread_local cudaEvent_t g_stage_events[FT_NSTAGES + 1];
static thread_local bool g_stage_armed = false;
static thread_local int64_t g_launches = 0;

void count_launches(int n) { g_launches += n; }

// Fault injection (ft_moe_debug_inject_stall): armed on the host for one forward call.
static thread_local bool g_stall_armed = false;
static thread_local bool g_stall_active = false;  // inside the forward call it was armed for
static thread_local uint64_t g_stall_wait_ns = 0;
static constexpr uint64_t kWaitNsMax = 2000000000ull;  // the kernels' default limit
static thread_local int g_stall_skip = 0;

void injected_stall(uint64_t *wait_ns, int *skip_producer)
{
    *wait_ns = g_stall_active ? g_stall_wait_ns : 0;
    *skip_producer = g_stall_active ? g_stall_skip : 0;
}

// Record the stage boundary event i, if timing is armed.
static cudaError_t stage_mark(int i, cudaStream_t s)
{
    if (!g_stage_armed) return cudaSuccess;
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    cudaError_t e = cudaStreamIsCapturing(s, &cs);
    if (e != cudaSuccess) return e;
    return cudaEventRecordWithFlags(g_stage_events[i], s,
                                    cs == cudaStreamCaptureStatusActive ? cudaEventRecordExternal : 0);
}

static ft_status fail(ft_status code, const char *fmt, ...)
{
    va_list ap;
    va_start(ap, fmt);
    vsnprintf(g_err, sizeof(g_err), fmt, ap);
    va_end(ap);
    return code;
}

static ft_status ok()
{
    g_err[0] = 0;
    return FT_OK;
}

ft_status report_error(ft_status code, const char *message)
{
    if (code == FT_OK) return ok();
    return fail(code, "%s", message);
}

static ft_status cuda_fail(cudaError_t e, const char *what)
{
    return fail(FT_ERR_CUDA, "%s: %s", what, cudaGetErrorString(e));
}

int sm_count()
{
    static int cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 148;
    if (cache[dev] == 0) {
        int n = 0;
        if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 148;
        cache[dev] = n;
    }
    return cache[dev];
}

static size_t round_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// Slot counts (T * top_k) up to this many run the decode regime as one fused launch.
constexpr int kFusedMaxSlots = 64;

static bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

// ---------------------------------------------------------------- geometry

struct Geometry {
    int H, I, E, k, g, Is, r, tp;
    int fmt;         // FT_FORMAT_*
    int Il, Isl;     // rank-local intermediate sizes (routed, shared)
    int rb, sb;      // first intermediate column of the rank's range (routed, shared)
};

static ft_status check_config(const ft_moe_config *cfg, Geometry &G)
{
    if (!cfg) return fail(FT_ERR_INVALID_ARG, "config is NULL");
    G.H = cfg->hidden; G.I = cfg->intermediate; G.E = cfg->num_experts; G.k = cfg->top_k;
    G.g = cfg->group; G.Is = cfg->shared_intermediate; G.r = cfg->tp_rank; G.tp = cfg->tp_size;
    if (G.H <= 0 || G.I <= 0 || G.E <= 0 || G.k <= 0 || G.Is < 0 || G.tp <= 0 || G.r < 0 || G.r >= G.tp)
        return fail(FT_ERR_INVALID_ARG, "config fields must be positive and 0 <= tp_rank < tp_size");
    if (cfg->shard_size < 0 || cfg->shared_shard_size < 0)
        return fail(FT_ERR_INVALID_ARG, "shard sizes must be >= 0 (0 = even split by tp_rank/tp_size)");
    G.fmt = cfg->format;
    if (G.fmt != FT_FORMAT_NVFP4 && G.fmt != FT_FORMAT_FP8_BLOCK)
        return fail(FT_ERR_INVALID_ARG, "unknown weight format %d", G.fmt);
    if (G.fmt == FT_FORMAT_FP8_BLOCK && G.g != 128)
        return fail(FT_ERR_UNSUPPORTED, "fp8_block needs group = 128 (its scale block; got %d)", G.g);
    if (G.fmt == FT_FORMAT_NVFP4 && G.g != 16 && G.g != 32)
        return fail(FT_ERR_UNSUPPORTED, "group must be 16 or 32 (got %d)", G.g);
    if (G.E > 1024 || G.k > 32 || G.k > G.E)
        return fail(FT_ERR_UNSUPPORTED, "need top_k <= 32, top_k <= num_experts <= 1024");
    if (G.H % G.g || G.H % 2)
        return fail(FT_ERR_INDIVISIBLE, "hidden %d is not a multiple of the %d-element scale block", G.H, G.g);
    if (cfg->shard_size > 0) {  // explicit (possibly asymmetric) range
        G.rb = cfg->shard_begin;
        G.Il = cfg->shard_size;
        if (G.rb < 0 || G.rb % G.g || G.Il % G.g || G.rb + G.Il > G.I)
            return fail(FT_ERR_INDIVISIBLE, "shard [%d, %d) is not a range of whole %d-element blocks inside [0, %d)",
                        G.rb, G.rb + G.Il, G.g, G.I);
    } else {
        if (G.I % G.tp)
            return fail(FT_ERR_INDIVISIBLE, "intermediate %d does not split across %d tp ranks", G.I, G.tp);
        G.Il = G.I / G.tp;
        G.rb = G.r * G.Il;
        if (G.Il % G.g)
            return fail(FT_ERR_INDIVISIBLE, "local intermediate %d is not a multiple of the %d-element scale block",
                        G.Il, G.g);
    }
    if (G.Is > 0 && cfg->shared_shard_size > 0) {
        G.sb = cfg->shared_shard_begin;
        G.Isl = cfg->shared_shard_size;
        if (G.sb < 0 || G.sb % G.g || G.Isl % G.g || G.sb + G.Isl > G.Is)
            return fail(FT_ERR_INDIVISIBLE, "shared shard [%d, %d) is not a range of whole %d-element blocks",
                        G.sb, G.sb + G.Isl, G.g);
    } else {
        if (G.Is % G.tp)
            return fail(FT_ERR_INDIVISIBLE, "shared intermediate %d does not split across %d tp ranks", G.Is, G.tp);
        G.Isl = G.Is / G.tp;
        G.sb = G.r * G.Isl;
        if (G.Isl % G.g)
            return fail(FT_ERR_INDIVISIBLE,
                        "local shared intermediate %d is not a multiple of the %d-element block", G.Isl, G.g);
    }
    if (G.H % 128) return fail(FT_ERR_UNSUPPORTED, "hidden must be a multiple of 128 (got %d)", G.H);
    return FT_OK;
}

static void spec(ft_bank_spec &s, int dtype, int64_t a, int64_t b, int64_t c, int nd)
{
    s.ndim = nd;
    s.dtype = dtype;
    s.shape[0] = a; s.shape[1] = b; s.shape[2] = nd == 3 ? c : 0;
    int64_t el = nd == 3 ? a * b * c : a * b;
    s.bytes = el * (dtype == FT_DTYPE_F32 ? 4 : 1);
}

static void bank_specs(const Geometry &G, int shared, ft_bank_spec out[FT_NBANKS])
{
    const int64_t E = shared ? 1 : G.E, Il = shared ? G.Isl : G.Il;
    if (G.fmt == FT_FORMAT_FP8_BLOCK) {
        spec(out[FT_GU], FT_DTYPE_U8, E, 2 * Il, G.H, 3);
        spec(out[FT_GU_SCALE], FT_DTYPE_F32, E, 2 * Il / 128, G.H / 128, 3);
        spec(out[FT_GU_GLOBAL], FT_DTYPE_F32, 0, 0, 0, 2);
        spec(out[FT_DN], FT_DTYPE_U8, E, G.H, Il, 3);
        spec(out[FT_DN_SCALE], FT_DTYPE_F32, E, G.H / 128, Il / 128, 3);
        spec(out[FT_DN_GLOBAL], FT_DTYPE_F32, 0, 0, 0, 2);
        return;
    }
    spec(out[FT_GU], FT_DTYPE_U8, E, 2 * Il, G.H / 2, 3);
    spec(out[FT_GU_SCALE], FT_DTYPE_E4M3, E, 2 * Il, G.H / G.g, 3);
    spec(out[FT_GU_GLOBAL], FT_DTYPE_F32, E, 2 * Il, 0, 2);
    spec(out[FT_DN], FT_DTYPE_U8, E, G.H, Il / 2, 3);
    spec(out[FT_DN_SCALE], FT_DTYPE_E4M3, E, G.H, Il / G.g, 3);
    spec(out[FT_DN_GLOBAL], FT_DTYPE_F32, E, G.H, 0, 2);
}

// Tensor-core (prefill) path when the routing gives the experts at least 32 slots on
// average and every tile shape fits; the warp-MMA (decode) path otherwise.
static bool use_tc(const Geometry &G, int T)
{
    if ((int64_t)T * G.k < (int64_t)32 * G.E || G.H % 256) return false;
    if (!tc_shape_ok(G.H, G.g, G.Il) || !tc_shape_ok(G.Il, G.g, G.H)) return false;
    if (G.Is && (!tc_shape_ok(G.H, G.g, G.Isl) || !tc_shape_ok(G.Isl, G.g, G.H))) return false;
    return true;
}

// The same for fp8_block banks (whole 128-row tiles, K a whole number of 128-blocks).
static bool use_tc_fp8(const Geometry &G, int T)
{
    if ((int64_t)T * G.k < (int64_t)32 * G.E || G.H % 256) return false;
    if (!tc_shape_ok_fp8(G.H, G.Il) || !tc_shape_ok_fp8(G.Il, G.H)) return false;
    if (G.Is && (!tc_shape_ok_fp8(G.H, G.Isl) || !tc_shape_ok_fp8(G.Isl, G.H))) return false;
    return true;
}

// Workspace regions of ft_moe_forward, each 256-byte aligned.
struct WsLayout {
    size_t status, split_cnt, gu_done, sorted, block_expert, expert_off, npad, scratch, h, h_sh, y, y_sh, total;
    size_t split_part;  // register-fed decode kernels: partial sums of units split between CTAs
    // tensor-core path only: f16 copies of the B operands and their per-row scales
    size_t xs, xs_scale, x16, x16_scale, h16, h16_scale, hsh16, hsh16_scale;
    size_t zero_bytes;  // [0, zero_bytes): status and split counts, cleared at the start of every forward
    int pmax;
};

static WsLayout ws_layout(const Geometry &G, int T)
{
    WsLayout L;
    const int64_t n = (int64_t)T * G.k;
    // sized for the larger padding block of the two paths (warp-MMA and tensor-core)
    const int64_t pmax = n + (int64_t)(n < G.E ? n : G.E) * (kTcBlock - 1);
    const int64_t tpad = (T + kTcBlock - 1) / kTcBlock * kTcBlock;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = round_up(o + bytes, 256); return at; };
    L.status = take(256);
    L.split_cnt = take(sizeof(int) * 2 * (size_t)kMaxSplitSlots);  // gate_up, down
    // fused decode kernel: per block (routed, then shared) finished gate_up units, and the
    // count of CTAs done with the down stage (the last int)
    L.gu_done = take(sizeof(int) * (size_t)(pmax / kGemvBlock + 1 + (T + kGemvBlock - 1) / kGemvBlock + 1));
    L.zero_bytes = o;
    L.sorted = take(sizeof(int) * (size_t)pmax);
    L.block_expert = take(sizeof(int) * (size_t)(pmax / kGemvBlock + 1));
    L.expert_off = take(sizeof(int) * (size_t)(G.E + 1));
    L.npad = take(sizeof(int));
    L.scratch = take(align_scratch_bytes((int)n, G.E));
    L.h = take(2 * (size_t)pmax * G.Il);
    L.h_sh = take(G.Is ? 2 * (size_t)tpad * G.Isl : 0);
    L.y = take(4 * (size_t)n * G.H);
    L.y_sh = take(G.Is ? 4 * (size_t)T * G.H : 0);
    L.split_part = take(sizeof(float) * (size_t)kMaxSplitSlots * kSplitPartFloats);
    const bool tc = G.fmt == FT_FORMAT_FP8_BLOCK ? use_tc_fp8(G, T) : use_tc(G, T);
    L.xs = take(tc ? 2 * (size_t)pmax * G.H : 0);
    L.xs_scale = take(tc ? 4 * (size_t)pmax : 0);
    L.x16 = take(tc && G.Is ? 2 * (size_t)tpad * G.H : 0);
    L.x16_scale = take(tc && G.Is ? 4 * (size_t)tpad : 0);
    L.h16 = take(tc ? 2 * (size_t)pmax * G.Il : 0);
    L.h16_scale = take(tc ? 4 * (size_t)pmax : 0);
    L.hsh16 = take(tc && G.Is ? 2 * (size_t)tpad * G.Isl : 0);
    L.hsh16_scale = take(tc && G.Is ? 4 * (size_t)tpad : 0);
    L.total = o;
    L.pmax = (int)pmax;
    return L;
}

// Workspace regions of ft_moe_forward_w4a4 (NVFP4 activations), each 256-byte aligned; the
// first regions (status word and counters, align outputs) are laid out as in ws_layout.
struct WsW4 {
    size_t status, split_cnt, sorted, block_expert, expert_off, npad, scratch, y, y_sh, zero_bytes;
    size_t xq_c, xq_s, xq_g, xs_c, xs_s, xs_g, h, hs, hq_c, hq_s, hq_g, hsq_c, hsq_s, hsq_g, total;
    int pmax, tpad;
};

static WsW4 ws_layout_w4a4(const Geometry &G, int T)
{
    WsW4 L;
    const int64_t n = (int64_t)T * G.k;
    const int64_t pmax = n + (int64_t)(n < G.E ? n : G.E) * (kTcBlock - 1);
    const int64_t tpad = (T + kTcBlock - 1) / kTcBlock * kTcBlock;
    size_t o = 0;
    auto take = [&](size_t bytes) { size_t at = o; o = round_up(o + bytes, 256); return at; };
    L.status = take(256);
    L.split_cnt = take(sizeof(int) * 2 * (size_t)kMaxSplitSlots);
    L.zero_bytes = o;
    L.sorted = take(sizeof(int) * (size_t)pmax);
    L.block_expert = take(sizeof(int) * (size_t)(pmax / kGemvBlock + 1));
    L.expert_off = take(sizeof(int) * (size_t)(G.E + 1));
    L.npad = take(sizeof(int));
    L.scratch = take(align_scratch_bytes((int)n, G.E));
    L.y = take(4 * (size_t)n * G.H);
    L.y_sh = take(G.Is ? 4 * (size_t)T * G.H : 0);
    const size_t sh = G.Is ? 1 : 0;
    L.xq_c = take((size_t)pmax * G.H / 2);
    L.xq_s = take((size_t)pmax * G.H / 16);
    L.xq_g = take(4 * (size_t)pmax);
    L.xs_c = take(sh * (size_t)tpad * G.H / 2);
    L.xs_s = take(sh * (size_t)tpad * G.H / 16);
    L.xs_g = take(sh * 4 * (size_t)tpad);
    L.h = take(4 * (size_t)pmax * G.Il);
    L.hs = take(sh * 4 * (size_t)tpad * G.Isl);
    L.hq_c = take((size_t)pmax * G.Il / 2);
    L.hq_s = take((size_t)pmax * G.Il / 16);
    L.hq_g = take(4 * (size_t)pmax);
    L.hsq_c = take(sh * (size_t)tpad * G.Isl / 2);
    L.hsq_s = take(sh * (size_t)tpad * G.Isl / 16);
    L.hsq_g = take(sh * 4 * (size_t)tpad);
    L.total = o;
    L.pmax = (int)pmax;
    L.tpad = (int)tpad;
    return L;
}

// Shapes the W4A4 kernels cover: NVFP4 banks, group 16 or 32, every K a whole number of
// 256-element stages and every row count a whole number of 128-row tiles (down: 256).
static ft_status check_w4a4(const Geometry &G)
{
    if (G.fmt != FT_FORMAT_NVFP4) return fail(FT_ERR_UNSUPPORTED, "W4A4 needs NVFP4 weight banks");
    if (G.H % 256 || !w4a4_shape_ok(G.H, G.Il) || !w4a4_shape_ok(G.Il, G.H) ||
        (G.Is && (!w4a4_shape_ok(G.H, G.Isl) || !w4a4_shape_ok(G.Isl, G.H))))
        return fail(FT_ERR_UNSUPPORTED,
                    "W4A4 needs hidden and the rank's intermediate sizes to be multiples of 256 (got H %d, I_l %d, I_sl %d)",
                    G.H, G.Il, G.Isl);
    return FT_OK;
}

// K-split for a merged lean launch: the smallest of 1, 2, 4, 8 that gives at least two
// CTA units per SM, as long as every K range stays a multiple of 128.
static int fast_ksplit(int blocks, int units_per_block_ks1, int K0, int K1 = 0)
{
    if (!K1) K1 = K0;
    int ks = 1;
    while (ks < 8 && blocks * units_per_block_ks1 * ks < 2 * sm_count() && (K0 / (2 * ks)) % 128 == 0 &&
           (K1 / (2 * ks)) % 128 == 0)
        ks *= 2;
    return ks;
}

// K-split of the NVFP4 lean decode kernels: doubled while the doubled unit count still fits
// twice over the SMs and every warp keeps at least min_kw elements of K (down: at most
// cap). Measured on qwen36 (T = 1, 8) and the dsv4 shape (T = 1, 16): fewer, longer
// streams per warp beat more, shorter ones once the units cover the SMs.
static int decode_ksplit(int blocks, int units_per_block_ks1, int K0, int K1, int min_kw, int cap)
{
    int ks = 1;
    while (ks < cap && blocks * units_per_block_ks1 * ks * 2 <= 2 * sm_count() && (K0 / (2 * ks)) % 128 == 0 &&
           (K1 / (2 * ks)) % 128 == 0 && K0 / (2 * ks) >= min_kw && K1 / (2 * ks) >= min_kw)
        ks *= 2;
    return ks;
}

// Generic register-fed launch for one problem (shapes the lean kernels do not cover).
// `rows` = I_l (gated) or H (down); max_blocks bounds the blocks.
static cudaError_t run_gemv(GemvParams p, bool gated, int max_blocks, int rows, cudaStream_t s)
{
    auto cdiv = [](int a, int b) { return (a + b - 1) / b; };
    const int ks2 = gemv_ksplit(max_blocks, cdiv(rows, 128), p.K);
    p.n_tiles = cdiv(rows, 16 * (8 / ks2));
    return gated ? launch_gemv_gated(p, ks2, max_blocks * p.n_tiles, s)
                 : launch_gemv_down(p, ks2, max_blocks * p.n_tiles, s);
}

static bool banks_ok(const ft_moe_banks *b, int fmt = FT_FORMAT_NVFP4)
{
    if (!b) return false;
    for (int i = 0; i < FT_NBANKS; ++i) {
        const bool none = fmt == FT_FORMAT_FP8_BLOCK && (i == FT_GU_GLOBAL || i == FT_DN_GLOBAL);
        if (none) continue;  // fp8_block has no globals: the pointer is not read
        if (!b->p[i] || !aligned(b->p[i], 16)) return false;
    }
    return true;
}

}  // namespace ftmoe

using namespace ftmoe;

extern "C" {

const char *ft_last_error(void) { return g_err; }

ft_status ft_moe_set_stage_events(void *const *events)
{
    if (!events) {
        g_stage_armed = false;
        return ok();
    }
    for (int i = 0; i <= FT_NSTAGES; ++i) {
        if (!events[i]) return fail(FT_ERR_INVALID_ARG, "stage event %d is NULL", i);
        g_stage_events[i] = static_cast<cudaEvent_t>(events[i]);
    }
    g_stage_armed = true;
    return ok();
}

int64_t ft_moe_launch_count(void) { return g_launches; }

ft_status ft_moe_debug_inject_stall(uint64_t wait_limit_ns, int32_t skip_producer)
{
    if (skip_producer != 0 && skip_producer != 1) return fail(FT_ERR_INVALID_ARG, "skip_producer must be 0 or 1");
    if (wait_limit_ns != 0 && (wait_limit_ns < 1000000ull || wait_limit_ns > kWaitNsMax))
        return fail(FT_ERR_INVALID_ARG, "wait limit must be 0 (default) or within [1 ms, 2 s]");
    g_stall_wait_ns = wait_limit_ns;
    g_stall_skip = skip_producer;
    g_stall_armed = true;
    return ok();
}

ft_status ft_moe_layout(const ft_moe_config *cfg, int32_t shared, ft_bank_spec out[FT_NBANKS])
{
    Geometry G;
    ft_status st = check_config(cfg, G);
    if (st) return st;
    if (!out) return fail(FT_ERR_INVALID_ARG, "out is NULL");
    if (shared != 0 && shared != 1) return fail(FT_ERR_INVALID_ARG, "shared must be 0 or 1");
    if (shared && G.Is == 0) return fail(FT_ERR_UNSUPPORTED, "layer has no shared expert");
    bank_specs(G, shared, out);
    return ok();
}

ft_status ft_moe_workspace_size(const ft_moe_config *cfg, int32_t T, size_t *bytes)
{
    Geometry G;
    ft_status st = check_config(cfg, G);
    if (st) return st;
    if (!bytes) return fail(FT_ERR_INVALID_ARG, "bytes is NULL");
    if (T < 0 || T > (1 << 20)) return fail(FT_ERR_UNSUPPORTED, "T must be in [0, 2^20]");
    *bytes = ws_layout(G, T).total;
    return ok();
}

static bool overlaps(const void *a, size_t na, const void *b, size_t nb)
{
    uintptr_t x = reinterpret_cast<uintptr_t>(a), y = reinterpret_cast<uintptr_t>(b);
    return x < y + nb && y < x + na;
}

ft_status ft_moe_pack(const ft_moe_config *cfg, int32_t shared, const ft_moe_pieces *src, const ft_moe_banks *dst,
                      void *stream)
{
    FT_NVTX_RANGE("ft_moe_pack");
    Geometry G;
    ft_status st = check_config(cfg, G);
    if (st) return st;
    if (shared != 0 && shared != 1) return fail(FT_ERR_INVALID_ARG, "shared must be 0 or 1");
    if (shared && G.Is == 0) return fail(FT_ERR_UNSUPPORTED, "layer has no shared expert");
    const bool fp8 = G.fmt == FT_FORMAT_FP8_BLOCK;
    if (!src || !src->gate || !src->gate_scale || !src->up || !src->up_scale || !src->down || !src->down_scale ||
        (!fp8 && (!src->gate_global || !src->up_global || !src->down_global)))
        return fail(FT_ERR_INVALID_ARG, "a source piece is NULL");
    if (!banks_ok(dst, G.fmt))
        return fail(FT_ERR_INVALID_ARG, "destination banks must be non-NULL and 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    // the rank's range [b0, b0 + Il) of the intermediate dimension (even or explicit split)
    const size_t E = shared ? 1 : G.E, I = shared ? G.Is : G.I, Il = shared ? G.Isl : G.Il, H = G.H, g = G.g;
    const size_t b0 = shared ? G.sb : G.rb;
    ft_bank_spec specs[FT_NBANKS];
    bank_specs(G, shared, specs);
    // fp8_block: one code byte per weight, fp32 scale_inv per 128 x 128 block, no globals
    const size_t sblk = (I / 128) * (H / 128) * 4;
    const size_t src_bytes[9] = {fp8 ? E * I * H : E * I * H / 2, fp8 ? E * sblk : E * I * H / g, fp8 ? 0 : E * I * 4,
                                 fp8 ? E * I * H : E * I * H / 2, fp8 ? E * sblk : E * I * H / g, fp8 ? 0 : E * I * 4,
                                 fp8 ? E * H * I : E * H * I / 2, fp8 ? E * sblk : E * H * I / g, fp8 ? 0 : E * H * 4};
    const void *srcs[9] = {src->gate, src->gate_scale, src->gate_global, src->up, src->up_scale,
                           src->up_global, src->down, src->down_scale, src->down_global};
    if (src->on_device) {
        for (int i = 0; i < 9; ++i)
            for (int j = 0; j < FT_NBANKS; ++j)
                if (overlaps(srcs[i], src_bytes[i], dst->p[j], (size_t)specs[j].bytes))
                    return fail(FT_ERR_INVALID_ARG, "pack destination overlaps its source");
    }
    struct Copy { const void *s; size_t sp; void *d; size_t dp; size_t w; size_t h; };
    auto u8 = [](const void *p, size_t off) { return static_cast<const uint8_t *>(p) + off; };
    auto w8 = [](void *p, size_t off) { return static_cast<uint8_t *>(p) + off; };
    const size_t hb = H / 128, lb = Il / 128, ib = I / 128;
    const Copy copies_fp8[6] = {
        {u8(src->gate, b0 * H), I * H, w8(dst->p[FT_GU], 0), 2 * Il * H, Il * H, E},
        {u8(src->up, b0 * H), I * H, w8(dst->p[FT_GU], Il * H), 2 * Il * H, Il * H, E},
        {u8(src->gate_scale, (b0 / 128) * hb * 4), ib * hb * 4, w8(dst->p[FT_GU_SCALE], 0), 2 * lb * hb * 4,
         lb * hb * 4, E},
        {u8(src->up_scale, (b0 / 128) * hb * 4), ib * hb * 4, w8(dst->p[FT_GU_SCALE], lb * hb * 4), 2 * lb * hb * 4,
         lb * hb * 4, E},
        {u8(src->down, b0), I, w8(dst->p[FT_DN], 0), Il, Il, E * H},
        {u8(src->down_scale, (b0 / 128) * 4), ib * 4, w8(dst->p[FT_DN_SCALE], 0), lb * 4, lb * 4, E * hb},
    };
    const Copy copies[9] = {
        {u8(src->gate, b0 * H / 2), I * H / 2, w8(dst->p[FT_GU], 0), 2 * Il * H / 2, Il * H / 2, E},
        {u8(src->up, b0 * H / 2), I * H / 2, w8(dst->p[FT_GU], Il * H / 2), 2 * Il * H / 2, Il * H / 2, E},
        {u8(src->gate_scale, b0 * H / g), I * H / g, w8(dst->p[FT_GU_SCALE], 0), 2 * Il * H / g, Il * H / g, E},
        {u8(src->up_scale, b0 * H / g), I * H / g, w8(dst->p[FT_GU_SCALE], Il * H / g), 2 * Il * H / g,
         Il * H / g, E},
        {u8(src->gate_global, b0 * 4), I * 4, w8(dst->p[FT_GU_GLOBAL], 0), 2 * Il * 4, Il * 4, E},
        {u8(src->up_global, b0 * 4), I * 4, w8(dst->p[FT_GU_GLOBAL], Il * 4), 2 * Il * 4, Il * 4, E},
        {u8(src->down, b0 / 2), I / 2, w8(dst->p[FT_DN], 0), Il / 2, Il / 2, E * H},
        {u8(src->down_scale, b0 / g), I / g, w8(dst->p[FT_DN_SCALE], 0), Il / g, Il / g, E * H},
        {u8(src->down_global, 0), E * H * 4, w8(dst->p[FT_DN_GLOBAL], 0), E * H * 4, E * H * 4, 1},
    };
    const Copy *list = fp8 ? copies_fp8 : copies;
    const int n_copies = fp8 ? 6 : 9;
    for (int ci = 0; ci < n_copies; ++ci) {
        const Copy &c = list[ci];
        cudaError_t e;
        if (src->on_device)
            e = launch_pack_copy2d(static_cast<const uint8_t *>(c.s), c.sp, static_cast<uint8_t *>(c.d), c.dp, c.w,
                                   c.h, s);
        else
            e = cudaMemcpy2DAsync(c.d, c.dp, c.s, c.sp, c.w, c.h, cudaMemcpyHostToDevice, s);
        if (e != cudaSuccess) return cuda_fail(e, "ft_moe_pack copy");
    }
    return ok();
}

ft_status ft_moe_route(const float *logits, int32_t T, int32_t E, int32_t k, int32_t *topk_ids, float *topk_w,
                       void *stream)
{
    FT_NVTX_RANGE("ft_moe_route");
    if (T < 0 || E <= 0 || k <= 0) return fail(FT_ERR_INVALID_ARG, "need T >= 0, E > 0, k > 0");
    if (E > 1024 || k > 32 || k > E) return fail(FT_ERR_UNSUPPORTED, "need k <= 32, k <= E <= 1024");
    if (T == 0) return ok();
    if (!logits || !topk_ids || !topk_w || !aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
        return fail(FT_ERR_INVALID_ARG, "route pointers must be non-NULL and 4-byte aligned");
    cudaError_t e = launch_route(logits, T, E, k, topk_ids, topk_w, static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    return ok();
}

ft_status ft_moe_route_gemm(const void *x, int32_t T, int32_t H, const void *w_router, int32_t E, int32_t k,
                            float *logits, int32_t *topk_ids, float *topk_w, void *stream)
{
    FT_NVTX_RANGE("ft_moe_route_gemm");
    if (T < 0 || E <= 0 || k <= 0 || H <= 0) return fail(FT_ERR_INVALID_ARG, "need T >= 0, H, E, k > 0");
    if (H % 32) return fail(FT_ERR_INVALID_ARG, "need H a multiple of 32");
    if (E > 1024 || k > 32 || k > E) return fail(FT_ERR_UNSUPPORTED, "need k <= 32, k <= E <= 1024");
    if (T == 0) return ok();
    if (!x || !w_router || !logits || !topk_ids || !topk_w || !aligned(x, 16) || !aligned(w_router, 16) ||
        !aligned(logits, 4) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
        return fail(FT_ERR_INVALID_ARG, "router pointers must be non-NULL; x and w_router 16-byte aligned");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = launch_router_gemm(static_cast<const uint16_t *>(x), static_cast<const uint16_t *>(w_router), T, H,
                                       E, logits, s);
    if (e != cudaSuccess) return cuda_fail(e, "router GEMM launch");
    e = launch_route(logits, T, E, k, topk_ids, topk_w, s);
    if (e != cudaSuccess) return cuda_fail(e, "route launch");
    return ok();
}

ft_status ft_moe_align_workspace_size(int32_t T, int32_t k, int32_t E, size_t *bytes)
{
    if (!bytes || T < 0 || k <= 0 || E <= 0) return fail(FT_ERR_INVALID_ARG, "bad align arguments");
    if (E > 1024 || T > (1 << 20) || k > 32) return fail(FT_ERR_UNSUPPORTED, "align limits exceeded");
    *bytes = 256 + align_scratch_bytes(T * k, E);
    return ok();
}

ft_status ft_moe_align(const int32_t *topk_ids, int32_t T, int32_t k, int32_t E, int32_t block, int32_t *sorted_slot,
                       int32_t *block_expert, int32_t *expert_off, int32_t *n_padded, void *workspace,
                       size_t workspace_bytes, void *stream)
{
    FT_NVTX_RANGE("ft_moe_align");
    if (T < 0 || k <= 0 || E <= 0 || block < 1 || block > 1024)
        return fail(FT_ERR_INVALID_ARG, "need T >= 0, k > 0, E > 0, 1 <= block <= 1024");
    if (E > 1024 || T > (1 << 20) || k > 32) return fail(FT_ERR_UNSUPPORTED, "align limits exceeded");
    if (!sorted_slot || !block_expert || !expert_off || !n_padded || !workspace || (T > 0 && !topk_ids))
        return fail(FT_ERR_INVALID_ARG, "align pointers must be non-NULL");
    if (!aligned(workspace, 256)) return fail(FT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    size_t need = 256 + align_scratch_bytes(T * k, E);
    if (workspace_bytes < need) return fail(FT_ERR_WORKSPACE, "align workspace needs %zu bytes", need);
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int *status = static_cast<int *>(workspace);
    cudaError_t e = cudaMemsetAsync(status, 0, sizeof(int), s);
    if (e == cudaSuccess)
        e = launch_align(topk_ids, T, k, E, block, sorted_slot, block_expert, expert_off, n_padded, status,
                         static_cast<char *>(workspace) + 256, s);
    if (e != cudaSuccess) return cuda_fail(e, "align launch");
    return ok();
}

ft_status ft_moe_forward(const ft_moe_config *cfg, const ft_moe_banks *routed, const ft_moe_banks *shared,
                         const void *x, int32_t T, const int32_t *topk_ids, const float *topk_w, void *out,
                         int32_t out_dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    FT_NVTX_RANGE("ft_moe_forward");
    Geometry G;
    ft_status st = check_config(cfg, G);
    if (st) return st;
    if (T < 0 || T > (1 << 20)) return fail(FT_ERR_UNSUPPORTED, "T must be in [0, 2^20]");
    if (out_dtype != FT_DTYPE_BF16 && out_dtype != FT_DTYPE_F32)
        return fail(FT_ERR_INVALID_ARG, "out_dtype must be FT_DTYPE_BF16 or FT_DTYPE_F32");
    if (!banks_ok(routed, G.fmt))
        return fail(FT_ERR_INVALID_ARG, "routed banks must be non-NULL and 16-byte aligned");
    if (G.Is > 0 && !banks_ok(shared, G.fmt))
        return fail(FT_ERR_INVALID_ARG, "shared banks required (shared_intermediate > 0), 16-byte aligned");
    if (G.Is == 0 && shared) return fail(FT_ERR_INVALID_ARG, "shared banks given but shared_intermediate is 0");
    if (T == 0) return ok();
    if (!x || !topk_ids || !topk_w || !out || !workspace)
        return fail(FT_ERR_INVALID_ARG, "x, topk_ids, topk_w, out and workspace must be non-NULL");
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
        return fail(FT_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    if (!aligned(workspace, 256)) return fail(FT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const WsLayout L = ws_layout(G, T);
    if (workspace_bytes < L.total) return fail(FT_ERR_WORKSPACE, "workspace needs %zu bytes", L.total);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    int *status = reinterpret_cast<int *>(ws + L.status);
    int *sorted = reinterpret_cast<int *>(ws + L.sorted);
    int *bexp = reinterpret_cast<int *>(ws + L.block_expert);
    int *eoff = reinterpret_cast<int *>(ws + L.expert_off);
    int *npad = reinterpret_cast<int *>(ws + L.npad);
    uint16_t *h = reinterpret_cast<uint16_t *>(ws + L.h);
    uint16_t *h_sh = reinterpret_cast<uint16_t *>(ws + L.h_sh);
    float *y = reinterpret_cast<float *>(ws + L.y);
    float *y_sh = reinterpret_cast<float *>(ws + L.y_sh);
    const int n_slots = T * G.k;

    struct Disarm {
        ~Disarm()
        {
            g_stage_armed = false;
            g_stall_armed = g_stall_active = false;
        }
    } disarm_on_return;
    g_stall_active = g_stall_armed;
    cudaError_t e;
    if ((e = stage_mark(FT_STAGE_ALIGN, s)) != cudaSuccess) return cuda_fail(e, "stage event");

    auto cdiv = [](int a, int b) { return (a + b - 1) / b; };
    const bool fp8 = G.fmt == FT_FORMAT_FP8_BLOCK;
    const bool tc_path = fp8 ? use_tc_fp8(G, T) : use_tc(G, T);
    if (fp8 && !tc_path) {
        // ---------------------------------------------------------------- fp8_block experts
        // register-fed grouped GEMV for every batch size: align, gate_up (+ shared), down
        // (+ shared) with the routing weight, then the ordered combine
        e = launch_align(topk_ids, T, G.k, G.E, kGemvBlock, sorted, bexp, eoff, npad, status, ws + L.scratch, s,
                         status, L.zero_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "align launch");
        const int max_blocks = (int)(((int64_t)n_slots + (n_slots < G.E ? n_slots : G.E) * (kGemvBlock - 1)) /
                                     kGemvBlock);
        const int tpad = cdiv(T, kGemvBlock);
        auto problem = [&](const ft_moe_banks *b, bool gated, int E, int Il) {
            GemvParams p = {};
            p.codes = static_cast<const uint8_t *>(b->p[gated ? FT_GU : FT_DN]);
            p.sinv = static_cast<const float *>(b->p[gated ? FT_GU_SCALE : FT_DN_SCALE]);
            p.R = gated ? 2 * Il : G.H;
            p.K = gated ? G.H : Il;
            p.e_codes = (int64_t)p.R * p.K;
            p.e_sinv = (int64_t)(p.R / 128) * (p.K / 128);
            p.group = 128;
            p.up_off = gated ? Il : 0;
            p.num_experts = E;
            p.status = status;
            return p;
        };
        GemvParams gu = problem(routed, true, G.E, G.Il), dn = problem(routed, false, G.E, G.Il);
        gu.act = static_cast<const uint16_t *>(x);
        gu.h_out = h; gu.h_ld = G.Il;
        dn.act = h; dn.y_out = y; dn.route_w = topk_w;
        for (GemvParams *p : {&gu, &dn}) {
            p->n_pos_dev = npad; p->sorted_slot = sorted; p->block_expert = bexp;
            p->n_slots = n_slots; p->top_k = G.k;
        }
        GemvParams gu_sh = {}, dn_sh = {};
        if (G.Is) {
            gu_sh = problem(shared, true, 1, G.Isl);
            dn_sh = problem(shared, false, 1, G.Isl);
            gu_sh.act = static_cast<const uint16_t *>(x);
            gu_sh.h_out = h_sh; gu_sh.h_ld = G.Isl;
            dn_sh.act = h_sh; dn_sh.y_out = y_sh;
            for (GemvParams *p : {&gu_sh, &dn_sh}) {
                p->n_pos_static = T; p->n_slots = T; p->top_k = 1;
            }
        }
        const int kmax_l = G.Il > G.Isl ? G.Il : G.Isl;
        int ks_gu = fast_ksplit(max_blocks + (G.Is ? tpad : 0), cdiv(kmax_l, 16 * 8), G.H);
        int ks_dn = fast_ksplit(max_blocks + (G.Is ? tpad : 0), cdiv(G.H, 32 * 8), G.Il, G.Is ? G.Isl : G.Il);
        if (!gemv_fp8_ok(G.H, ks_gu)) ks_gu = 1;
        if (!gemv_fp8_ok(G.Il, ks_dn) || (G.Is && !gemv_fp8_ok(G.Isl, ks_dn))) ks_dn = 1;
        FastLaunch F = {};
        F.prob[0] = gu;
        F.prob[0].n_tiles = cdiv(G.Il, 16 * (8 / ks_gu));
        F.nprob = 1;
        if (G.Is) {
            F.prob[1] = gu_sh;
            F.prob[1].n_tiles = cdiv(G.Isl, 16 * (8 / ks_gu));
            F.nprob = 2;
        }
        // K split evenly over the CTAs (whole 128-K blocks; with ks_gu = 1)
        F.split_part = reinterpret_cast<float *>(ws + L.split_part);
        F.split_cnt = reinterpret_cast<int *>(ws + L.split_cnt);
        if ((e = stage_mark(FT_STAGE_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        int max_units = max_blocks * F.prob[0].n_tiles + (G.Is ? tpad * F.prob[1].n_tiles : 0);
        if ((e = launch_gemv_fp8(F, true, ks_gu, max_units, s)) != cudaSuccess) return cuda_fail(e, "gate_up launch");
        if ((e = stage_mark(FT_STAGE_SHARED_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        FastLaunch D = {};
        D.prob[0] = dn;
        D.prob[0].n_tiles = cdiv(G.H, 32 * (8 / ks_dn));
        D.nprob = 1;
        if (G.Is) {
            D.prob[1] = dn_sh;
            D.prob[1].n_tiles = D.prob[0].n_tiles;
            D.nprob = 2;
        }
        if ((e = stage_mark(FT_STAGE_DOWN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        max_units = (max_blocks + (G.Is ? tpad : 0)) * D.prob[0].n_tiles;
        if ((e = launch_gemv_fp8(D, false, ks_dn, max_units, s)) != cudaSuccess) return cuda_fail(e, "down launch");
        if ((e = stage_mark(FT_STAGE_SHARED_DOWN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        if ((e = stage_mark(FT_STAGE_COMBINE, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        e = launch_combine(y, G.Is ? y_sh : nullptr, T, G.k, G.H, out, out_dtype, s);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
        if ((e = stage_mark(FT_NSTAGES, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        return ok();
    }
    if (tc_path) {
        // ---------------------------------------------------------------- tensor-core path
        // fp8_block banks: codes of one byte, scale_inv per 128 x 128 block, no globals
        auto fp8_fields = [&](TcParams &t, const ft_moe_banks *b, bool gate_up, int il) {
            if (!fp8) return;
            t.fp8 = 1;
            t.sinv = static_cast<const float *>(b->p[gate_up ? FT_GU_SCALE : FT_DN_SCALE]);
            t.e_sinv = gate_up ? (int64_t)(2 * il / 128) * (G.H / 128) : (int64_t)(G.H / 128) * (il / 128);
            t.scales = nullptr;
            t.glob = nullptr;
        };
        e = launch_align(topk_ids, T, G.k, G.E, kTcBlock, sorted, bexp, eoff, npad, status, ws + L.scratch, s,
                         status, L.zero_bytes);
        if (e != cudaSuccess) return cuda_fail(e, "align launch");
        const int max_blocks_tc = L.pmax / kTcBlock, tpad_tc = cdiv(T, kTcBlock);
        TcParams gp = {};
        gp.scales = static_cast<const uint8_t *>(routed->p[FT_GU_SCALE]);
        gp.glob = static_cast<const float *>(routed->p[FT_GU_GLOBAL]);
        gp.R = 2 * G.Il; gp.K = G.H; gp.group = G.g; gp.up_off = G.Il; gp.n_mtiles = G.Il / 128;
        gp.n_pos_dev = npad; gp.sorted_slot = sorted; gp.block_expert = bexp; gp.n_slots = n_slots; gp.top_k = G.k;
        gp.num_experts = G.E;
        gp.h_out = h; gp.h_ld = G.Il; gp.status = status;
        fp8_fields(gp, routed, true, G.Il);
        if ((e = stage_mark(FT_STAGE_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        auto f16buf = [&](size_t off) { return reinterpret_cast<uint16_t *>(ws + off); };
        auto f32buf = [&](size_t off) { return reinterpret_cast<float *>(ws + off); };
        const uint16_t *xb = static_cast<const uint16_t *>(x);
        e = launch_rows_to_f16(xb, G.H, sorted, npad, 0, n_slots, G.k, L.pmax, f16buf(L.xs), f32buf(L.xs_scale), s, status);
        if (e != cudaSuccess) return cuda_fail(e, "row conversion launch");
        gp.act_scale = f32buf(L.xs_scale);
        // routed and shared expert in one launch (units of the routed experts first)
        TcParams gprob[2] = {gp, gp};
        TcOperands gops[2] = {{routed->p[FT_GU], (int64_t)G.E * 2 * G.Il, f16buf(L.xs), L.pmax}, {}};
        int n_gprob = 1, gunits = max_blocks_tc * gp.n_mtiles;
        const int tp = tpad_tc * kTcBlock;
        if (G.Is) {
            TcParams sp = gp;
            sp.scales = static_cast<const uint8_t *>(shared->p[FT_GU_SCALE]);
            sp.glob = static_cast<const float *>(shared->p[FT_GU_GLOBAL]);
            sp.R = 2 * G.Isl; sp.up_off = G.Isl; sp.n_mtiles = G.Isl / 128;
            sp.n_pos_dev = nullptr; sp.n_pos_static = T; sp.sorted_slot = nullptr; sp.block_expert = nullptr;
            sp.n_slots = T; sp.top_k = 1; sp.num_experts = 1; sp.h_out = h_sh; sp.h_ld = G.Isl;
            sp.act_scale = f32buf(L.x16_scale);
            fp8_fields(sp, shared, true, G.Isl);
            e = launch_rows_to_f16(xb, G.H, nullptr, nullptr, tp, T, 1, tp, f16buf(L.x16), f32buf(L.x16_scale), s, status);
            if (e != cudaSuccess) return cuda_fail(e, "row conversion launch");
            gprob[1] = sp;
            gops[1] = {shared->p[FT_GU], 2 * (int64_t)G.Isl, f16buf(L.x16), tp};
            n_gprob = 2;
            gunits += tpad_tc * sp.n_mtiles;
        }
        if ((e = launch_tc_gemm(gprob, gops, n_gprob, true, gunits, s)) != cudaSuccess)
            return cuda_fail(e, "gate_up launch");
        if ((e = stage_mark(FT_STAGE_SHARED_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        if ((e = stage_mark(FT_STAGE_DOWN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        TcParams dp = {};
        dp.scales = static_cast<const uint8_t *>(routed->p[FT_DN_SCALE]);
        dp.glob = static_cast<const float *>(routed->p[FT_DN_GLOBAL]);
        dp.R = G.H; dp.K = G.Il; dp.group = G.g; dp.up_off = 0; dp.n_mtiles = G.H / 256;
        dp.n_pos_dev = npad; dp.sorted_slot = sorted; dp.block_expert = bexp; dp.n_slots = n_slots; dp.top_k = G.k;
        dp.num_experts = G.E;
        dp.y_out = y; dp.y_ld = G.H; dp.route_w = topk_w; dp.status = status;
        dp.act_scale = f32buf(L.h16_scale);
        fp8_fields(dp, routed, false, G.Il);
        // h rows are already in sorted-position order: convert them in place of a gather
        e = launch_rows_to_f16(h, G.Il, nullptr, npad, 0, L.pmax, 1, L.pmax, f16buf(L.h16), f32buf(L.h16_scale), s, status);
        if (e != cudaSuccess) return cuda_fail(e, "row conversion launch");
        TcParams dprob[2] = {dp, dp};
        TcOperands dops[2] = {{routed->p[FT_DN], (int64_t)G.E * G.H, f16buf(L.h16), L.pmax}, {}};
        int n_dprob = 1, dunits = max_blocks_tc * dp.n_mtiles;
        if (G.Is) {
            TcParams sd = dp;
            sd.scales = static_cast<const uint8_t *>(shared->p[FT_DN_SCALE]);
            sd.glob = static_cast<const float *>(shared->p[FT_DN_GLOBAL]);
            sd.K = G.Isl; sd.n_pos_dev = nullptr; sd.n_pos_static = T; sd.sorted_slot = nullptr;
            sd.block_expert = nullptr; sd.n_slots = T; sd.top_k = 1; sd.num_experts = 1; sd.y_out = y_sh; sd.route_w = nullptr;
            sd.act_scale = f32buf(L.hsh16_scale);
            fp8_fields(sd, shared, false, G.Isl);
            e = launch_rows_to_f16(h_sh, G.Isl, nullptr, nullptr, tp, T, 1, tp, f16buf(L.hsh16),
                                   f32buf(L.hsh16_scale), s, status);
            if (e != cudaSuccess) return cuda_fail(e, "row conversion launch");
            dprob[1] = sd;
            dops[1] = {shared->p[FT_DN], G.H, f16buf(L.hsh16), tp};
            n_dprob = 2;
            dunits += tpad_tc * sd.n_mtiles;
        }
        if ((e = launch_tc_gemm(dprob, dops, n_dprob, false, dunits, s)) != cudaSuccess)
            return cuda_fail(e, "down launch");
        if ((e = stage_mark(FT_STAGE_SHARED_DOWN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        if ((e = stage_mark(FT_STAGE_COMBINE, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        e = launch_combine(y, G.Is ? y_sh : nullptr, T, G.k, G.H, out, out_dtype, s);
        if (e != cudaSuccess) return cuda_fail(e, "combine launch");
        if ((e = stage_mark(FT_NSTAGES, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        return ok();
    }

    e = launch_align(topk_ids, T, G.k, G.E, kGemvBlock, sorted, bexp, eoff, npad, status, ws + L.scratch, s,
                         status, L.zero_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "align launch");
    const int max_blocks = (int)(((int64_t)n_slots + (n_slots < G.E ? n_slots : G.E) * (kGemvBlock - 1)) / kGemvBlock);
    const int tpad = (T + kGemvBlock - 1) / kGemvBlock;

    // The four problems of the decode regime: routed and shared gate_up (+ SwiGLU into
    // h / h_sh), routed and shared down (+ routing weight into y / y_sh).
    GemvParams gu = {}, gu_sh = {}, dn = {}, dn_sh = {};
    gu.codes = static_cast<const uint8_t *>(routed->p[FT_GU]);
    gu.scales = static_cast<const uint8_t *>(routed->p[FT_GU_SCALE]);
    gu.glob = static_cast<const float *>(routed->p[FT_GU_GLOBAL]);
    gu.e_codes = (int64_t)G.Il * G.H; gu.e_scales = (int64_t)2 * G.Il * G.H / G.g; gu.e_glob = 2 * G.Il;
    gu.R = 2 * G.Il; gu.K = G.H; gu.group = G.g; gu.up_off = G.Il;
    gu.act = static_cast<const uint16_t *>(x);
    gu.n_pos_dev = npad; gu.sorted_slot = sorted; gu.block_expert = bexp;
    gu.n_slots = n_slots; gu.top_k = G.k; gu.num_experts = G.E; gu.status = status;
    gu.h_out = h; gu.h_ld = G.Il;
    dn.codes = static_cast<const uint8_t *>(routed->p[FT_DN]);
    dn.scales = static_cast<const uint8_t *>(routed->p[FT_DN_SCALE]);
    dn.glob = static_cast<const float *>(routed->p[FT_DN_GLOBAL]);
    dn.e_codes = (int64_t)G.H * G.Il / 2; dn.e_scales = (int64_t)G.H * G.Il / G.g; dn.e_glob = G.H;
    dn.R = G.H; dn.K = G.Il; dn.group = G.g; dn.act = h;
    dn.n_pos_dev = npad; dn.sorted_slot = sorted; dn.block_expert = bexp;
    dn.n_slots = n_slots; dn.top_k = G.k; dn.num_experts = G.E; dn.status = status;
    dn.y_out = y; dn.route_w = topk_w;
    if (G.Is) {
        gu_sh = gu;
        gu_sh.codes = static_cast<const uint8_t *>(shared->p[FT_GU]);
        gu_sh.scales = static_cast<const uint8_t *>(shared->p[FT_GU_SCALE]);
        gu_sh.glob = static_cast<const float *>(shared->p[FT_GU_GLOBAL]);
        gu_sh.e_codes = (int64_t)G.Isl * G.H; gu_sh.e_scales = (int64_t)2 * G.Isl * G.H / G.g;
        gu_sh.e_glob = 2 * G.Isl; gu_sh.R = 2 * G.Isl; gu_sh.up_off = G.Isl;
        gu_sh.n_pos_dev = nullptr; gu_sh.n_pos_static = T; gu_sh.sorted_slot = nullptr;
        gu_sh.block_expert = nullptr; gu_sh.n_slots = T; gu_sh.top_k = 1; gu_sh.num_experts = 1;
        gu_sh.h_out = h_sh; gu_sh.h_ld = G.Isl;
        dn_sh = dn;
        dn_sh.codes = static_cast<const uint8_t *>(shared->p[FT_DN]);
        dn_sh.scales = static_cast<const uint8_t *>(shared->p[FT_DN_SCALE]);
        dn_sh.glob = static_cast<const float *>(shared->p[FT_DN_GLOBAL]);
        dn_sh.e_codes = (int64_t)G.H * G.Isl / 2; dn_sh.e_scales = (int64_t)G.H * G.Isl / G.g;
        dn_sh.K = G.Isl; dn_sh.act = h_sh;
        dn_sh.n_pos_dev = nullptr; dn_sh.n_pos_static = T; dn_sh.sorted_slot = nullptr;
        dn_sh.block_expert = nullptr; dn_sh.n_slots = T; dn_sh.top_k = 1; dn_sh.num_experts = 1;
        dn_sh.y_out = y_sh; dn_sh.route_w = nullptr;
    }
    // after the down stage: the combine, out[t] = sum_j y[t k + j] (+ y_sh[t]), in that order
    auto combine = [&]() -> cudaError_t {
        cudaError_t err;
        if ((err = stage_mark(FT_STAGE_SHARED_DOWN, s)) != cudaSuccess) return err;
        if ((err = stage_mark(FT_STAGE_COMBINE, s)) != cudaSuccess) return err;
        if ((err = launch_combine(y, G.Is ? y_sh : nullptr, T, G.k, G.H, out, out_dtype, s)) != cudaSuccess) return err;
        return stage_mark(FT_NSTAGES, s);
    };

    // Lean register-fed kernels: gate_up (+ shared expert), down (+ shared expert) and the
    // ordered combine, fused into one persistent launch for small batches.
    const int ks_gu = decode_ksplit(max_blocks + (G.Is ? tpad : 0), cdiv(G.Il > G.Isl ? G.Il : G.Isl, 16 * 8), G.H,
                                    G.H, 512, 8);
    const int ks_dn = decode_ksplit(max_blocks + (G.Is ? tpad : 0), cdiv(G.H, 32 * 8), G.Il, G.Is ? G.Isl : G.Il,
                                    256, 2);
    if (gemv_fast_ok(G.H, G.g, ks_gu, 2 * (G.Il > G.Isl ? G.Il : G.Isl)) && gemv_fast_ok(G.Il, G.g, ks_dn, G.H) &&
        (!G.Is || gemv_fast_ok(G.Isl, G.g, ks_dn, G.H))) {
        FusedLaunch FL = {};
        FastLaunch &F = FL.gu;
        F.prob[0] = gu;
        F.prob[0].n_tiles = cdiv(G.Il, 16 * (8 / ks_gu));
        F.nprob = 1;
        if (G.Is) {
            F.prob[1] = gu_sh;
            F.prob[1].n_tiles = cdiv(G.Isl, 16 * (8 / ks_gu));
            F.nprob = 2;
        }
        F.split_part = reinterpret_cast<float *>(ws + L.split_part);
        F.split_cnt = reinterpret_cast<int *>(ws + L.split_cnt);
        FastLaunch &D = FL.dn;
        D.prob[0] = dn;
        D.prob[0].n_tiles = cdiv(G.H, 32 * (8 / ks_dn));
        D.nprob = 1;
        if (G.Is) {
            D.prob[1] = dn_sh;
            D.prob[1].n_tiles = D.prob[0].n_tiles;
            D.nprob = 2;
        }
        // down units are short (I_l / 128 steps): splitting them costs more than it balances
        D.split_part = nullptr;
        D.split_cnt = nullptr;
        FL.gu_done = reinterpret_cast<int *>(ws + L.gu_done);
        FL.shared_base = max_blocks;
        FL.done = FL.gu_done + max_blocks + tpad;
        FL.y = y;
        FL.y_sh = G.Is ? y_sh : nullptr;
        FL.out = out;
        FL.out_dtype = out_dtype;
        FL.T = T;
        FL.k = G.k;
        FL.H = G.H;
        FL.status = status;
        injected_stall(&FL.wait_ns, &FL.skip_publish);
        const int gu_units = max_blocks * F.prob[0].n_tiles + (G.Is ? tpad * F.prob[1].n_tiles : 0);
        const int dn_units = (max_blocks + (G.Is ? tpad : 0)) * D.prob[0].n_tiles;
        if ((e = stage_mark(FT_STAGE_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        if (n_slots <= kFusedMaxSlots) {
            // small batches: one launch, the stages meeting through per-block counters
            if ((e = launch_gemv_fused(FL, ks_gu, ks_dn, gu_units > dn_units ? gu_units : dn_units, s)) !=
                cudaSuccess)
                return cuda_fail(e, "fused decode launch");
            for (int st_ = FT_STAGE_SHARED_GATE_UP; st_ <= FT_NSTAGES; ++st_)
                if ((e = stage_mark(st_, s)) != cudaSuccess) return cuda_fail(e, "stage event");
            return ok();
        }
        // larger batches: gate_up and down as their own launches (the kernel boundary costs
        // less than the cross-CTA waits), then the ordered combine
        if ((e = launch_gemv_fast(F, true, ks_gu, gu_units, s)) != cudaSuccess) return cuda_fail(e, "gate_up launch");
        if ((e = stage_mark(FT_STAGE_SHARED_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        if ((e = stage_mark(FT_STAGE_DOWN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
        if ((e = launch_gemv_fast(D, false, ks_dn, dn_units, s)) != cudaSuccess) return cuda_fail(e, "down launch");
        if ((e = combine()) != cudaSuccess) return cuda_fail(e, "combine launch");
        return ok();
    }

    // Generic kernels, one launch per problem, separate combine.
    if ((e = stage_mark(FT_STAGE_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    if ((e = run_gemv(gu, true, max_blocks, G.Il, s)) != cudaSuccess) return cuda_fail(e, "gate_up launch");
    if ((e = stage_mark(FT_STAGE_SHARED_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    if (G.Is && (e = run_gemv(gu_sh, true, tpad, G.Isl, s)) != cudaSuccess)
        return cuda_fail(e, "shared gate_up launch");
    if ((e = stage_mark(FT_STAGE_DOWN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    if ((e = run_gemv(dn, false, max_blocks, G.H, s)) != cudaSuccess) return cuda_fail(e, "down launch");
    if ((e = stage_mark(FT_STAGE_SHARED_DOWN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    if (G.Is && (e = run_gemv(dn_sh, false, tpad, G.H, s)) != cudaSuccess) return cuda_fail(e, "shared down launch");
    if ((e = stage_mark(FT_STAGE_COMBINE, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    e = launch_combine(y, G.Is ? y_sh : nullptr, T, G.k, G.H, out, out_dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    if ((e = stage_mark(FT_NSTAGES, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    return ok();
}

ft_status ft_moe_workspace_size_w4a4(const ft_moe_config *cfg, int32_t T, size_t *bytes)
{
    Geometry G;
    ft_status st = check_config(cfg, G);
    if (st) return st;
    if ((st = check_w4a4(G))) return st;
    if (!bytes) return fail(FT_ERR_INVALID_ARG, "bytes is NULL");
    if (T < 0 || T > (1 << 20)) return fail(FT_ERR_UNSUPPORTED, "T must be in [0, 2^20]");
    *bytes = ws_layout_w4a4(G, T).total;
    return ok();
}

ft_status ft_moe_forward_w4a4(const ft_moe_config *cfg, const ft_moe_banks *routed, const ft_moe_banks *shared,
                              const void *x, int32_t T, const int32_t *topk_ids, const float *topk_w, void *out,
                              int32_t out_dtype, void *workspace, size_t workspace_bytes, void *stream)
{
    FT_NVTX_RANGE("ft_moe_forward_w4a4");
    Geometry G;
    ft_status st = check_config(cfg, G);
    if (st) return st;
    if ((st = check_w4a4(G))) return st;
    if (T < 0 || T > (1 << 20)) return fail(FT_ERR_UNSUPPORTED, "T must be in [0, 2^20]");
    if (out_dtype != FT_DTYPE_BF16 && out_dtype != FT_DTYPE_F32)
        return fail(FT_ERR_INVALID_ARG, "out_dtype must be FT_DTYPE_BF16 or FT_DTYPE_F32");
    if (!banks_ok(routed)) return fail(FT_ERR_INVALID_ARG, "routed banks must be non-NULL and 16-byte aligned");
    if (G.Is > 0 && !banks_ok(shared))
        return fail(FT_ERR_INVALID_ARG, "shared banks required (shared_intermediate > 0), 16-byte aligned");
    if (G.Is == 0 && shared) return fail(FT_ERR_INVALID_ARG, "shared banks given but shared_intermediate is 0");
    if (T == 0) return ok();
    if (!x || !topk_ids || !topk_w || !out || !workspace)
        return fail(FT_ERR_INVALID_ARG, "x, topk_ids, topk_w, out and workspace must be non-NULL");
    if (!aligned(x, 16) || !aligned(out, 16) || !aligned(topk_ids, 4) || !aligned(topk_w, 4))
        return fail(FT_ERR_INVALID_ARG, "x and out must be 16-byte aligned");
    if (!aligned(workspace, 256)) return fail(FT_ERR_INVALID_ARG, "workspace must be 256-byte aligned");
    const WsW4 L = ws_layout_w4a4(G, T);
    if (workspace_bytes < L.total) return fail(FT_ERR_WORKSPACE, "workspace needs %zu bytes", L.total);

    cudaStream_t s = static_cast<cudaStream_t>(stream);
    char *ws = static_cast<char *>(workspace);
    auto at_i = [&](size_t off) { return reinterpret_cast<int *>(ws + off); };
    auto at_u8 = [&](size_t off) { return reinterpret_cast<uint8_t *>(ws + off); };
    auto at_f = [&](size_t off) { return reinterpret_cast<float *>(ws + off); };
    int *status = at_i(L.status), *sorted = at_i(L.sorted), *bexp = at_i(L.block_expert), *npad = at_i(L.npad);
    const int n_slots = T * G.k, tpad = L.tpad;
    struct Disarm {
        ~Disarm()
        {
            g_stage_armed = false;
            g_stall_armed = g_stall_active = false;
        }
    } disarm_on_return;
    g_stall_active = g_stall_armed;
    cudaError_t e;
    if ((e = stage_mark(FT_STAGE_ALIGN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    e = launch_align(topk_ids, T, G.k, G.E, kTcBlock, sorted, bexp, at_i(L.expert_off), npad, status,
                     ws + L.scratch, s, status, L.zero_bytes);
    if (e != cudaSuccess) return cuda_fail(e, "align launch");
    if ((e = stage_mark(FT_STAGE_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    // NVFP4 activations: x per expert-sorted position (routed) and per token (shared)
    e = launch_quant_nvfp4(x, false, G.H, sorted, npad, 0, n_slots, G.k, L.pmax, at_u8(L.xq_c), at_u8(L.xq_s),
                           at_f(L.xq_g), s, status);
    if (e == cudaSuccess && G.Is)
        e = launch_quant_nvfp4(x, false, G.H, nullptr, nullptr, tpad, T, 1, tpad, at_u8(L.xs_c), at_u8(L.xs_s),
                               at_f(L.xs_g), s, status);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    auto problem = [&](const ft_moe_banks *b, bool gate_up, bool is_shared) {
        W4Params q = {};
        const int il = is_shared ? G.Isl : G.Il;
        q.w_scales = static_cast<const uint8_t *>(b->p[gate_up ? FT_GU_SCALE : FT_DN_SCALE]);
        q.w_glob = static_cast<const float *>(b->p[gate_up ? FT_GU_GLOBAL : FT_DN_GLOBAL]);
        q.R = gate_up ? 2 * il : G.H;
        q.K = gate_up ? G.H : il;
        q.group = G.g;
        q.up_off = gate_up ? il : 0;
        q.n_mtiles = gate_up ? il / 128 : G.H / 256;
        if (is_shared) {
            q.n_pos_static = T; q.n_slots = T; q.top_k = 1; q.num_experts = 1;
        } else {
            q.n_pos_dev = npad; q.sorted_slot = sorted; q.block_expert = bexp; q.n_slots = n_slots; q.top_k = G.k;
            q.num_experts = G.E;
        }
        q.status = status;
        return q;
    };
    W4Params gp[2] = {problem(routed, true, false), {}};
    gp[0].a_scales = at_u8(L.xq_s); gp[0].a_glob = at_f(L.xq_g); gp[0].h_out = at_f(L.h); gp[0].h_ld = G.Il;
    W4Operands gops[2] = {{routed->p[FT_GU], (int64_t)G.E * 2 * G.Il, at_u8(L.xq_c), L.pmax}, {}};
    const int max_blocks = L.pmax / kTcBlock, tblocks = tpad / kTcBlock;
    int nprob = 1, units = max_blocks * gp[0].n_mtiles;
    if (G.Is) {
        gp[1] = problem(shared, true, true);
        gp[1].a_scales = at_u8(L.xs_s); gp[1].a_glob = at_f(L.xs_g); gp[1].h_out = at_f(L.hs); gp[1].h_ld = G.Isl;
        gops[1] = {shared->p[FT_GU], 2 * (int64_t)G.Isl, at_u8(L.xs_c), tpad};
        nprob = 2;
        units += tblocks * gp[1].n_mtiles;
    }
    if ((e = launch_w4a4_gemm(gp, gops, nprob, true, units, s)) != cudaSuccess) return cuda_fail(e, "gate_up launch");
    if ((e = stage_mark(FT_STAGE_SHARED_GATE_UP, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    if ((e = stage_mark(FT_STAGE_DOWN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    // h (fp32, position rows) as NVFP4
    e = launch_quant_nvfp4(at_f(L.h), true, G.Il, nullptr, npad, 0, L.pmax, 1, L.pmax, at_u8(L.hq_c), at_u8(L.hq_s),
                           at_f(L.hq_g), s, status);
    if (e == cudaSuccess && G.Is)
        e = launch_quant_nvfp4(at_f(L.hs), true, G.Isl, nullptr, nullptr, tpad, tpad, 1, tpad, at_u8(L.hsq_c),
                               at_u8(L.hsq_s), at_f(L.hsq_g), s, status);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    float *y = at_f(L.y), *y_sh = at_f(L.y_sh);
    W4Params dp[2] = {problem(routed, false, false), {}};
    dp[0].a_scales = at_u8(L.hq_s); dp[0].a_glob = at_f(L.hq_g); dp[0].y_out = y; dp[0].y_ld = G.H;
    dp[0].route_w = topk_w;
    W4Operands dops[2] = {{routed->p[FT_DN], (int64_t)G.E * G.H, at_u8(L.hq_c), L.pmax}, {}};
    nprob = 1;
    units = max_blocks * dp[0].n_mtiles;
    if (G.Is) {
        dp[1] = problem(shared, false, true);
        dp[1].a_scales = at_u8(L.hsq_s); dp[1].a_glob = at_f(L.hsq_g); dp[1].y_out = y_sh; dp[1].y_ld = G.H;
        dops[1] = {shared->p[FT_DN], G.H, at_u8(L.hsq_c), tpad};
        nprob = 2;
        units += tblocks * dp[1].n_mtiles;
    }
    if ((e = launch_w4a4_gemm(dp, dops, nprob, false, units, s)) != cudaSuccess) return cuda_fail(e, "down launch");
    if ((e = stage_mark(FT_STAGE_SHARED_DOWN, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    if ((e = stage_mark(FT_STAGE_COMBINE, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    e = launch_combine(y, G.Is ? y_sh : nullptr, T, G.k, G.H, out, out_dtype, s);
    if (e != cudaSuccess) return cuda_fail(e, "combine launch");
    if ((e = stage_mark(FT_NSTAGES, s)) != cudaSuccess) return cuda_fail(e, "stage event");
    return ok();
}

ft_status ft_moe_quantize_nvfp4(const void *src, int32_t src_dtype, int32_t rows, int32_t K, uint8_t *codes,
                                uint8_t *scales, float *glob, void *stream)
{
    FT_NVTX_RANGE("ft_moe_quantize_nvfp4");
    if (src_dtype != FT_DTYPE_BF16 && src_dtype != FT_DTYPE_F32)
        return fail(FT_ERR_INVALID_ARG, "src_dtype must be FT_DTYPE_BF16 or FT_DTYPE_F32");
    if (rows < 0 || K <= 0 || K % 16) return fail(FT_ERR_INVALID_ARG, "need rows >= 0 and K a positive multiple of 16");
    if (rows == 0) return ok();
    if (!src || !codes || !scales || !glob || !aligned(codes, 8) || !aligned(src, 16) || !aligned(glob, 4))
        return fail(FT_ERR_INVALID_ARG, "pointers must be non-NULL; src 16-byte and codes 8-byte aligned");
    cudaError_t e = launch_quant_nvfp4(src, src_dtype == FT_DTYPE_F32, K, nullptr, nullptr, rows, rows, 1, rows, codes,
                                       scales, glob, static_cast<cudaStream_t>(stream), nullptr);
    if (e != cudaSuccess) return cuda_fail(e, "quantize launch");
    return ok();
}

ft_status ft_moe_dequant(const ft_moe_config *cfg, int32_t shared, const ft_moe_banks *banks, int32_t which,
                         int32_t expert, void *out_bf16, void *stream)
{
    FT_NVTX_RANGE("ft_moe_dequant");
    Geometry G;
    ft_status st = check_config(cfg, G);
    if (st) return st;
    if (shared != 0 && shared != 1) return fail(FT_ERR_INVALID_ARG, "shared must be 0 or 1");
    if (shared && G.Is == 0) return fail(FT_ERR_UNSUPPORTED, "layer has no shared expert");
    if (G.fmt != FT_FORMAT_NVFP4) return fail(FT_ERR_UNSUPPORTED, "dequant export is for NVFP4 banks");
    if (!banks_ok(banks) || !out_bf16 || !aligned(out_bf16, 16))
        return fail(FT_ERR_INVALID_ARG, "banks and out must be non-NULL and 16-byte aligned");
    const int E = shared ? 1 : G.E, Il = shared ? G.Isl : G.Il;
    if (expert < 0 || expert >= E) return fail(FT_ERR_INVALID_ARG, "expert %d out of range", expert);
    int rows, K, cidx, sidx;
    if (which == FT_GU) { rows = 2 * Il; K = G.H; cidx = FT_GU; sidx = FT_GU_SCALE; }
    else if (which == FT_DN) { rows = G.H; K = Il; cidx = FT_DN; sidx = FT_DN_SCALE; }
    else return fail(FT_ERR_INVALID_ARG, "which must be FT_GU or FT_DN");
    const uint8_t *codes = static_cast<const uint8_t *>(banks->p[cidx]) + (size_t)expert * rows * (K / 2);
    const uint8_t *scales = static_cast<const uint8_t *>(banks->p[sidx]) + (size_t)expert * rows * (K / G.g);
    cudaError_t e = launch_dequant(codes, scales, rows, K, G.g, static_cast<uint16_t *>(out_bf16),
                                   static_cast<cudaStream_t>(stream));
    if (e != cudaSuccess) return cuda_fail(e, "dequant launch");
    return ok();
}

ft_status ft_moe_read_status(const void *workspace, void *stream)
{
    FT_NVTX_RANGE("ft_moe_read_status");
    if (!workspace) return fail(FT_ERR_INVALID_ARG, "workspace is NULL");
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) return cuda_fail(e, "stream synchronize");
    int v = 0;
    e = cudaMemcpy(&v, workspace, sizeof(int), cudaMemcpyDeviceToHost);
    if (e != cudaSuccess) return cuda_fail(e, "status read");
    if (v == FT_OK) return ok();
    if (v == FT_ERR_INVALID_ROUTING) return fail(FT_ERR_INVALID_ROUTING, "invalid routing ids were skipped");
    if (v == FT_ERR_TIMEOUT) return fail(FT_ERR_TIMEOUT, "a bounded device wait gave up");
    return fail(FT_ERR_CUDA, "unexpected device status %d", v);
}

}  // extern "C"
