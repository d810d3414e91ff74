/*
 * CPU oracle for the NVFP4 (W4A16) routed-MoE expert forward.
 *
 * TEST INFRASTRUCTURE ONLY. This file is the plain, slow, fp64 statement of what
 * the layer computes. It is compiled into liboracle.so and loaded only by the
 * tests, by __graft_entry__.smoke() and by bench.py's CPU-baseline leg. It shares
 * no code, header, table or helper with the CUDA library, and neither side
 * includes or links the other.
 *
 * Sources (pages about tensor-parallel sharding of quantized MoE experts):
 *  - "[TP=2] Quantized MoE expert parallelism on heterogeneous consumer CUDA GPUs
 *    -- a working NVFP4 port", section 4 "The patch" (expert sharding rule, the
 *    linearity argument: MoE output = sum_i silu(gate_i)*up_i @ down_i) and its
 *    diff of nvfp4.py (bank layout: gate_up [2I, H/2], gate_up_scale [2I, H/GROUP],
 *    per-row globals expanded from the checkpoint's weight_scale_2) and of
 *    nvfp4_banks.py (_shard_expert_tensor: gate/up narrow dim 0, down narrow the
 *    last dim, globals whole).
 *  - "Offloaded MoE ignores tensor parallelism", section "What it touches" item 1
 *    (gate_up rows [0,I) gate and [I,2I) up: a rank's slice is two disjoint row
 *    ranges; down is a column slice) and the follow-up comment (norm_topk_prob:
 *    softmax, top-k, renormalise; replicated router; SUM of partials is exact).
 *  - "feat(qwen3_5_moe): tensor-parallel weight sharding", Implementation notes
 *    (companion scales split along their weight's axis; per-output-row global).
 *  - "[1/3] feat(dsv4): add tensor-parallel DeepSeek-V4 runtime", table "Tensor
 *    ownership and collectives" (shared SwiGLU expert on the same split, added to
 *    the routed partial before the one reduction).
 *
 * Readings where the pages are silent:
 *  - element 2m of a packed row sits in the LOW nibble of byte m, 2m+1 in the high;
 *  - e2m1 nibble = S.EE.M (bit 3 sign) valued sign * {0,.5,1,1.5,2,3,4,6}[bits 0-2];
 *  - block scales are OCP E4M3 "fn" (bias 7, no infinities, S.1111.111 = NaN);
 *  - weight_global is a per-output-row fp32 multiplier;
 *  - routing: softmax over all experts, the k largest probabilities (ties to the
 *    lower expert index) in descending order, renormalised to sum 1;
 *  - SwiGLU h_i = silu(g_i) * u_i with silu(z) = z / (1 + e^-z), gate rows first;
 *  - the shared expert is added with weight 1 after the k routed terms.
 *
 * fp8_block experts (the second expert format of the same pages: "feat(qwen3_5_moe):
 * tensor-parallel weight sharding", Summary and Implementation notes -- an fp8-block
 * weight carries a 128-block weight_scale_inv, split along the same axis as its weight;
 * "[1/3] feat(dsv4)...", Checkpoint loading -- FP8 128x128 blocks cannot be cut at
 * arbitrary boundaries; "Offloaded MoE ignores tensor parallelism", item 2 -- I/tp a
 * multiple of 128): W[n][k] = e4m3(code[n][k]) * scale_inv[n/128][k/128], one code byte
 * per element, no per-row global. Reading where the pages are silent: scale_inv is the
 * fp32 multiplier that dequantises (the weight is code times scale_inv).
 *
 * Parity pins for every function here live in tests/test_oracle_pins.py.
 * The absolute output values are "parity unpinned" against the pages: they print
 * no worked numeric example of the MoE arithmetic.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* Negative-control switch used only by tests: a nonzero value plants one known
 * mistake (see ORC_MUT_*), so the pins can be shown to catch it. */
int orc_mutation = 0;
enum {
    ORC_MUT_NONE = 0,
    ORC_MUT_NIBBLE_ORDER = 1,   /* even element read from the high nibble */
    ORC_MUT_SWAP_GATE_UP = 2,   /* silu applied to up instead of gate */
    ORC_MUT_DROP_GLOBAL = 3,    /* weight_global ignored */
    ORC_MUT_SCALE_INDEX = 4,    /* block scale taken from the next group */
    ORC_MUT_E2M1_SIGN = 5,      /* e2m1 sign bit ignored */
    ORC_MUT_NO_RENORM = 6,      /* routing weights not renormalised */
    ORC_MUT_TIE_HIGH = 7,       /* routing ties go to the higher index */
    ORC_MUT_DOWN_ROWS = 8,      /* down sliced along rows instead of columns */
    ORC_MUT_DROP_SHARED = 9,    /* shared expert left out */
    ORC_MUT_DROP_ROUTE_W = 10,  /* routed terms not weighted */
    ORC_MUT_E4M3_BIAS = 11,     /* e4m3 exponent bias 8 instead of 7 */
    ORC_MUT_UP_SLICE = 12,      /* up rows taken from the gate half */
    ORC_MUT_ROUTER_T = 13,      /* router weight read transposed (square shapes only) */
    ORC_MUT_FP8_BLOCK_T = 14,   /* fp8_block: scale block indexed [k/128][n/128] */
    ORC_MUT_DEQUANT_T = 15,     /* dense matrices written column-major ([K][rows]) */
    ORC_MUT_W4A4_NO_H = 16,     /* W4A4: h enters down unquantized */
    ORC_MUT_E2M1_TIE_UP = 17,   /* e2m1 rounding: ties away from zero */
    ORC_MUT_ROW_SCALE = 18,     /* activation row scale amax / 6 (448 forgotten) */
};

/* ---------------------------------------------------------------- formats */

/* e2m1 value table: the eight magnitudes of a 3-bit E2M1 code. */
static const double E2M1_MAG[8] = {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0};

double orc_e2m1(unsigned nibble)
{
    double mag = E2M1_MAG[nibble & 7u];
    int neg = (nibble >> 3) & 1u;
    if (orc_mutation == ORC_MUT_E2M1_SIGN) neg = 0;
    return neg ? -mag : mag;
}

/* OCP FP8 E4M3 ("fn"): 1 sign, 4 exponent (bias 7), 3 mantissa bits; exponent 0
 * is subnormal (m/8 * 2^-6); S.1111.111 is NaN; there are no infinities. */
double orc_e4m3(unsigned byte)
{
    unsigned s = (byte >> 7) & 1u, e = (byte >> 3) & 15u, m = byte & 7u;
    int bias = (orc_mutation == ORC_MUT_E4M3_BIAS) ? 8 : 7;
    double v;
    if (e == 15u && m == 7u) return NAN;
    if (e == 0u) v = ldexp((double)m / 8.0, 1 - bias);
    else v = ldexp(1.0 + (double)m / 8.0, (int)e - bias);
    return s ? -v : v;
}

/* bf16 bit pattern of a double, round to nearest even (exact when representable). */
static uint16_t to_bf16_bits(double v)
{
    float f = (float)v;
    uint32_t u;
    memcpy(&u, &f, 4);
    if ((u & 0x7F800000u) == 0x7F800000u && (u & 0x7FFFFFu)) return (uint16_t)((u >> 16) | 0x40u);
    u += 0x7FFFu + ((u >> 16) & 1u);
    return (uint16_t)(u >> 16);
}

double orc_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, 4);
    return (double)f;
}

/* The dequantised weight value e2m1(code) * e4m3(scale) as a bf16 bit pattern.
 * The product has at most 6 significant bits and lies in [2^-10, 2688], so it is
 * exactly representable in bf16. */
uint16_t orc_dequant_bf16(unsigned nibble, unsigned scale_byte)
{
    return to_bf16_bits(orc_e2m1(nibble) * orc_e4m3(scale_byte));
}

/* Value tables filled from the two decoders above at the start of every exported
 * matrix routine (so a planted mutation is honoured); they only avoid calling
 * ldexp once per weight element. */
static double e2m1_tab[16], e4m3_tab[256];

static void fill_tables(void)
{
    for (unsigned i = 0; i < 16; ++i) e2m1_tab[i] = orc_e2m1(i);
    for (unsigned i = 0; i < 256; ++i) e4m3_tab[i] = orc_e4m3(i);
}

/* Code of element k of a packed row (two e2m1 codes per byte). */
static unsigned code_at(const uint8_t *row, int k)
{
    unsigned byte = row[k >> 1];
    int high = k & 1;
    if (orc_mutation == ORC_MUT_NIBBLE_ORDER) high = !high;
    return high ? (byte >> 4) & 15u : byte & 15u;
}

/* W[n][k] = e2m1(code[n][k]) * e4m3(scale[n][k/g]) * global[n]
 * for one expert's [rows, K] matrix stored as codes [rows][K/2],
 * scales [rows][K/g], globals [rows]. */
static double weight_at(const uint8_t *codes, const uint8_t *scales, const float *glob,
                        int n, int k, int K, int g)
{
    int grp = k / g;
    if (orc_mutation == ORC_MUT_SCALE_INDEX) grp = (grp + 1) % (K / g);
    double w = e2m1_tab[code_at(codes + (size_t)n * (K / 2), k)] *
               e4m3_tab[scales[(size_t)n * (K / g) + grp]];
    if (orc_mutation != ORC_MUT_DROP_GLOBAL) w *= (double)glob[n];
    return w;
}

/* fp8_block: W[n][k] = e4m3(code[n][k]) * scale_inv[n/128][k/128] for one expert's
 * [rows, K] matrix stored as codes [rows][K] and scale_inv [rows/128][K/128]. */
static double fp8_weight_at(const uint8_t *codes, const float *sinv, int n, int k, int K)
{
    int nb = n / 128, kb = k / 128, kblocks = K / 128;
    size_t s = (orc_mutation == ORC_MUT_FP8_BLOCK_T) ? (size_t)kb * kblocks + nb : (size_t)nb * kblocks + kb;
    return e4m3_tab[codes[(size_t)n * K + k]] * (double)sinv[s];
}

void orc_dequant_fp8_matrix(const uint8_t *codes, const float *sinv, int rows, int K, double *out)
{
    fill_tables();
    for (int n = 0; n < rows; ++n)
        for (int k = 0; k < K; ++k) {
            size_t at = (orc_mutation == ORC_MUT_DEQUANT_T) ? (size_t)k * rows + n : (size_t)n * K + k;
            out[at] = fp8_weight_at(codes, sinv, n, k, K);
        }
}

/* Dense dequantised matrix of one expert, W as above, row-major [rows][K]. */
void orc_dequant_matrix(const uint8_t *codes, const uint8_t *scales, const float *glob,
                        int rows, int K, int g, double *out)
{
    fill_tables();
    for (int n = 0; n < rows; ++n)
        for (int k = 0; k < K; ++k) {
            size_t at = (orc_mutation == ORC_MUT_DEQUANT_T) ? (size_t)k * rows + n : (size_t)n * K + k;
            out[at] = weight_at(codes, scales, glob, n, k, K, g);
        }
}

/* ---------------------------------------------------------------- routing */

typedef struct { double p; int idx; } scored;

static int by_prob_desc(const void *a, const void *b)
{
    const scored *x = (const scored *)a, *y = (const scored *)b;
    if (x->p > y->p) return -1;
    if (x->p < y->p) return 1;
    if (orc_mutation == ORC_MUT_TIE_HIGH) return (x->idx > y->idx) ? -1 : (x->idx < y->idx);
    return (x->idx < y->idx) ? -1 : (x->idx > y->idx);
}

/* Router: p = softmax(logits_t) over E experts; keep the k largest (descending,
 * ties to the lower index); w_j = p_j / sum of the kept p. Returns 0, or -1 on bad
 * arguments. */
int orc_route(const float *logits, int T, int E, int k, int32_t *ids, double *w)
{
    if (T < 0 || E <= 0 || k <= 0 || k > E) return -1;
    scored *s = (scored *)malloc(sizeof(scored) * (size_t)E);
    if (!s) return -1;
    for (int t = 0; t < T; ++t) {
        const float *l = logits + (size_t)t * E;
        double m = -INFINITY, sum = 0.0;
        for (int e = 0; e < E; ++e) m = fmax(m, (double)l[e]);
        for (int e = 0; e < E; ++e) { s[e].p = exp((double)l[e] - m); s[e].idx = e; sum += s[e].p; }
        for (int e = 0; e < E; ++e) s[e].p /= sum;
        qsort(s, (size_t)E, sizeof(scored), by_prob_desc);
        double kept = 0.0;
        for (int j = 0; j < k; ++j) kept += s[j].p;
        for (int j = 0; j < k; ++j) {
            ids[(size_t)t * k + j] = s[j].idx;
            w[(size_t)t * k + j] = (orc_mutation == ORC_MUT_NO_RENORM) ? s[j].p : s[j].p / kept;
        }
    }
    free(s);
    return 0;
}

/* ---------------------------------------------------------------- align */

/* Expert-sorted, tile-padded slot order. Slot s = t*k + j. Slots are grouped by
 * expert in increasing expert order, kept in increasing slot order inside an
 * expert, and each expert's run is padded with the sentinel T*k up to a multiple
 * of B. Experts with no slots get no blocks. Outputs:
 *   sorted_slot[n_padded], block_expert[n_padded / B], expert_off[E+1]
 *   (start of each expert's padded run; expert_off[E] = n_padded).
 * Returns 0, or -1 on an out-of-range id or bad arguments. Caller sizes
 * sorted_slot for T*k + E*(B-1) entries. */
/* Router logits of the replicated router ("[1/3] feat(dsv4): add tensor-parallel
 * DeepSeek-V4 runtime", table "Tensor ownership and collectives": the router is
 * replicated and every rank computes the same routing): logits[t][e] = sum_h
 * x[t][h] * W[e][h] over the bf16 values of x [T][H] and W [E][H]. Every product of
 * two bf16 values is exact in fp64 (16 significant bits), so the only rounding is
 * the fp64 summation (relative error below H * 2^-53 of absum). absum[t][e] = sum_h
 * |x[t][h] * W[e][h]|, the scale of any rounding error of a lower-precision sum. */
void orc_router_logits(const uint16_t *x, const uint16_t *w, int T, int H, int E, double *logits, double *absum)
{
    for (int t = 0; t < T; ++t) {
        for (int e = 0; e < E; ++e) {
            double acc = 0.0, mag = 0.0;
            for (int h = 0; h < H; ++h) {
                const uint16_t wb = orc_mutation == ORC_MUT_ROUTER_T ? w[(size_t)h * E + e] : w[(size_t)e * H + h];
                const double prod = orc_bf16_to_double(x[(size_t)t * H + h]) * orc_bf16_to_double(wb);
                acc += prod;
                mag += fabs(prod);
            }
            logits[(size_t)t * E + e] = acc;
            absum[(size_t)t * E + e] = mag;
        }
    }
}

int orc_align(const int32_t *ids, int T, int k, int E, int B,
              int32_t *sorted_slot, int32_t *block_expert, int32_t *expert_off, int32_t *n_padded)
{
    if (T < 0 || k <= 0 || E <= 0 || B <= 0) return -1;
    int n = T * k, pos = 0;
    for (int s = 0; s < n; ++s)
        if (ids[s] < 0 || ids[s] >= E) return -1;
    for (int e = 0; e < E; ++e) {
        expert_off[e] = pos;
        int start = pos;
        for (int s = 0; s < n; ++s)
            if (ids[s] == e) sorted_slot[pos++] = s;
        while ((pos - start) % B) sorted_slot[pos++] = n;
        for (int b = start / B; b < pos / B; ++b) block_expert[b] = e;
    }
    expert_off[E] = pos;
    *n_padded = pos;
    return 0;
}

/* ---------------------------------------------------------------- tp slicing */

/* Rank-local bank of `E` experts from checkpoint-shaped full-I pieces.
 * gate_up rows [0, I_l) = gate rows [r*I_l, (r+1)*I_l); rows [I_l, 2*I_l) = up rows
 * [r*I_l, (r+1)*I_l) -- in the fused [2I, .] view these are the two disjoint ranges
 * [r*I_l, ...) and [I + r*I_l, ...). Scales and globals follow their rows.
 * down keeps all H rows and takes code columns [r*I_l/2, (r+1)*I_l/2) and scale
 * columns [r*I_l/g, (r+1)*I_l/g); down_global stays whole. */
int orc_slice(int E, int H, int I, int g, int tp_rank, int tp_size,
              const uint8_t *gate, const uint8_t *gate_scale, const float *gate_global,
              const uint8_t *up, const uint8_t *up_scale, const float *up_global,
              const uint8_t *down, const uint8_t *down_scale, const float *down_global,
              uint8_t *gu, uint8_t *gu_scale, float *gu_global,
              uint8_t *dn, uint8_t *dn_scale, float *dn_global)
{
    if (tp_size <= 0 || tp_rank < 0 || tp_rank >= tp_size || I % tp_size) return -1;
    int Il = I / tp_size;
    if (Il % g || H % g || H % 2 || Il % 2) return -1;
    size_t hr = (size_t)H / 2, hs = (size_t)H / g;
    for (int e = 0; e < E; ++e) {
        for (int i = 0; i < Il; ++i) {
            size_t src = (size_t)e * I + (size_t)tp_rank * Il + i;
            size_t up_src = (orc_mutation == ORC_MUT_UP_SLICE) ? (size_t)e * I + i : src;
            size_t dg = (size_t)e * 2 * Il + i, du = dg + Il;
            memcpy(gu + dg * hr, gate + src * hr, hr);
            memcpy(gu + du * hr, up + up_src * hr, hr);
            memcpy(gu_scale + dg * hs, gate_scale + src * hs, hs);
            memcpy(gu_scale + du * hs, up_scale + up_src * hs, hs);
            gu_global[dg] = gate_global[src];
            gu_global[du] = up_global[up_src];
        }
        for (int n = 0; n < H; ++n) {
            size_t row = (size_t)e * H + n;
            if (orc_mutation == ORC_MUT_DOWN_ROWS) {
                /* planted mistake: rows of the rank's share of H, all columns packed */
                size_t srow = (size_t)e * H + ((size_t)tp_rank * H / tp_size + n / tp_size);
                memcpy(dn + row * (Il / 2), down + srow * (I / 2), (size_t)Il / 2);
                memcpy(dn_scale + row * (Il / g), down_scale + srow * (I / g), (size_t)Il / g);
            } else {
                memcpy(dn + row * (Il / 2), down + row * (I / 2) + (size_t)tp_rank * Il / 2, (size_t)Il / 2);
                memcpy(dn_scale + row * (Il / g), down_scale + row * (I / g) + (size_t)tp_rank * Il / g,
                       (size_t)Il / g);
            }
            dn_global[row] = down_global[row];
        }
    }
    return 0;
}

/* Rank-local bank for an explicit intermediate range [begin, begin + len), the
 * asymmetric split the "[TP=2] Quantized MoE expert parallelism ... NVFP4 port" page
 * leaves open (section 8: a shard ratio weighted toward the faster card was not
 * attempted). The slicing rule is the even split's (section 4, _shard_expert_tensor:
 * gate and up rows of the range, down columns of the range, globals of those rows,
 * down_global whole) with the range given instead of derived; the linearity argument
 * of section 4 makes the partials of any partition of [0, I) sum to the full output.
 * begin and len must be multiples of the scale block. */
int orc_slice_range(int E, int H, int I, int g, int begin, int len,
                    const uint8_t *gate, const uint8_t *gate_scale, const float *gate_global,
                    const uint8_t *up, const uint8_t *up_scale, const float *up_global,
                    const uint8_t *down, const uint8_t *down_scale, const float *down_global,
                    uint8_t *gu, uint8_t *gu_scale, float *gu_global,
                    uint8_t *dn, uint8_t *dn_scale, float *dn_global)
{
    if (begin < 0 || len <= 0 || begin + len > I || begin % g || len % g || H % g || H % 2) return -1;
    size_t hr = (size_t)H / 2, hs = (size_t)H / g;
    for (int e = 0; e < E; ++e) {
        for (int i = 0; i < len; ++i) {
            size_t src = (size_t)e * I + (size_t)begin + i;
            size_t up_src = (orc_mutation == ORC_MUT_UP_SLICE) ? (size_t)e * I + i : src;
            size_t dg = (size_t)e * 2 * len + i, du = dg + len;
            memcpy(gu + dg * hr, gate + src * hr, hr);
            memcpy(gu + du * hr, up + up_src * hr, hr);
            memcpy(gu_scale + dg * hs, gate_scale + src * hs, hs);
            memcpy(gu_scale + du * hs, up_scale + up_src * hs, hs);
            gu_global[dg] = gate_global[src];
            gu_global[du] = up_global[up_src];
        }
        for (int n = 0; n < H; ++n) {
            size_t row = (size_t)e * H + n;
            memcpy(dn + row * (len / 2), down + row * (I / 2) + (size_t)begin / 2, (size_t)len / 2);
            memcpy(dn_scale + row * (len / g), down_scale + row * (I / g) + (size_t)begin / g, (size_t)len / g);
            dn_global[row] = down_global[row];
        }
    }
    return 0;
}

/* fp8_block rank-local bank for the intermediate range [begin, begin + len) (begin
 * and len multiples of 128, the scale block): gate and up rows of the range with their
 * scale_inv block rows (gate first), down columns of the range with their scale_inv
 * block columns -- the rule of "feat(qwen3_5_moe): tensor-parallel weight sharding"
 * (gate/up split along output rows, down along input columns, companions with their
 * weight). Pieces: gate, up [E][I][H] u8 and [E][I/128][H/128] f32; down [E][H][I] u8
 * and [E][H/128][I/128] f32. Bank: gu [E][2len][H], gu_sinv [E][2len/128][H/128],
 * dn [E][H][len], dn_sinv [E][H/128][len/128]. */
int orc_slice_fp8_range(int E, int H, int I, int begin, int len,
                        const uint8_t *gate, const float *gate_sinv, const uint8_t *up, const float *up_sinv,
                        const uint8_t *down, const float *down_sinv,
                        uint8_t *gu, float *gu_sinv, uint8_t *dn, float *dn_sinv)
{
    if (begin < 0 || len <= 0 || begin + len > I || begin % 128 || len % 128 || H % 128 || I % 128) return -1;
    size_t hb = (size_t)H / 128, ib = (size_t)I / 128, lb = (size_t)len / 128;
    for (int e = 0; e < E; ++e) {
        for (int i = 0; i < len; ++i) {
            size_t src = (size_t)e * I + (size_t)begin + i;
            size_t up_src = (orc_mutation == ORC_MUT_UP_SLICE) ? (size_t)e * I + i : src;
            memcpy(gu + ((size_t)e * 2 * len + i) * H, gate + src * H, (size_t)H);
            memcpy(gu + ((size_t)e * 2 * len + len + i) * H, up + up_src * H, (size_t)H);
        }
        for (size_t b = 0; b < lb; ++b) {
            size_t src = (size_t)e * ib + (size_t)begin / 128 + b;
            memcpy(gu_sinv + ((size_t)e * 2 * lb + b) * hb, gate_sinv + src * hb, hb * sizeof(float));
            memcpy(gu_sinv + ((size_t)e * 2 * lb + lb + b) * hb, up_sinv + src * hb, hb * sizeof(float));
        }
        for (int n = 0; n < H; ++n) {
            size_t row = (size_t)e * H + n;
            memcpy(dn + row * len, down + row * I + begin, (size_t)len);
        }
        for (size_t nb = 0; nb < hb; ++nb) {
            size_t row = (size_t)e * hb + nb;
            memcpy(dn_sinv + row * lb, down_sinv + row * ib + (size_t)begin / 128, lb * sizeof(float));
        }
    }
    return 0;
}

/* ---------------------------------------------------------------- W4A4: NVFP4 activations
 *
 * The native FP4 variant feeds the tensor cores e2m1 activations too (W4A4), which the
 * pages' sm_86/sm_89 cards could not run ("[TP=2] Quantized MoE expert parallelism ... NVFP4
 * port", section 2: no native FP4 tensor cores there, so NVFP4 ran as W4A16). The pages do
 * not define how activations are quantized; the reading taken here is NVFP4's own two-level
 * scaling applied per activation row: a row scale glob = amax / (6 * 448) in fp32, one e4m3
 * block scale per 16 elements s = e4m3(block amax / (6 * glob)), codes q = e2m1(x * r) with
 * r = 1 / (s * glob) the block's reciprocal, both conversions rounding to nearest with ties
 * to even and saturating; value q * s * glob. Every step is one correctly rounded fp32
 * operation in this order, the precision the kernels take these decisions in. */

/* e4m3 code of a finite v >= 0: the nearest non-negative finite e4m3 value, ties to the
 * even code, values above 448 saturating to 448 (chosen by scanning all 127 codes). */
static unsigned e4m3_code_rne(float v)
{
    if (!(v > 0.0f)) return 0u;
    unsigned best = 0;
    double bd = INFINITY;
    for (unsigned c = 0; c < 0x7Fu; ++c) {
        double d = fabs(orc_e4m3(c) - (double)v);
        if (d < bd || (d == bd && (c & 1u) == 0u)) { bd = d; best = c; }
    }
    return best;
}

/* e2m1 code of a finite v: sign bit 3, magnitude the nearest of {0,.5,1,1.5,2,3,4,6}
 * (ties to the even code, above 6 saturating to 6). */
static unsigned e2m1_code_rne(float v)
{
    unsigned sign = v < 0.0f ? 8u : 0u;
    double a = fabs((double)v), bd = INFINITY;
    unsigned best = 0;
    for (unsigned c = 0; c < 8u; ++c) {
        double d = fabs(E2M1_MAG[c] - a);
        int tie_wins = (orc_mutation == ORC_MUT_E2M1_TIE_UP) ? 1 : (c & 1u) == 0u;
        if (d < bd || (d == bd && tie_wins)) { bd = d; best = c; }
    }
    return sign | best;
}

unsigned orc_e4m3_code(float v) { return e4m3_code_rne(v); }
unsigned orc_e2m1_code(float v) { return e2m1_code_rne(v); }

/* NVFP4 quantization of `rows` rows of K fp32 values (K a multiple of 16): codes
 * [rows][K/2] (element 2m in the low nibble of byte m), e4m3 block scales [rows][K/16],
 * fp32 row scales [rows]. */
void orc_quant_nvfp4(const float *x, int rows, int K, uint8_t *codes, uint8_t *scales, float *glob)
{
    for (int r = 0; r < rows; ++r) {
        const float *xr = x + (size_t)r * K;
        float amax = 0.0f;
        for (int k = 0; k < K; ++k) if (fabsf(xr[k]) > amax) amax = fabsf(xr[k]);
        float g = amax / (orc_mutation == ORC_MUT_ROW_SCALE ? 6.0f : 2688.0f);
        glob[r] = g;
        for (int b = 0; b < K / 16; ++b) {
            float bmax = 0.0f;
            for (int i = 0; i < 16; ++i) if (fabsf(xr[16 * b + i]) > bmax) bmax = fabsf(xr[16 * b + i]);
            unsigned sc = 0;
            if (g > 0.0f) {
                float six_g = 6.0f * g;
                sc = e4m3_code_rne(bmax / six_g);
            }
            scales[(size_t)r * (K / 16) + b] = (uint8_t)sc;
            float sv = (float)orc_e4m3(sc);
            float d = sv * g;
            float rcp = d > 0.0f ? 1.0f / d : 0.0f;
            for (int i = 0; i < 16; i += 2) {
                unsigned lo = 0, hi = 0;
                if (sv > 0.0f) {
                    float q0 = xr[16 * b + i] * rcp, q1 = xr[16 * b + i + 1] * rcp;
                    lo = e2m1_code_rne(q0);
                    hi = e2m1_code_rne(q1);
                }
                codes[(size_t)r * (K / 2) + 8 * b + i / 2] = (uint8_t)(lo | (hi << 4));
            }
        }
    }
}

/* The values of one quantized row (K elements): out[k] = e2m1 * e4m3 * glob, exact in fp64. */
static void nvfp4_row_values(const uint8_t *codes, const uint8_t *scales, float glob, int K, double *out)
{
    for (int k = 0; k < K; ++k) {
        unsigned byte = codes[k >> 1];
        unsigned q = (k & 1) ? (byte >> 4) & 15u : byte & 15u;
        out[k] = orc_e2m1(q) * orc_e4m3(scales[k / 16]) * (double)glob;
    }
}

/* Quantize one fp32 row and return its values in fp64 (scratch: K/2 + K/16 bytes). */
static void quant_dequant_row(const float *x, int K, uint8_t *scratch, double *out)
{
    float g;
    orc_quant_nvfp4(x, 1, K, scratch, scratch + K / 2, &g);
    nvfp4_row_values(scratch, scratch + K / 2, g, K, out);
}

/* ---------------------------------------------------------------- expert MLP */

typedef struct {
    const uint8_t *gu, *gu_scale;   /* [E][2*Il][H/2], [E][2*Il][H/g] */
    const float *gu_global;         /* [E][2*Il] */
    const uint8_t *dn, *dn_scale;   /* [E][H][Il/2], [E][H][Il/g] */
    const float *dn_global;         /* [E][H] */
    int32_t E, H, Il, g;
    int32_t fmt;                    /* 0: NVFP4 as above; 1: fp8_block -- gu [E][2*Il][H] and
                                       dn [E][H][Il] code bytes, gu_scale / dn_scale fp32
                                       scale_inv [E][2*Il/128][H/128] / [E][H/128][Il/128],
                                       no globals */
} orc_bank;

/* W of expert e's gate_up (which = 0) or down (which = 1) matrix at [n][k]. */
static double bank_weight(const orc_bank *b, int which, int e, int n, int k)
{
    int rows = which ? b->H : 2 * b->Il, K = which ? b->Il : b->H;
    const uint8_t *codes = which ? b->dn : b->gu;
    if (b->fmt == 1) {
        const float *sinv = (const float *)(which ? b->dn_scale : b->gu_scale);
        return fp8_weight_at(codes + (size_t)e * rows * K, sinv + (size_t)e * (rows / 128) * (K / 128), n, k, K);
    }
    const uint8_t *scales = which ? b->dn_scale : b->gu_scale;
    const float *glob = which ? b->dn_global : b->gu_global;
    return weight_at(codes + (size_t)e * rows * (K / 2), scales + (size_t)e * rows * (K / b->g),
                     glob + (size_t)e * rows, n, k, K, b->g);
}

/* Pre-activations G[n] = sum_k x[k] * W_gu[e][n][k], n < 2*Il (gate rows first). */
static void expert_gate_up(const orc_bank *b, int e, const uint16_t *x_row, double *G)
{
    int H = b->H, rows = 2 * b->Il;
    for (int n = 0; n < rows; ++n) {
        double acc = 0.0;
        for (int k = 0; k < H; ++k) acc += orc_bf16_to_double(x_row[k]) * bank_weight(b, 0, e, n, k);
        G[n] = acc;
    }
}

/* The same on fp64 activations (the dequantized NVFP4 activations of the W4A4 variant). */
static void expert_gate_up_f64(const orc_bank *b, int e, const double *x, double *G)
{
    int H = b->H, rows = 2 * b->Il;
    for (int n = 0; n < rows; ++n) {
        double acc = 0.0;
        for (int k = 0; k < H; ++k) acc += x[k] * bank_weight(b, 0, e, n, k);
        G[n] = acc;
    }
}

/* h[i] = silu(G[i]) * G[Il + i], silu(z) = z / (1 + exp(-z)). */
void orc_swiglu(const double *G, int Il, double *h)
{
    for (int i = 0; i < Il; ++i) {
        double gate = G[i], up = G[Il + i];
        if (orc_mutation == ORC_MUT_SWAP_GATE_UP) { double t = gate; gate = up; up = t; }
        h[i] = gate / (1.0 + exp(-gate)) * up;
    }
}

/* y[n] = sum_i h[i] * W_dn[e][n][i], n < H. */
static void expert_down(const orc_bank *b, int e, const double *h, double *y)
{
    int H = b->H, Il = b->Il;
    for (int n = 0; n < H; ++n) {
        double acc = 0.0;
        for (int i = 0; i < Il; ++i) acc += h[i] * bank_weight(b, 1, e, n, i);
        y[n] = acc;
    }
}

void orc_expert_gate_up(const orc_bank *b, int e, const uint16_t *x_row, double *G)
{
    fill_tables();
    expert_gate_up(b, e, x_row, G);
}

void orc_expert_gate_up_f64(const orc_bank *b, int e, const double *x, double *G)
{
    fill_tables();
    expert_gate_up_f64(b, e, x, G);
}

void orc_expert_down(const orc_bank *b, int e, const double *h, double *y)
{
    fill_tables();
    expert_down(b, e, h, y);
}

typedef struct {
    const orc_bank *routed, *shared;
    const uint16_t *x;
    const int32_t *ids;
    const double *w;
    const int32_t *tokens;
    int n_tokens, k, H, first, last;
    double *out;
    int status;
    int w4a4;  /* NVFP4 activations: x before gate_up and h (as fp32) before down are quantized */
} fwd_job;

static void *fwd_worker(void *arg)
{
    fwd_job *j = (fwd_job *)arg;
    int H = j->H;
    int maxI = j->routed ? j->routed->Il : 0;
    if (j->shared && j->shared->Il > maxI) maxI = j->shared->Il;
    size_t maxK = (size_t)(H > maxI ? H : maxI);
    double *G = (double *)malloc(sizeof(double) * 2 * (size_t)maxI);
    double *h = (double *)malloc(sizeof(double) * (size_t)maxI);
    double *y = (double *)malloc(sizeof(double) * (size_t)H);
    /* W4A4 scratch: fp32 rows, their quantized values, quantizer output bytes */
    float *rowf = (float *)malloc(sizeof(float) * maxK);
    double *xq = (double *)malloc(sizeof(double) * (size_t)H);
    double *hq = (double *)malloc(sizeof(double) * ((size_t)maxI + 1));
    uint8_t *qs = (uint8_t *)malloc(maxK / 2 + maxK / 16 + 16);
    if ((maxI && (!G || !h)) || !y || !rowf || !xq || !hq || !qs) {
        j->status = -1;
        free(G); free(h); free(y); free(rowf); free(xq); free(hq); free(qs);
        return NULL;
    }
    for (int r = j->first; r < j->last; ++r) {
        int t = j->tokens[r];
        const uint16_t *xt = j->x + (size_t)t * H;
        double *o = j->out + (size_t)r * H;
        for (int n = 0; n < H; ++n) o[n] = 0.0;
        if (j->w4a4) {  /* the token's activations as NVFP4 (bf16 values are exact in fp32) */
            for (int k = 0; k < H; ++k) rowf[k] = (float)orc_bf16_to_double(xt[k]);
            quant_dequant_row(rowf, H, qs, xq);
        }
        /* one expert of `bank` with routing weight wq: gate_up, SwiGLU, (quantized h), down */
        for (int q = 0; q <= j->k; ++q) {
            const orc_bank *bank;
            int e;
            double wq;
            if (q < j->k) {
                if (!j->routed) continue;
                bank = j->routed;
                e = j->ids[(size_t)t * j->k + q];
                wq = (orc_mutation == ORC_MUT_DROP_ROUTE_W) ? 1.0 : j->w[(size_t)t * j->k + q];
            } else {
                if (!j->shared || orc_mutation == ORC_MUT_DROP_SHARED) continue;
                bank = j->shared;
                e = 0;
                wq = 1.0;
            }
            if (j->w4a4) expert_gate_up_f64(bank, e, xq, G);
            else expert_gate_up(bank, e, xt, G);
            orc_swiglu(G, bank->Il, h);
            if (j->w4a4 && orc_mutation != ORC_MUT_W4A4_NO_H) {  /* h enters down as NVFP4 too, quantized from fp32 */
                for (int i = 0; i < bank->Il; ++i) rowf[i] = (float)h[i];
                quant_dequant_row(rowf, bank->Il, qs, hq);
                expert_down(bank, e, hq, y);
            } else {
                expert_down(bank, e, h, y);
            }
            for (int n = 0; n < H; ++n) o[n] += wq * y[n];
        }
    }
    free(G); free(h); free(y); free(rowf); free(xq); free(hq); free(qs);
    return NULL;
}

/* Rank-local MoE partial for the listed tokens:
 *   out[r][:] = sum_{j<k} w[t][j] * down_e(swiglu(gate_up_e(x_t))) + shared(x_t),
 * with e = ids[t][j], t = tokens[r]; terms added in the order j = 0..k-1, then the
 * shared expert. `routed` or `shared` may be NULL. Tokens are split statically
 * across `nthreads` POSIX threads (each token is independent). Returns 0 or -1. */
static int moe_forward(const orc_bank *routed, const orc_bank *shared, const uint16_t *x, int H,
                       const int32_t *ids, const double *w, int k, const int32_t *tokens, int n_tokens,
                       double *out, int nthreads, int w4a4);

int orc_moe_forward(const orc_bank *routed, const orc_bank *shared, const uint16_t *x, int H,
                    const int32_t *ids, const double *w, int k,
                    const int32_t *tokens, int n_tokens, double *out, int nthreads)
{
    return moe_forward(routed, shared, x, H, ids, w, k, tokens, n_tokens, out, nthreads, 0);
}

/* The W4A4 variant of the same partial: as orc_moe_forward, with the token's activations
 * quantized to NVFP4 (orc_quant_nvfp4, one row per token over H) before gate_up, and each
 * expert's h rounded to fp32 and quantized to NVFP4 (one row per expert and token over the
 * rank's I_l) before down; weights as in the W4A16 layer, sums exact in fp64. Banks must be
 * NVFP4 with H and I_l multiples of 16. */
int orc_moe_forward_w4a4(const orc_bank *routed, const orc_bank *shared, const uint16_t *x, int H,
                         const int32_t *ids, const double *w, int k,
                         const int32_t *tokens, int n_tokens, double *out, int nthreads)
{
    if (H % 16 || (routed && (routed->fmt != 0 || routed->Il % 16)) || (shared && (shared->fmt != 0 || shared->Il % 16)))
        return -1;
    return moe_forward(routed, shared, x, H, ids, w, k, tokens, n_tokens, out, nthreads, 1);
}

static int moe_forward(const orc_bank *routed, const orc_bank *shared, const uint16_t *x, int H,
                       const int32_t *ids, const double *w, int k, const int32_t *tokens, int n_tokens,
                       double *out, int nthreads, int w4a4)
{
    if (n_tokens < 0 || H <= 0 || (routed && (k <= 0 || !ids || !w))) return -1;
    fill_tables();
    if (nthreads < 1) nthreads = 1;
    if (nthreads > n_tokens) nthreads = n_tokens > 0 ? n_tokens : 1;
    fwd_job *jobs = (fwd_job *)calloc((size_t)nthreads, sizeof(fwd_job));
    pthread_t *th = (pthread_t *)calloc((size_t)nthreads, sizeof(pthread_t));
    if (!jobs || !th) { free(jobs); free(th); return -1; }
    int rc = 0;
    for (int i = 0; i < nthreads; ++i) {
        fwd_job *j = &jobs[i];
        j->routed = routed; j->shared = shared; j->x = x; j->ids = ids; j->w = w;
        j->tokens = tokens; j->n_tokens = n_tokens; j->k = k; j->H = H; j->out = out; j->w4a4 = w4a4;
        j->first = (int)((long long)n_tokens * i / nthreads);
        j->last = (int)((long long)n_tokens * (i + 1) / nthreads);
    }
    for (int i = 1; i < nthreads; ++i)
        if (pthread_create(&th[i], NULL, fwd_worker, &jobs[i])) { jobs[i].status = -1; th[i] = 0; }
    fwd_worker(&jobs[0]);
    for (int i = 1; i < nthreads; ++i)
        if (th[i]) pthread_join(th[i], NULL);
    for (int i = 0; i < nthreads; ++i) rc |= jobs[i].status;
    free(jobs); free(th);
    return rc ? -1 : 0;
}
