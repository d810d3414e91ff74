// Device-side building blocks shared by the libftmoe kernels (sm_103a).
//
// The NVFP4 weight element is W[n][k] = e2m1(code) * e4m3(scale[n][k/group]) *
// global[n] (bank layout of the NVFP4 expert kernel, "[TP=2] Quantized MoE expert
// parallelism ... NVFP4 port", section 4). The kernels feed the tensor cores with the
// exact bf16 value code*scale and apply global[n] to the fp32 accumulator of row n,
// which is the same sum (the global is constant along k).
#pragma once

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "ft_moe.h"

namespace ftmoe {

constexpr int kWarp = 32;

// First error wins; later errors leave the first one in place.
__device__ __forceinline__ void raise_status(int *status, int code)
{
    if (status) atomicCAS(status, 0, code);
}

// ---------------------------------------------------------------- dequantisation

// Four packed code bytes (eight e2m1 codes, element 2m in the low nibble of byte m)
// -> four f16x2 registers holding the exact code values, lower element in the lower
// half. cvt.rn.f16x2.e2m1x2 is exact: every e2m1 value is an f16 value.
__device__ __forceinline__ void e2m1x8_to_f16x2(uint32_t codes, uint32_t (&f)[4])
{
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "mov.b32 {q0, q1, q2, q3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, q0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, q1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, q2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, q3;\n\t}"
        : "=r"(f[0]), "=r"(f[1]), "=r"(f[2]), "=r"(f[3])
        : "r"(codes));
}

// f16x2 holding e2m1 code values -> bf16x2 holding code * 2^-112, exactly.
// An f16 normal 2^(E-15)(1+M/1024) whose low three mantissa bits are zero (true for
// every e2m1 value) re-read with its exponent field E in the low bits of a bf16
// exponent and M>>3 as the bf16 mantissa is 2^(E-127)(1+M/1024) = value * 2^-112.
// Zero maps to zero and the sign bit stays in place.
__device__ __forceinline__ uint32_t f16x2_codes_to_bf16x2_scaled(uint32_t f)
{
    return ((f & 0x7FFF7FFFu) >> 3) | (f & 0x80008000u);
}

__device__ __forceinline__ uint32_t bf16x2_mul(uint32_t a, uint32_t b)
{
    uint32_t d;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
    return d;
}

// Two e4m3 scale bytes (low byte = first) -> two bf16x2 registers, each holding the
// scale * 2^112 in both halves (exact: <= 4 significant bits, inside bf16 range).
__device__ __forceinline__ void e4m3x2_to_bf16x2_scaled(uint32_t two_bytes, uint32_t &s0, uint32_t &s1)
{
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
        : "=r"(h2)
        : "r"(two_bytes));
    __half2 hh = *reinterpret_cast<__half2 *>(&h2);
    float f0 = __low2float(hh) * 0x1p112f;
    float f1 = __high2float(hh) * 0x1p112f;
    __nv_bfloat16 b0 = __float2bfloat16_rn(f0), b1 = __float2bfloat16_rn(f1);
    uint32_t u0 = *reinterpret_cast<uint16_t *>(&b0), u1 = *reinterpret_cast<uint16_t *>(&b1);
    s0 = u0 | (u0 << 16);
    s1 = u1 | (u1 << 16);
}

// Eight codes sharing one scale -> four bf16x2 registers of exact code*scale values.
__device__ __forceinline__ void dequant8(uint32_t codes, uint32_t scale_bf16x2, uint32_t (&out)[4])
{
    uint32_t f[4];
    e2m1x8_to_f16x2(codes, f);
#pragma unroll
    for (int i = 0; i < 4; ++i) out[i] = bf16x2_mul(f16x2_codes_to_bf16x2_scaled(f[i]), scale_bf16x2);
}

// Two e4m3 scale bytes (low byte = first) -> two f16x2 registers, each holding one
// scale in both halves (every e4m3 value is an f16 value).
__device__ __forceinline__ void e4m3x2_to_f16x2_bcast(uint32_t two_bytes, uint32_t &s0, uint32_t &s1)
{
    uint32_t h2;
    asm("{\n\t.reg .b16 t;\n\tcvt.u16.u32 t, %1;\n\tcvt.rn.f16x2.e4m3x2 %0, t;\n\t}"
        : "=r"(h2)
        : "r"(two_bytes));
    s0 = __byte_perm(h2, 0, 0x1010);
    s1 = __byte_perm(h2, 0, 0x3232);
}

// Eight codes sharing one scale -> four f16x2 registers of exact code*scale values:
// |code*scale| lies in [2^-10, 2688] with at most 6 significant bits, so the f16
// product is exact.
__device__ __forceinline__ void dequant8_f16(uint32_t codes, uint32_t scale_f16x2, uint32_t (&out)[4])
{
    uint32_t f[4];
    e2m1x8_to_f16x2(codes, f);
#pragma unroll
    for (int i = 0; i < 4; ++i) asm("mul.rn.f16x2 %0, %1, %2;" : "=r"(out[i]) : "r"(f[i]), "r"(scale_f16x2));
}

// ---------------------------------------------------------------- dependent launch

// Every kernel of the library starts with pdl_wait(): it returns once the kernels before
// it in the stream have completed and their memory is visible, so a kernel launched
// early (programmatic dependent launch) never reads or overwrites what they still use.
// pdl_trigger() then lets the next kernel's CTAs be scheduled while this one runs.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }
__device__ __forceinline__ void pdl_enter()
{
    pdl_wait();
    pdl_trigger();
}

// ---------------------------------------------------------------- activation row scaling

// 2^e for integer e in [-126, 127], built from its bits (exact).
__device__ __forceinline__ float pow2f(int e) { return __int_as_float((127 + e) << 23); }

// Row scale exponent e for a row whose largest magnitude is m: m * 2^-e lies in
// [2^14, 2^15), clamped to [-126, 127] so that 2^e and 2^-e stay finite normals;
// zero and non-finite rows keep e = 0.
__device__ __forceinline__ int row_scale_exp(float m)
{
    if (!(m > 0.f && m <= 3.3895314e38f)) return 0;
    return min(max(ilogbf(m) - 14, -126), 127);
}

// ---------------------------------------------------------------- warp MMA

// D(16x8, f32) += A(16x16, f16, row) * B(16x8, f16, col).
__device__ __forceinline__ void mma_f16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                              uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

// D(16x8, f32) += A(16x16, bf16, row) * B(16x8, bf16, col).
__device__ __forceinline__ void mma_bf16_16816(float (&d)[4], uint32_t a0, uint32_t a1, uint32_t a2,
                                               uint32_t a3, uint32_t b0, uint32_t b1)
{
    asm volatile(
        "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
        "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
        : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
        : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
}

__device__ __forceinline__ uint2 ldg_nc_v2(const void *p)
{
    uint2 v;
    asm volatile("ld.global.nc.L1::no_allocate.v2.u32 {%0, %1}, [%2];"
                 : "=r"(v.x), "=r"(v.y)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_nc_v4(const void *p)
{
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

__device__ __forceinline__ uint4 ldg_v4(const void *p)
{
    return __ldg(reinterpret_cast<const uint4 *>(p));
}

// ---------------------------------------------------------------- routing-derived indices

// In a bounds-checking build (FTMOE_BOUNDS_CHECK defined) every index a kernel derives from
// the routing tables is checked before it addresses memory; a bad one sets FT_ERR_BOUNDS in
// the status word (first error wins) and is replaced by a harmless one. In the regular
// build these return their argument.
#ifdef FTMOE_BOUNDS_CHECK
__device__ __forceinline__ void bounds_error(int *status) { raise_status(status, FT_ERR_BOUNDS); }
// An expert id for addressing an expert's bank: in [0, E), else expert 0.
__device__ __forceinline__ int chk_expert(int e, int E, int *status)
{
    if (e >= 0 && e < E) return e;
    bounds_error(status);
    return 0;
}
// A slot read from the sorted order: >= n_slots marks padding; negative is an error, read as padding.
__device__ __forceinline__ int chk_slot(int sl, int n_slots, int *status)
{
    if (sl >= 0) return sl;
    bounds_error(status);
    return n_slots;
}
// A padded position count: a multiple of the block within the buffers' capacity, else 0.
__device__ __forceinline__ int chk_count(int n, int block, int cap, int *status)
{
    if (n >= 0 && n <= cap && n % block == 0) return n;
    bounds_error(status);
    return 0;
}
#else
__device__ __forceinline__ int chk_expert(int e, int, int *) { return e; }
__device__ __forceinline__ int chk_slot(int sl, int, int *) { return sl; }
__device__ __forceinline__ int chk_count(int n, int, int, int *) { return n; }
#endif
// Capacity of the padded positions of n_slots slots over E experts in blocks of B.
__host__ __device__ __forceinline__ int padded_capacity(int n_slots, int E, int B)
{
    return n_slots + (n_slots < E ? n_slots : E) * (B - 1);
}

// silu(z) = z / (1 + e^-z) with the fast exponential and division: relative error of a
// few 1e-7 for |z| < 64, far below the bf16 rounding of h that follows. For z < -88
// the denominator is +inf and the result -0; for large z it is z.
__device__ __forceinline__ float silu(float z) { return __fdividef(z, 1.0f + __expf(-z)); }

// ---------------------------------------------------------------- mbarrier + bulk copy

__device__ __forceinline__ uint32_t smem_u32(const void *p)
{
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count)
{
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count));
}

// Make barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void fence_mbar_init()
{
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

// Order this thread's earlier generic-proxy shared-memory accesses before later
// async-proxy accesses (a bulk copy that overwrites data just read).
__device__ __forceinline__ void fence_proxy_async_smem()
{
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes)
{
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
                 : "memory");
}

// Global -> shared bulk copy (16-byte aligned addresses, size a multiple of 16) that
// signals `bar` with its byte count on completion.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar)
{
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar))
        : "memory");
}

// Per-thread asynchronous global -> shared copies (L2 only), grouped by commit.
__device__ __forceinline__ void cp_async_16(void *dst, const void *src)
{
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_8(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 8;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_4(void *dst, const void *src)
{
    asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(smem_u32(dst)), "l"(src) : "memory");
}

__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }

template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Bounded wait for phase `parity` of `bar`: false after `limit` polls (the caller then
// records FT_ERR_TIMEOUT and winds down instead of spinning forever).
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t *bar, uint32_t parity, uint32_t limit)
{
    for (uint32_t i = 0; i < limit; ++i)
        if (mbar_try_wait(bar, parity)) return true;
    return false;
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar)
{
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}

__device__ __forceinline__ uint64_t globaltimer()
{
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Default limit of every mbarrier wait in the pipelined kernels: about two seconds (a
// launch may pass a shorter one, see ft_moe_debug_inject_stall).
constexpr uint64_t kWaitNs = 2000000000ull;

// try_wait that lets the hardware suspend the thread for up to `hint_ns` nanoseconds
// while the phase is incomplete (it resumes as soon as the phase completes), so that
// waiting warps do not spin on the issue slots the math warps need.
__device__ __forceinline__ bool mbar_try_wait_hint(uint64_t *bar, uint32_t parity, uint32_t hint_ns)
{
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, %3;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity), "r"(hint_ns)
        : "memory");
    return ok != 0;
}

// Wait for phase `parity` of `bar`: false after limit_ns nanoseconds (about two seconds
// by default), or as soon as another role of the CTA has set *abort_flag (non-null)
// after giving up itself.
// After one plain poll the thread parks in try_wait with a suspend-time hint: the hardware
// resumes it when the phase completes (or after the hint), so a waiting warp takes no issue
// slots from the warps that have work. (Spinning on plain polls instead, the epilogue,
// producer and MMA warps of the tensor-core kernels starved their dequantising warps.)
constexpr uint32_t kSuspendHintNs = 1000;

__device__ __forceinline__ bool mbar_wait_timed(uint64_t *bar, uint32_t parity, volatile int *abort_flag,
                                                uint64_t limit_ns = kWaitNs)
{
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = globaltimer();
    for (;;) {
        if (mbar_try_wait_hint(bar, parity, kSuspendHintNs)) return true;
        if (abort_flag && *abort_flag) return false;
        if (globaltimer() - t0 > limit_ns) return false;
    }
}

__device__ __forceinline__ uint32_t lanemask_lt()
{
    uint32_t m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

}  // namespace ftmoe
