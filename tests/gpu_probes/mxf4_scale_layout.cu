// Layout check for tcgen05.mma kind::mxf4nvf4 block_scale scale_vec::4X (M = 128, N = 128,
// K = 64), the layout the W4A4 kernels write their scales in: which tensor-memory (lane,
// column, byte) holds the scale of row m (A) or column n (B) for K block b. Each of 32 single
// MMAs has nonzero codes (1.0) in one 16-element block only and all other scales 1.0; every
// scale byte of the probed operand is a distinct power of two encoding its position, so each
// fp32 output (16 x the scale read) decodes which byte was used. Test infrastructure.
#include <cstdio>
#include <cstdint>
#include <cmath>
#include <cuda_runtime.h>

__device__ __forceinline__ uint32_t smem_u32(const void *p) { return (uint32_t)__cvta_generic_to_shared(p); }

__device__ __forceinline__ uint8_t e4m3_pow2(int e)  // 2^e, e in [-9, 6]
{
    if (e >= -6) return (uint8_t)((e + 7) << 3);
    return (uint8_t)(1 << (e + 9));  // -7 -> 4, -8 -> 2, -9 -> 1
}

__device__ __forceinline__ uint64_t sw128_desc(uint32_t a)
{
    uint64_t d = 0;
    d |= (uint64_t)((a & 0x3FFFFu) >> 4);
    d |= (uint64_t)1 << 16;
    d |= (uint64_t)(1024 >> 4) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)2 << 61;
    return d;
}

constexpr int NPROBE = 32;
constexpr uint32_t kSfaCol = 128, kSfbCol = 192, kSfCols = 16;

// per probe: side (0: A encoded, 1: B encoded), block b0, encoding enc
__global__ void __launch_bounds__(128, 1) probe(float *out, int *status)
{
    __shared__ __align__(1024) uint8_t A[128 * 128];
    __shared__ __align__(1024) uint8_t B[128 * 128];
    __shared__ __align__(8) uint64_t bar;
    __shared__ uint32_t tmem_base;
    const int t = threadIdx.x, warp = t >> 5;
    if (warp == 0) {
        asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(&tmem_base)), "r"(256));
        asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;");
    }
    if (t == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(&bar)), "r"(1));
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
    __syncthreads();
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    const uint32_t tmem = tmem_base;
    const uint32_t idesc = (1u << 7) | (1u << 10) | ((128u >> 3) << 17) | ((128u >> 4) << 24);
    bool dead = false;
    for (int p = 0; p < NPROBE && !dead; ++p) {
        const int side = p / 16, b0 = (p / 4) % 4, enc = p % 4;
        // codes: row t of A and of B, 32 logical bytes (K = 64) in the 128-byte swizzled row
        for (int j = 0; j < 128; ++j) {
            const int q = j >> 4, phys = t * 128 + ((q ^ (t & 7)) << 4) + (j & 15);
            const bool in_k = j < 32;
            const bool in_b0 = j >= 8 * b0 && j < 8 * b0 + 8;
            A[phys] = in_k && (side == 0 ? in_b0 : true) ? 0x22 : 0;
            B[phys] = in_k && (side == 1 ? in_b0 : true) ? 0x22 : 0;
        }
        // scales: this thread's TMEM lane t, kSfCols columns of A's and of B's regions
        uint32_t sa[kSfCols], sb[kSfCols];
        for (int j = 0; j < (int)kSfCols; ++j) {
            uint32_t enc_word = 0;
            for (int y = 0; y < 4; ++y) {
                int f = enc == 0 ? j : enc == 1 ? y : enc == 2 ? (t % 16) : (t / 8);
                enc_word |= (uint32_t)e4m3_pow2(f - 9) << (8 * y);
            }
            const uint32_t one = 0x38383838u;
            sa[j] = side == 0 ? enc_word : one;
            sb[j] = side == 1 ? enc_word : one;
        }
        const uint32_t lane_addr = tmem + ((uint32_t)(32 * warp) << 16);
        asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                     ::"r"(lane_addr + kSfaCol), "r"(sa[0]), "r"(sa[1]), "r"(sa[2]), "r"(sa[3]), "r"(sa[4]), "r"(sa[5]),
                     "r"(sa[6]), "r"(sa[7]), "r"(sa[8]), "r"(sa[9]), "r"(sa[10]), "r"(sa[11]), "r"(sa[12]), "r"(sa[13]),
                     "r"(sa[14]), "r"(sa[15]) : "memory");
        asm volatile("tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
                     ::"r"(lane_addr + kSfbCol), "r"(sb[0]), "r"(sb[1]), "r"(sb[2]), "r"(sb[3]), "r"(sb[4]), "r"(sb[5]),
                     "r"(sb[6]), "r"(sb[7]), "r"(sb[8]), "r"(sb[9]), "r"(sb[10]), "r"(sb[11]), "r"(sb[12]), "r"(sb[13]),
                     "r"(sb[14]), "r"(sb[15]) : "memory");
        asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        if (t == 0) {
            const uint64_t ad = sw128_desc(smem_u32(A)), bd = sw128_desc(smem_u32(B));
            asm volatile(
                "{\n\t.reg .pred pp;\n\tsetp.ne.b32 pp, %6, 0;\n\t"
                "tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], pp;\n\t}"
                ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(tmem + kSfaCol), "r"(tmem + kSfbCol), "r"(0) : "memory");
            asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(&bar)) : "memory");
        }
        // bounded wait for phase p & 1
        uint32_t ok = 0;
        for (long it = 0; it < 20000000 && !ok; ++it) {
            asm volatile("{\n\t.reg .pred q;\n\tmbarrier.try_wait.parity.shared::cta.b64 q, [%1], %2;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                         : "=r"(ok) : "r"(smem_u32(&bar)), "r"((uint32_t)(p & 1)) : "memory");
        }
        if (!__all_sync(0xFFFFFFFFu, ok)) { if (t == 0) atomicExch(status, 1); }
        __syncthreads();
        if (*(volatile int *)status) { dead = true; break; }
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
        for (int c0 = 0; c0 < 128; c0 += 16) {
            uint32_t r[16];
            asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
                         : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                           "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
                         : "r"(lane_addr + c0));
            asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
            for (int i = 0; i < 16; ++i) out[((size_t)p * 128 + t) * 128 + c0 + i] = __uint_as_float(r[i]);
        }
        asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
        __syncthreads();
        asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
    }
    __syncthreads();
    if (warp == 0) asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "r"(256));
}

static int decode(float v)  // f with v = 16 * 2^(f - 9), or -99
{
    if (!(v > 0)) return -99;
    double f = std::log2(v / 16.0) + 9.0;
    double r = std::round(f);
    return std::fabs(f - r) < 1e-6 ? (int)r : -99;
}

int main()
{
    float *d_out;
    int *d_st;
    if (cudaMalloc(&d_out, sizeof(float) * NPROBE * 128 * 128) != cudaSuccess) return 2;
    if (cudaMalloc(&d_st, sizeof(int)) != cudaSuccess) return 2;
    cudaMemset(d_out, 0, sizeof(float) * NPROBE * 128 * 128);
    cudaMemset(d_st, 0, sizeof(int));
    probe<<<1, 128>>>(d_out, d_st);
    cudaError_t e = cudaDeviceSynchronize();
    printf("kernel: %s\n", cudaGetErrorString(e));
    if (e != cudaSuccess) return 1;
    int st = 0;
    cudaMemcpy(&st, d_st, sizeof(int), cudaMemcpyDeviceToHost);
    if (st) { printf("a wait ran out\n"); return 1; }
    static float h[NPROBE * 128 * 128];
    cudaMemcpy(h, d_out, sizeof(h), cudaMemcpyDeviceToHost);
    auto at = [&](int p, int m, int n) { return h[((size_t)p * 128 + m) * 128 + n]; };
    // expected: A row m, block b -> lane m, column m / 32, byte b (for every output column);
    //           B column n, block b, output row m -> lane 32 (m / 32) + n % 32, column n / 32, byte b
    long bad_a = 0, bad_b = 0;
    for (int b0 = 0; b0 < 4; ++b0)
        for (int m = 0; m < 128; ++m)
            for (int n = 0; n < 128; ++n) {
                for (int side = 0; side < 2; ++side) {
                    int f[4];
                    for (int enc = 0; enc < 4; ++enc) f[enc] = decode(at(side * 16 + b0 * 4 + enc, m, n));
                    const int x = side ? n : m;
                    const int lane = side ? 32 * (m / 32) + n % 32 : m;
                    const bool ok = f[0] == x / 32 && f[1] == b0 && f[2] == lane % 16 && f[3] == lane / 8;
                    if (!ok) (side ? bad_b : bad_a)++;
                }
            }
    printf("A mismatches %ld\nB mismatches %ld\n", bad_a, bad_b);
    printf(bad_a == 0 && bad_b == 0 ? "LAYOUT OK\n" : "LAYOUT DIFFERS\n");
    return 0;
}
