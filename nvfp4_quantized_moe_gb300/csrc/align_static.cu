// ft_moe_align_static: moe_align with library-owned scratch, for callers that must not
// allocate device memory: an engine that plans every device byte at start-up and forbids
// allocation afterwards, or a caller whose device memory is fixed by someone else (a
// shared arena it may not grow). Their only device memory is the inputs and outputs they
// already own. The scratch that the multi-pass sort needs (per-chunk expert counts,
// per-slot ranks) and the status word live in one file-scope array that every GPU
// loading this library keeps until the process exits. The entry point still issues CUDA
// calls (a memset, kernel launches, a device-to-device copy), so it cannot be called
// where the CUDA API is off limits, such as inside a stream host callback.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "ft_moe.h"
#include "ftmoe_internal.h"

namespace ftmoe {

namespace {

constexpr int kStaticMaxSlots = 65536;  // T * k
constexpr int kStaticMaxExperts = 1024;
constexpr size_t kStatusBytes = 256;
constexpr size_t kChunkCountBytes =
    ((size_t)(kStaticMaxSlots + kAlignChunk - 1) / kAlignChunk * kStaticMaxExperts * sizeof(int) + 255) / 256 * 256;
constexpr size_t kRankBytes = ((size_t)kStaticMaxSlots * sizeof(int) + 255) / 256 * 256;
constexpr size_t kScratchBytes = kStatusBytes + kChunkCountBytes + kRankBytes;  // 393,472 bytes

// Status word at offset 0, then the align scratch.
static __device__ __align__(256) unsigned char g_align_scratch[kScratchBytes];

typedef CUresult (*CtxGetCurrentFn)(CUcontext *);

// cuCtxGetCurrent through the runtime's driver entry point (no link against libcuda).
CtxGetCurrentFn ctx_get_current()
{
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &ptr, 12000, cudaEnableDefault, &q) ==
                cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(ptr);
    });
    return fn;
}

std::mutex g_scratch_mu;
struct ScratchEntry {
    CUcontext ctx;
    void *addr;
};
ScratchEntry g_scratch_addr[64];  // per device ordinal: the context it was looked up in

// Device address of g_align_scratch in the current device's context. Looked up once per
// device and context with that device current (the host-side symbol is only a stand-in
// and must never reach a kernel); a new context on the device (after cudaDeviceReset)
// looks it up again, since the module and its array may then sit elsewhere.
cudaError_t scratch_address(void **out)
{
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    CtxGetCurrentFn get = ctx_get_current();
    if (!get) return cudaErrorInitializationError;
    CUcontext ctx = nullptr;  // null until the runtime has bound a context to this thread
    if (get(&ctx) != CUDA_SUCCESS) return cudaErrorInitializationError;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    ScratchEntry &slot = g_scratch_addr[dev];
    if (!ctx || !slot.addr || slot.ctx != ctx) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_align_scratch);  // binds the device's primary context
        if (e != cudaSuccess) return e;
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return cudaErrorInitializationError;
        slot.ctx = ctx;
        slot.addr = p;
    }
    *out = slot.addr;
    return cudaSuccess;
}

}  // namespace

}  // namespace ftmoe

using namespace ftmoe;

extern "C" ft_status ft_moe_align_static(const int32_t *topk_ids, int32_t T, int32_t k, int32_t E, int32_t block,
                                         int32_t *sorted_slot, int32_t *block_expert, int32_t *expert_off,
                                         int32_t *n_padded, int32_t *status, void *stream)
{
    FT_NVTX_RANGE("ft_moe_align_static");
    if (T < 0 || k <= 0 || E <= 0 || block < 1 || block > 1024)
        return report_error(FT_ERR_INVALID_ARG, "need T >= 0, k > 0, E > 0, 1 <= block <= 1024");
    if (k > 32 || E > kStaticMaxExperts || (int64_t)T * k > kStaticMaxSlots)
        return report_error(FT_ERR_UNSUPPORTED,
                            "ft_moe_align_static handles at most 65536 slots (T*k), 1024 experts and top_k 32; "
                            "use ft_moe_align with a caller workspace for larger inputs");
    if (!sorted_slot || !block_expert || !expert_off || !n_padded || (T > 0 && !topk_ids))
        return report_error(FT_ERR_INVALID_ARG, "align pointers must be non-NULL");
    void *scratch = nullptr;
    cudaError_t e = scratch_address(&scratch);
    if (e != cudaSuccess) return report_error(FT_ERR_CUDA, cudaGetErrorString(e));
    cudaStream_t s = static_cast<cudaStream_t>(stream);
    int *dev_status = static_cast<int *>(scratch);
    e = cudaMemsetAsync(dev_status, 0, sizeof(int), s);  // the status word must start at FT_OK
    if (e == cudaSuccess)
        e = launch_align(topk_ids, T, k, E, block, sorted_slot, block_expert, expert_off, n_padded, dev_status,
                         static_cast<char *>(scratch) + kStatusBytes, s);
    if (e == cudaSuccess && status)
        e = cudaMemcpyAsync(status, dev_status, sizeof(int), cudaMemcpyDeviceToDevice, s);
    if (e != cudaSuccess) return report_error(FT_ERR_CUDA, cudaGetErrorString(e));
    return report_error(FT_OK, "");
}
