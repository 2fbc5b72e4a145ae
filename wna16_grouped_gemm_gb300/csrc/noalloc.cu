// Allocation-free entry point: the routed-expert forward with its scratch in a
// fixed, file-scope device array instead of a caller-provided workspace.
//
// Some callers cannot call cudaMalloc (or any allocating routine) once they
// are running: a serving loop whose device memory is entirely owned by
// another allocator, or code on a latency-critical path that must not risk
// the failure or the implicit device synchronisation an allocation can bring.
// They still own and pass every input and output; only the scratch (routing
// lists, permuted activations, h, y, split-K sums) moves into g_scratch below.
#include <cuda.h>
#include <cuda_runtime.h>

#include <mutex>

#include "../../include/wna16_moe.h"
#include "gemm.h"

namespace {

// Largest scratch a call may need; a decode batch of 4 tokens over 256
// experts (hidden 4096, intermediate 2048, top-8) needs under 3 MiB, and
// batches up to roughly 160 tokens of that shape fit.
constexpr size_t kScratchBytes = size_t(32) << 20;

// Every GPU that loads this library holds this array until the process exits.
__device__ __align__(256) unsigned char g_scratch[kScratchBytes];

// Device address of g_scratch per device.  In host code `g_scratch` names a
// host-side stand-in, not device memory, so the address must come from
// cudaGetSymbolAddress, taken with that device current.  The address belongs
// to the device's current context: it is cached together with that context
// and looked up again when the context changes (after cudaDeviceReset, or a
// primary-context reset, the old address is stale).
using CtxGetCurrentFn = CUresult (*)(CUcontext*);

CtxGetCurrentFn ctx_get_current() {
    static CtxGetCurrentFn fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void* p = nullptr;
        cudaDriverEntryPointQueryResult q{};
        if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 12000, cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<CtxGetCurrentFn>(p);
    });
    return fn;
}

std::mutex g_mu;
constexpr int kMaxDevices = 64;
struct ScratchAddr {
    CUcontext ctx = nullptr;
    void* ptr = nullptr;
};
ScratchAddr g_scratch_addr[kMaxDevices];

int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return wna16::set_error(WNA16_ERR_CUDA, "cudaGetDevice: %s", cudaGetErrorString(e));
    if (dev < 0 || dev >= kMaxDevices)
        return wna16::set_error(WNA16_ERR_UNSUPPORTED, "device %d: at most %d devices", dev, kMaxDevices);
    CtxGetCurrentFn get = ctx_get_current();
    if (!get) return wna16::set_error(WNA16_ERR_CUDA, "cuCtxGetCurrent is not available from the driver");
    CUcontext ctx = nullptr;
    if (get(&ctx) != CUDA_SUCCESS) return wna16::set_error(WNA16_ERR_CUDA, "cuCtxGetCurrent failed");
    std::lock_guard<std::mutex> lock(g_mu);
    ScratchAddr& a = g_scratch_addr[dev];
    if (!a.ptr || !ctx || a.ctx != ctx) {
        // (with no current context yet, the runtime makes the device's primary
        // context current here)
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_scratch);
        if (e != cudaSuccess || !p)
            return wna16::set_error(WNA16_ERR_CUDA, "cudaGetSymbolAddress(scratch): %s", cudaGetErrorString(e));
        if (get(&ctx) != CUDA_SUCCESS || !ctx) return wna16::set_error(WNA16_ERR_CUDA, "cuCtxGetCurrent failed");
        a.ctx = ctx;
        a.ptr = p;
    }
    *out = a.ptr;
    return WNA16_OK;
}

}  // namespace

extern "C" int wna16_moe_forward_noalloc(const void* x, const int32_t* topk_ids, const float* topk_weights,
                                         const int32_t* w13_packed, const uint16_t* w13_scales,
                                         const int32_t* w2_packed, const uint16_t* w2_scales, int64_t T, int64_t K,
                                         int64_t N, int64_t E, int topk, int group_size, int group_size_w2, int bits,
                                         float swiglu_limit, void* out, void* stream) {
    const size_t need = wna16_moe_workspace_size(T, K, N, E, topk, bits);
    if (need == 0)   // unsupported sizes: let the regular entry point report exactly why
        return wna16_moe_forward(x, topk_ids, topk_weights, w13_packed, w13_scales, w2_packed, w2_scales, T, K, N, E,
                                 topk, group_size, group_size_w2, bits, swiglu_limit, out, nullptr, 0, stream);
    if (need > kScratchBytes)
        return wna16::set_error(WNA16_ERR_WORKSPACE_TOO_SMALL,
                                "wna16_moe_forward_noalloc: these sizes need %zu bytes of scratch, the static scratch "
                                "holds %zu (use wna16_moe_forward with a workspace)",
                                need, kScratchBytes);
    void* scratch = nullptr;
    if (int rc = scratch_address(&scratch)) return rc;
    return wna16_moe_forward(x, topk_ids, topk_weights, w13_packed, w13_scales, w2_packed, w2_scales, T, K, N, E, topk,
                             group_size, group_size_w2, bits, swiglu_limit, out, scratch, kScratchBytes, stream);
}
