// moe_route_topk_static: the router for callers that cannot allocate device memory.
//
// Some callers cannot call cudaMalloc or hand the library a workspace: code that
// runs while a caching allocator or a host framework owns all device memory,
// plugins whose host gives them no scratch buffers, and latency-critical threads
// that must not risk the device-wide synchronisation cudaMalloc/cudaFree can
// trigger.  This entry point runs the same two router kernels as moe_route_topk,
// with their scratch (status word, fp32 logits and error bounds) in the
// file-scope device array below instead of a caller workspace.
#include <string.h>

#include "moe_internal.cuh"

namespace {

// Largest M * E this entry point accepts (1 MiB of logits and bounds).
constexpr size_t kStaticRouteMaxME = 131072;
// logits and bounds, plus the row norms of x and W_r (at most kStaticRouteMaxME + 4096)
constexpr size_t kStaticScratchBytes = 256 + 2 * kStaticRouteMaxME * sizeof(float) +
                                       (kStaticRouteMaxME + 4096) * sizeof(float) + 1024;
// Every GPU that loads this library holds this array until the process exits.
__device__ __align__(256) unsigned char g_route_scratch[kStaticScratchBytes];

// Device address of g_route_scratch per device, looked up once per device.  Atomic
// entries: two host threads making their first call on one device at the same time
// both look the address up and store the same value.
std::atomic<void *> g_scratch_ptr[moe::kMaxDevices];

cudaError_t scratch_for_current_device(void **out) {
    int dev = 0;
    cudaError_t e = moe::current_device(&dev);
    if (e != cudaSuccess) return e;
    void *p = g_scratch_ptr[dev].load(std::memory_order_relaxed);
    if (p == nullptr) {
        // The symbol's host-side name is only a stand-in; the kernels need the
        // device address, valid for the current device.
        e = cudaGetSymbolAddress(&p, g_route_scratch);
        if (e != cudaSuccess) return e;
        g_scratch_ptr[dev].store(p, std::memory_order_relaxed);
    }
    *out = p;
    return cudaSuccess;
}

}  // namespace

extern "C" moe_status moe_route_topk_static(const uint16_t *x, int M, int H, const uint16_t *Wr, int E,
                                            const float *skew, int k, int32_t *idx, float *w,
                                            moe_stream_t stream) {
    if (M < 0 || x == nullptr || Wr == nullptr || idx == nullptr || w == nullptr) return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > moe::kMaxK || k > E) return MOE_ERR_INVALID_ARG;
    if (E > 4096 || H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (((uintptr_t)x % 16) != 0 || ((uintptr_t)Wr % 16) != 0) return MOE_ERR_INVALID_ARG;
    if ((size_t)M * (size_t)E > kStaticRouteMaxME) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (moe::route_workspace_bytes(E, M, k) > kStaticScratchBytes) return MOE_ERR_UNSUPPORTED_SHAPE;
    void *scratch = nullptr;
    if (scratch_for_current_device(&scratch) != cudaSuccess) return MOE_ERR_CUDA;
    cudaStream_t st = (cudaStream_t)stream;
    // The status word must start at zero; logits and bounds are rewritten in full.
    if (cudaMemsetAsync(scratch, 0, sizeof(moe::StatusWord), st) != cudaSuccess) return MOE_ERR_CUDA;
    return moe::launch_route(x, M, H, Wr, E, skew, k, idx, w, scratch, st) == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
