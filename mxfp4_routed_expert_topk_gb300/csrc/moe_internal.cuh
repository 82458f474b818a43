// Internal declarations shared by the library's translation units.
#pragma once

#include <cuda_runtime.h>
#include <cuda_fp16.h>
#include <cuda_bf16.h>
#include <stddef.h>
#include <stdint.h>

#include <atomic>
#include <utility>

#include "../../include/moe.h"

namespace moe {

constexpr int kMaxK = 32;      // slots per row
constexpr int kMaxDecodeRows = 32;
constexpr int kGroupRows = 16; // gate/up interleave granularity in W_gu

// Device-side view of a resident pool (all offsets in bytes within a record).
struct PoolView {
    uint8_t *base;
    uint64_t rec;       // bytes per expert record
    int E, H, I;
    int Ip;             // I rounded up to a multiple of 128 (W_d row length in elements)
    uint64_t off_d;     // W_d codes
    uint64_t off_sgu;   // W_gu scales
    uint64_t off_sd;    // W_d scales
    int ld_gu;          // bytes per W_gu code row  = H/2
    int ld_d;           // bytes per W_d code row   = Ip/2
    int lds_gu;         // scale bytes per W_gu row = H/32
    int lds_d;          // scale bytes per W_d row  = Ip/32
    // the same scale bytes once more in the order of the tensor-core path: for each
    // K tile kt of 128 elements and 128-row tile mt, 512 bytes in which row
    // mt*128 + 32q + l keeps its blocks 4kt..4kt+3 at bytes 16l + 4q + 0..3
    uint64_t off_sgu_mma;  // W_gu: [H/128][nmt_gu][512]
    uint64_t off_sd_mma;   // W_d:  [Ip/128][nmt_d][512]
    int nmt_gu;         // 128-row tiles of W_gu = ceil(2I/128)
    int nmt_d;          // 128-row tiles of W_d  = H/128
};

}  // namespace moe

struct moe_pool {
    moe::PoolView v;
    size_t bytes;
};

namespace moe {

// ------------------------------------------------------------ status word
// The first 256 bytes of every workspace: [0] first error code, [1] detail,
// [2] count of exact-arithmetic fallbacks taken by the router (diagnostic).
struct StatusWord {
    unsigned int code;
    unsigned int detail;
    unsigned int exact_fallbacks;
    unsigned int pad[61];  // kernel counters: see the kSt* slots
};
// Counter slots in StatusWord::pad.  The grid barrier's counter, polled by every
// CTA, sits alone in the second 128-byte line of the word.
constexpr int kStRouteTicket = 0;   // route_single: CTAs done with their logits
constexpr int kStExitCount = 2;     // decode_fused: CTAs past the grid barrier
constexpr int kStGridBarrier = 32;  // decode_fused: grid barrier arrivals (byte 140)

__device__ __forceinline__ void set_status(StatusWord *s, unsigned int code, unsigned int detail) {
    if (s == nullptr) return;
    if (atomicCAS(&s->code, 0u, code) == 0u) s->detail = detail;
}

__host__ __device__ inline size_t align_up(size_t v, size_t a) { return (v + a - 1) / a * a; }

// ---------------------------------------------------------- small helpers

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) {
    return __uint_as_float(((unsigned int)b) << 16);
}

// E8M0 byte -> 2^(b-127) as fp32 (b = 0 gives the subnormal 2^-127, b = 255 NaN).
__device__ __forceinline__ float e8m0_to_float(unsigned int b) {
    float v = __uint_as_float(b << 23);
    v = (b == 0u) ? __uint_as_float(0x00400000u) : v;
    v = (b == 255u) ? __uint_as_float(0x7fc00000u) : v;
    return v;
}

// Four packed bytes of E2M1 pairs -> four f16x2 (low nibble -> low half).
__device__ __forceinline__ void e2m1x8_to_f16x2x4(unsigned int q, unsigned int &h0, unsigned int &h1,
                                                   unsigned int &h2, unsigned int &h3) {
    asm("{\n\t.reg .b8 a0, a1, a2, a3;\n\t"
        "mov.b32 {a0, a1, a2, a3}, %4;\n\t"
        "cvt.rn.f16x2.e2m1x2 %0, a0;\n\t"
        "cvt.rn.f16x2.e2m1x2 %1, a1;\n\t"
        "cvt.rn.f16x2.e2m1x2 %2, a2;\n\t"
        "cvt.rn.f16x2.e2m1x2 %3, a3;\n\t}"
        : "=r"(h0), "=r"(h1), "=r"(h2), "=r"(h3)
        : "r"(q));
}

__device__ __forceinline__ unsigned int hfma2_u32(unsigned int a, unsigned int b, unsigned int c) {
    unsigned int d;
    asm("fma.rn.f16x2 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
    return d;
}

__device__ __forceinline__ float f16x2_sum_to_float(unsigned int v) {
    __half2 h = *reinterpret_cast<__half2 *>(&v);
    return __low2float(h) + __high2float(h);
}

// 16-byte streaming load that does not allocate in L1.
__device__ __forceinline__ uint4 ldg_stream16(const void *p) {
    uint4 r;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
                 : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
                 : "l"(p));
    return r;
}

__device__ __forceinline__ unsigned char ldg_stream_u8(const void *p) {
    unsigned short r;
    asm volatile("ld.global.nc.L1::no_allocate.u8 %0, [%1];" : "=h"(r) : "l"(p));
    return (unsigned char)r;
}

// Kernel tracing (api.cu): bracket one launch of kernel `name` with events.
void trace_pre(const char *name, cudaStream_t st);
void trace_post(const char *name, cudaStream_t st);

// Programmatic dependent launch: a kernel launched with programmatic stream
// serialization may start while the previous kernel in the stream finishes; this
// waits until that kernel has completed and its memory is visible (a no-op for a
// kernel launched without the attribute).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }

// Let the next kernel of the stream (launched with programmatic stream serialization)
// start once every CTA of this grid has called this or exited; it still waits, in
// griddep_wait, for this grid to complete before it reads what this grid writes.
__device__ __forceinline__ void griddep_launch_dependents() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Launch `kernel` on `st` with programmatic stream serialization: its CTAs may be
// scheduled once every CTA of the previous kernel of the stream has let them
// (griddepcontrol.launch_dependents) or exited, and it must execute
// griddepcontrol.wait before it reads anything that kernel writes.  (Dependents start
// only after all of the previous grid's CTAs are running, so they never keep it from
// finishing.)
template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem, cudaStream_t st,
                              Args &&...args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

struct TraceScope {
    const char *name;
    cudaStream_t st;
    TraceScope(const char *n, cudaStream_t s) : name(n), st(s) { trace_pre(name, st); }
    ~TraceScope() { trace_post(name, st); }
};

// Values the library caches per device: device attributes and each kernel's raised
// dynamic shared-memory limit (a function attribute belongs to one device), so that
// one process may use several devices.  Entries are atomics: host threads making
// their first calls on a device at the same time store the same value.
constexpr int kMaxDevices = 64;
struct PerDevice {
    std::atomic<int> v[kMaxDevices];
    explicit PerDevice(int init) {
        for (auto &a : v) a.store(init, std::memory_order_relaxed);
    }
};

inline cudaError_t current_device(int *dev) {
    cudaError_t e = cudaGetDevice(dev);
    if (e != cudaSuccess) return e;
    return (*dev >= 0 && *dev < kMaxDevices) ? cudaSuccess : cudaErrorInvalidDevice;
}

// Attribute `attr` of the current device, read once per device (cache: init 0).
inline cudaError_t device_attr(cudaDeviceAttr attr, PerDevice &cache, int *out) {
    int dev = 0;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    int v = cache.v[dev].load(std::memory_order_relaxed);
    if (v == 0) {
        e = cudaDeviceGetAttribute(&v, attr, dev);
        if (e != cudaSuccess) return e;
        cache.v[dev].store(v, std::memory_order_relaxed);
    }
    *out = v;
    return cudaSuccess;
}

// Raise a kernel's dynamic shared memory limit on the current device to `bytes` if
// needed (per kernel and device, remembered in `cur`, init 0).  Returns the error of
// the attribute call.
template <typename K>
inline cudaError_t ensure_dynamic_smem(K kernel, size_t bytes, PerDevice &cur) {
    if (bytes <= 48 * 1024) return cudaSuccess;
    int dev = 0;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    if ((int)bytes <= cur.v[dev].load(std::memory_order_relaxed)) return cudaSuccess;
    e = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
    if (e == cudaSuccess) {
        int old = cur.v[dev].load(std::memory_order_relaxed);
        while (old < (int)bytes && !cur.v[dev].compare_exchange_weak(old, (int)bytes, std::memory_order_relaxed)) {
        }
    }
    return e;
}

// Launch helpers implemented per translation unit.
cudaError_t launch_pool_kernel(const PoolView &v, int mode, uint64_t seed, int e_lo, int e_hi,
                               const uint8_t *codes, const uint8_t *scales, uint8_t *out_codes,
                               uint8_t *out_scales, cudaStream_t st);

size_t route_workspace_bytes(int E, int M, int k);
// xhat != nullptr: route x_hat = prescale(x) (the exact power-of-two pre-scale of
// launch_prescale) and write it to xhat.
cudaError_t launch_route(const uint16_t *x, int M, int H, const uint16_t *Wr, int E, const float *skew,
                         int k, int32_t *idx, float *w, void *ws, cudaStream_t st, uint16_t *xhat = nullptr);

size_t decode_workspace_bytes(int E, int H, int I, int M, int k);
// The single-token fused decode runs at most this many CTAs; its workspace holds
// h [k][I] after the status word.
constexpr int kMaxFusedGrid = 1024;
inline size_t decode_fused_workspace_bytes(int I, int k) { return 256 + align_up((size_t)k * I * sizeof(float), 256); }
cudaError_t launch_decode(const PoolView &v, const uint16_t *x, int M, const int32_t *idx, const float *w,
                          int k, const uint16_t *residual, uint16_t *y, void *ws, cudaStream_t st);

// Single-token fused decode; cudaErrorNotSupported when the shape does not allow it.
cudaError_t launch_decode_fused(const PoolView &v, const uint16_t *x, const int32_t *idx, const float *w, int k,
                                const uint16_t *residual, uint16_t *y, void *ws, cudaStream_t st);

cudaError_t launch_prescale(const uint16_t *x, int M, int H, uint16_t *out, cudaStream_t st);

// Test support (moe_debug_*): the wait limit of the translation units whose kernels
// wait, and extra arrivals the fused decode kernel's grid barrier waits for.
cudaError_t set_wait_limit_decode_fused(uint64_t ns);
cudaError_t set_wait_limit_gemm(uint64_t ns);
void set_barrier_extra(unsigned int extra);
void set_cta_pairs(int mode);  // grouped GEMMs on CTA pairs: 0 never, 1 always, 2 MXFP8 rows only

size_t grouped_workspace_bytes(int E, int H, int I, int T, int k);
cudaError_t launch_grouped(const PoolView &v, const uint16_t *x, int T, const int32_t *idx, int k,
                           int act_mode, int32_t *perm, int32_t *inv_perm, int32_t *offsets,
                           void *partial, int partial_dtype, void *ws, cudaStream_t st);
cudaError_t launch_combine(const void *partial, int partial_dtype, const int32_t *inv_perm, const float *w,
                           int T, int k, int H, const uint16_t *residual, uint16_t *y, cudaStream_t st);
// Diagnostics: the MXFP8 h of the last grouped call on `ws`, in sorted row order.
cudaError_t launch_read_h(const PoolView &v, int T, int k, int act_mode, const int32_t *offsets, const void *ws,
                          uint8_t *hq, uint8_t *hs, cudaStream_t st);

}  // namespace moe
