// The extern "C" entry points of include/moe.h: argument validation, workspace
// layout and launches.  No entry point allocates device memory.
#include <stdlib.h>
#include <string.h>

#include "moe_internal.cuh"

using namespace moe;

namespace {

bool shape_ok(int E, int H, int I) {
    return E >= 1 && E <= 65536 && H >= 128 && H <= 32768 && H % 128 == 0 && I >= 32 && I <= 32768 && I % 32 == 0;
}

PoolView make_view(uint8_t *base, int E, int H, int I) {
    PoolView v;
    v.base = base;
    v.E = E;
    v.H = H;
    v.I = I;
    v.Ip = (I + 127) / 128 * 128;
    v.ld_gu = H / 2;
    v.ld_d = v.Ip / 2;
    v.lds_gu = H / 32;
    v.lds_d = v.Ip / 32;
    const uint64_t gu_codes = (uint64_t)2 * I * v.ld_gu;
    const uint64_t d_codes = (uint64_t)H * v.ld_d;
    const uint64_t gu_scales = (uint64_t)2 * I * v.lds_gu;
    const uint64_t d_scales = (uint64_t)H * v.lds_d;
    v.off_d = gu_codes;
    v.off_sgu = gu_codes + d_codes;
    v.off_sd = v.off_sgu + gu_scales;
    v.nmt_gu = (2 * I + 127) / 128;
    v.nmt_d = H / 128;
    const uint64_t gu_mma = (uint64_t)(H / 128) * v.nmt_gu * 512;
    const uint64_t d_mma = (uint64_t)(v.Ip / 128) * v.nmt_d * 512;
    v.off_sgu_mma = align_up(v.off_sd + d_scales, 1024);
    v.off_sd_mma = v.off_sgu_mma + align_up(gu_mma, 1024);
    v.rec = align_up(v.off_sd_mma + d_mma, 1024);
    return v;
}

moe_status cuda_status(cudaError_t e) { return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA; }

// ---------------------------------------------------------------- tracing
constexpr int kTraceCap = 65536;
struct Trace {
    char name[64] = {0};
    bool on = false;
    int n = 0;
    cudaEvent_t *ev = nullptr;  // 2 * kTraceCap
} g_trace;

bool aligned(const void *p, size_t a) { return ((uintptr_t)p % a) == 0; }

}  // namespace

namespace moe {

void trace_pre(const char *name, cudaStream_t st) {
    if (!g_trace.on || g_trace.n >= kTraceCap || strcmp(name, g_trace.name) != 0) return;
    cudaEventRecord(g_trace.ev[2 * g_trace.n], st);
}

void trace_post(const char *name, cudaStream_t st) {
    if (!g_trace.on || g_trace.n >= kTraceCap || strcmp(name, g_trace.name) != 0) return;
    cudaEventRecord(g_trace.ev[2 * g_trace.n + 1], st);
    g_trace.n++;
}

}  // namespace moe

extern "C" {

moe_status moe_trace_begin(const char *kernel_name) {
    if (kernel_name == nullptr || strlen(kernel_name) >= sizeof(g_trace.name)) return MOE_ERR_INVALID_ARG;
    if (g_trace.ev == nullptr) {
        g_trace.ev = (cudaEvent_t *)calloc(2 * kTraceCap, sizeof(cudaEvent_t));
        if (g_trace.ev == nullptr) return MOE_ERR_INVALID_ARG;
        for (int i = 0; i < 2 * kTraceCap; i++)
            if (cudaEventCreate(&g_trace.ev[i]) != cudaSuccess) return MOE_ERR_CUDA;
    }
    strcpy(g_trace.name, kernel_name);
    g_trace.n = 0;
    g_trace.on = true;
    return MOE_OK;
}

moe_status moe_trace_end(int *launches, double *total_ms) {
    if (launches == nullptr || total_ms == nullptr) return MOE_ERR_INVALID_ARG;
    g_trace.on = false;
    *launches = g_trace.n;
    *total_ms = 0.0;
    // always: on return, all work issued while tracing has finished
    if (cudaDeviceSynchronize() != cudaSuccess) return MOE_ERR_CUDA;
    if (g_trace.n == 0) return MOE_OK;
    double tot = 0.0;
    for (int i = 0; i < g_trace.n; i++) {
        float ms = 0.f;
        if (cudaEventElapsedTime(&ms, g_trace.ev[2 * i], g_trace.ev[2 * i + 1]) != cudaSuccess) return MOE_ERR_CUDA;
        tot += ms;
    }
    *total_ms = tot;
    return MOE_OK;
}

size_t moe_pool_record_bytes(int H, int I) {
    if (!shape_ok(1, H, I)) return 0;
    return (size_t)make_view(nullptr, 1, H, I).rec;
}

size_t moe_pool_bytes(int E, int H, int I) {
    if (!shape_ok(E, H, I)) return 0;
    return (size_t)E * make_view(nullptr, E, H, I).rec;
}

moe_status moe_pool_create(moe_pool **out, void *dev_mem, size_t bytes, int E, int H, int I) {
    if (out == nullptr || dev_mem == nullptr) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (!shape_ok(E, H, I)) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(dev_mem, 1024)) return MOE_ERR_INVALID_ARG;
    if (bytes < moe_pool_bytes(E, H, I)) return MOE_ERR_INVALID_ARG;
    moe_pool *p = (moe_pool *)malloc(sizeof(moe_pool));
    if (p == nullptr) return MOE_ERR_INVALID_ARG;
    p->v = make_view((uint8_t *)dev_mem, E, H, I);
    p->bytes = bytes;
    *out = p;
    return MOE_OK;
}

void moe_pool_destroy(moe_pool *pool) { free(pool); }

moe_status moe_pool_fill_synthetic(moe_pool *pool, uint64_t seed, int e_lo, int e_hi, moe_stream_t stream) {
    if (pool == nullptr) return MOE_ERR_INVALID_ARG;
    if (e_lo < 0 || e_hi > pool->v.E || e_lo > e_hi) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_pool_kernel(pool->v, 0, seed, e_lo, e_hi, nullptr, nullptr, nullptr, nullptr,
                                          (cudaStream_t)stream));
}

moe_status moe_pool_upload_expert(moe_pool *pool, int e, const uint8_t *codes_dev, const uint8_t *scales_dev,
                                  moe_stream_t stream) {
    if (pool == nullptr || codes_dev == nullptr || scales_dev == nullptr) return MOE_ERR_INVALID_ARG;
    if (e < 0 || e >= pool->v.E || !aligned(codes_dev, 8)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_pool_kernel(pool->v, 1, 0, e, e + 1, codes_dev, scales_dev, nullptr, nullptr,
                                          (cudaStream_t)stream));
}

moe_status moe_pool_download_expert(const moe_pool *pool, int e, uint8_t *codes_dev, uint8_t *scales_dev,
                                    moe_stream_t stream) {
    if (pool == nullptr || codes_dev == nullptr || scales_dev == nullptr) return MOE_ERR_INVALID_ARG;
    if (e < 0 || e >= pool->v.E || !aligned(codes_dev, 8)) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_pool_kernel(pool->v, 2, 0, e, e + 1, nullptr, nullptr, codes_dev, scales_dev,
                                          (cudaStream_t)stream));
}

moe_status moe_workspace_size(int op, int E, int H, int I, int rows, int k, size_t *bytes) {
    if (bytes == nullptr) return MOE_ERR_INVALID_ARG;
    *bytes = 0;
    if (rows < 0 || k < 1 || k > kMaxK || k > E) return MOE_ERR_INVALID_ARG;
    switch (op) {
        case MOE_OP_ROUTE:
            if (E < 1 || E > 4096 || H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
            *bytes = route_workspace_bytes(E, rows, k);
            return MOE_OK;
        case MOE_OP_DECODE:
            if (!shape_ok(E, H, I) || rows > kMaxDecodeRows) return MOE_ERR_UNSUPPORTED_SHAPE;
            *bytes = decode_workspace_bytes(E, H, I, rows, k);
            return MOE_OK;
        case MOE_OP_GROUPED:
            if (!shape_ok(E, H, I) || I % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
            *bytes = grouped_workspace_bytes(E, H, I, rows, k);
            return MOE_OK;
        default:
            return MOE_ERR_INVALID_ARG;
    }
}

moe_status moe_clear_status(void *ws, moe_stream_t stream) {
    if (ws == nullptr) return MOE_ERR_INVALID_ARG;
    return cuda_status(cudaMemsetAsync(ws, 0, sizeof(StatusWord), (cudaStream_t)stream));
}

moe_status moe_check_status(void *ws, moe_stream_t stream) {
    if (ws == nullptr) return MOE_ERR_INVALID_ARG;
    StatusWord h;
    cudaStream_t st = (cudaStream_t)stream;
    if (cudaStreamSynchronize(st) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemcpy(&h, ws, sizeof(h), cudaMemcpyDeviceToHost) != cudaSuccess) return MOE_ERR_CUDA;
    if (cudaMemset(ws, 0, sizeof(StatusWord)) != cudaSuccess) return MOE_ERR_CUDA;
    return (moe_status)h.code;
}

const char *moe_status_string(moe_status s) {
    switch (s) {
        case MOE_OK: return "ok";
        case MOE_ERR_INVALID_ARG: return "invalid argument";
        case MOE_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
        case MOE_ERR_WORKSPACE: return "workspace too small";
        case MOE_ERR_CUDA: return "CUDA error";
        case MOE_ERR_BAD_INDEX: return "expert index out of range";
        case MOE_ERR_TIMEOUT: return "bounded device wait expired";
        case MOE_ERR_NONFINITE: return "non-finite router input";
        default: return "unknown status";
    }
}

moe_status moe_route_topk(const uint16_t *x, int M, int H, const uint16_t *Wr, int E, const float *skew, int k,
                          int32_t *idx, float *w, void *ws, size_t ws_bytes, moe_stream_t stream) {
    if (M < 0 || x == nullptr || Wr == nullptr || idx == nullptr || w == nullptr || ws == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > kMaxK || k > E) return MOE_ERR_INVALID_ARG;
    if (E > 4096 || H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || !aligned(Wr, 16) || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < route_workspace_bytes(E, M, k)) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_route(x, M, H, Wr, E, skew, k, idx, w, ws, (cudaStream_t)stream));
}

moe_status moe_route_topk_prescaled(const uint16_t *x, int M, int H, const uint16_t *Wr, int E, const float *skew,
                                    int k, int32_t *idx, float *w, uint16_t *xhat, void *ws, size_t ws_bytes,
                                    moe_stream_t stream) {
    if (M < 0 || x == nullptr || Wr == nullptr || idx == nullptr || w == nullptr || xhat == nullptr || ws == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (k < 1 || k > kMaxK || k > E) return MOE_ERR_INVALID_ARG;
    if (E > 4096 || H < 8 || H % 8 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(x, 16) || !aligned(xhat, 16) || !aligned(Wr, 16) || !aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < route_workspace_bytes(E, M, k)) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_route(x, M, H, Wr, E, skew, k, idx, w, ws, (cudaStream_t)stream, xhat));
}

moe_status moe_expert_forward_decode(const moe_pool *pool, const uint16_t *x, int M, const int32_t *idx,
                                     const float *w, int k, const uint16_t *residual, uint16_t *y, void *ws,
                                     size_t ws_bytes, moe_stream_t stream) {
    if (pool == nullptr || x == nullptr || idx == nullptr || w == nullptr || y == nullptr || ws == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (M < 0 || k < 1 || k > kMaxK || k > pool->v.E) return MOE_ERR_INVALID_ARG;
    if (M > kMaxDecodeRows) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(ws, 256)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < decode_workspace_bytes(pool->v.E, pool->v.H, pool->v.I, M, k)) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_decode(pool->v, x, M, idx, w, k, residual, y, ws, (cudaStream_t)stream));
}

moe_status moe_prescale(const uint16_t *x, int M, int H, uint16_t *out, moe_stream_t stream) {
    if (x == nullptr || out == nullptr || M < 0 || H < 1) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_prescale(x, M, H, out, (cudaStream_t)stream));
}

moe_status moe_expert_forward_grouped(const moe_pool *pool, const uint16_t *x, int T, const int32_t *idx, int k,
                                      int act_mode, int32_t *perm, int32_t *inv_perm, int32_t *offsets,
                                      void *partial, int partial_dtype, void *ws, size_t ws_bytes,
                                      moe_stream_t stream) {
    if (pool == nullptr || x == nullptr || idx == nullptr || perm == nullptr || inv_perm == nullptr ||
        offsets == nullptr || partial == nullptr || ws == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (T < 0 || k < 1 || k > kMaxK || k > pool->v.E) return MOE_ERR_INVALID_ARG;
    if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_MXFP4) return MOE_ERR_INVALID_ARG;
    if (partial_dtype != MOE_PARTIAL_F32 && partial_dtype != MOE_PARTIAL_BF16) return MOE_ERR_INVALID_ARG;
    if (pool->v.I % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(ws, 256) || !aligned(x, 16) || !aligned(partial, 16)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < grouped_workspace_bytes(pool->v.E, pool->v.H, pool->v.I, T, k)) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_grouped(pool->v, x, T, idx, k, act_mode, perm, inv_perm, offsets, partial,
                                      partial_dtype, ws, (cudaStream_t)stream));
}

moe_status moe_combine(const void *partial, int partial_dtype, const int32_t *inv_perm, const float *w, int T, int k,
                       int H, const uint16_t *residual, uint16_t *y, moe_stream_t stream) {
    if (partial == nullptr || inv_perm == nullptr || w == nullptr || y == nullptr) return MOE_ERR_INVALID_ARG;
    if (T < 0 || k < 1 || k > kMaxK || H < 1) return MOE_ERR_INVALID_ARG;
    if (partial_dtype != MOE_PARTIAL_F32 && partial_dtype != MOE_PARTIAL_BF16) return MOE_ERR_INVALID_ARG;
    return cuda_status(launch_combine(partial, partial_dtype, inv_perm, w, T, k, H, residual, y, (cudaStream_t)stream));
}

moe_status moe_grouped_read_h(const moe_pool *pool, int T, int k, int act_mode, const int32_t *offsets,
                              const void *ws, size_t ws_bytes, uint8_t *hq, uint8_t *hs, moe_stream_t stream) {
    if (pool == nullptr || offsets == nullptr || ws == nullptr || hq == nullptr || hs == nullptr)
        return MOE_ERR_INVALID_ARG;
    if (T < 0 || k < 1 || k > kMaxK || k > pool->v.E) return MOE_ERR_INVALID_ARG;
    if (act_mode != MOE_ACT_MXFP8 && act_mode != MOE_ACT_MXFP4) return MOE_ERR_INVALID_ARG;
    if (pool->v.I % 64 != 0) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (!aligned(ws, 256) || !aligned(hq, 16)) return MOE_ERR_INVALID_ARG;
    if (ws_bytes < grouped_workspace_bytes(pool->v.E, pool->v.H, pool->v.I, T, k)) return MOE_ERR_WORKSPACE;
    return cuda_status(launch_read_h(pool->v, T, k, act_mode, offsets, ws, hq, hs, (cudaStream_t)stream));
}

moe_status moe_debug_set_wait_limit(uint64_t ns) {
    const uint64_t lim = ns == 0 ? 1000ull * 1000ull * 1000ull : ns;
    if (set_wait_limit_decode_fused(lim) != cudaSuccess) return MOE_ERR_CUDA;
    if (set_wait_limit_gemm(lim) != cudaSuccess) return MOE_ERR_CUDA;
    return MOE_OK;
}

moe_status moe_grouped_set_cta_pairs(int mode) {
    if (mode < 0 || mode > 2) return MOE_ERR_INVALID_ARG;
    set_cta_pairs(mode);
    return MOE_OK;
}

moe_status moe_debug_set_barrier_extra(int extra) {
    if (extra < 0 || extra > 1024) return MOE_ERR_INVALID_ARG;
    set_barrier_extra((unsigned int)extra);
    return MOE_OK;
}

}  // extern "C"
