// Internal declarations of the expert-major prefill path.
#pragma once

#include <cuda_fp16.h>

#include "moe_internal.cuh"

namespace moe {

constexpr int kMaxSortE = 4096;  // experts supported by the grouped path

// Activation rows of the grouped GEMMs.  nparts = 1: one MXFP8 row per pair (OCP
// rule, the prefill path).  nparts = 3: the value is the sum of three E4M3 parts
// with their own E8M0 scales (see split_exp), which represents a bf16 row exactly
// for elements within about 20 binades of their 32-block's max (the multi-token
// decode path); row 3r+q holds part q of sorted pair r.
struct GroupedWs {
    int *local_rank;  // [P]
    int *cnt;         // [nblocks][E]
    int *prior;       // [nblocks][E]
    int32_t *uexp;    // [E] the experts with at least one pair, ascending
    int32_t *n_union; // [1] their number
    uint8_t *xq;      // [nparts*P][H]    E4M3 rows of x in sorted order
    uint8_t *xs;      // [nparts*P][H/32] their E8M0 scales
    uint8_t *hq;      // [nparts*P][I]    E4M3 rows of h in sorted order
    uint8_t *hs;      // [nparts*P][Ip/32], Ip = I rounded up to 128 (tail bytes unused)
    size_t end;       // total bytes
};

__host__ __device__ inline GroupedWs grouped_ws_layout(void *ws, int E, int H, int I, int T, int k, int nparts = 1) {
    GroupedWs g;
    const size_t P = (size_t)T * k;
    const size_t R = P * (size_t)nparts;
    const size_t nblocks = (P + 1023) / 1024;
    char *base = (char *)ws;
    size_t o = 256;
    g.local_rank = (int *)(base + o);  o += align_up(P * 4, 1024);
    g.cnt = (int *)(base + o);         o += align_up(nblocks * E * 4, 1024);
    g.prior = (int *)(base + o);       o += align_up(nblocks * E * 4, 1024);
    g.uexp = (int32_t *)(base + o);    o += align_up((size_t)E * 4, 256);
    g.n_union = (int32_t *)(base + o); o += 256;
    g.xq = (uint8_t *)(base + o);      o += align_up(R * H, 1024);
    g.xs = (uint8_t *)(base + o);      o += align_up(R * (H / 32), 1024);
    g.hq = (uint8_t *)(base + o);      o += align_up(R * I, 1024);
    g.hs = (uint8_t *)(base + o);      o += align_up(R * (((size_t)I + 127) / 128 * 4), 1024);
    g.end = o;
    return g;
}

// The multi-token decode through the grouped GEMMs: the grouped workspace with three
// activation parts, then the sort's outputs and the fp32 expert output rows.
struct DecodeMultiWs {
    GroupedWs g;
    int32_t *perm;      // [P]
    int32_t *inv_perm;  // [P]
    int32_t *offsets;   // [E+1]
    float *partial;     // [P][H]
    size_t end;
};

__host__ __device__ inline DecodeMultiWs decode_multi_ws_layout(void *ws, int E, int H, int I, int M, int k) {
    DecodeMultiWs d;
    d.g = grouped_ws_layout(ws, E, H, I, M, k, 3);
    const size_t P = (size_t)M * k;
    char *base = (char *)ws;
    size_t o = d.g.end;
    d.perm = (int32_t *)(base + o);     o += align_up(P * 4, 256);
    d.inv_perm = (int32_t *)(base + o); o += align_up(P * 4, 256);
    d.offsets = (int32_t *)(base + o);  o += align_up(((size_t)E + 1) * 4, 256);
    d.partial = (float *)(base + o);    o += align_up(P * H * 4, 1024);
    d.end = o;
    return d;
}

// E8M0 exponent of one E4M3 part of a 32-element block with max |v| = amax: the
// block's largest value scales into [128, 256), below E4M3's 448, so nothing
// saturates and the part is v rounded (RNE) to E4M3 precision.
__device__ __forceinline__ int split_exp(float amax) {
    if (!(amax > 0.f) || !isfinite(amax)) return -127;
    int ex;
    frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
    return max(-127, min(127, ex - 1 - 7));
}

__device__ __forceinline__ uint8_t e4m3_rn(float v) {
    unsigned short pair;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.f), "f"(v));
    return (uint8_t)(pair & 0xFF);
}

__device__ __forceinline__ float e4m3_value(uint8_t q) {
    unsigned int h2;
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(h2) : "h"((unsigned short)q));
    return __half2float(__ushort_as_half((unsigned short)(h2 & 0xFFFFu)));
}

// One part of the split: the E4M3 code of r at exponent X, and r less what the
// code represents (exact in fp32: the code keeps the leading bits of r).
__device__ __forceinline__ uint8_t split_part(float &r, int X) {
    const uint8_t q = e4m3_rn(ldexpf(r, -X));
    r -= ldexpf(e4m3_value(q), X);
    return q;
}

// The two grouped block-scaled GEMMs (gate/up with SwiGLU and MXFP8 epilogue,
// then down), over the sorted rows.
cudaError_t launch_grouped_gemms(const PoolView &v, int T, int k, const int32_t *offsets, const GroupedWs &g,
                                 void *partial, int partial_dtype, StatusWord *st, cudaStream_t stream,
                                 int nparts = 1);

// Multi-token decode (M > 1) through the grouped GEMMs with three-part activations;
// cudaErrorNotSupported for shapes the GEMMs do not take.
cudaError_t launch_decode_multi(const PoolView &v, const uint16_t *x, int M, const int32_t *idx, const float *w, int k,
                                const uint16_t *residual, uint16_t *y, void *ws, cudaStream_t st);
size_t decode_multi_workspace_bytes(int E, int H, int I, int M, int k);

}  // namespace moe
