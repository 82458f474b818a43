// Internal declarations of the expert-major prefill path.
#pragma once

#include "moe_internal.cuh"

namespace moe {

constexpr int kMaxSortE = 4096;  // experts supported by the grouped path

// Workspace of the grouped path (after the 256-byte status word).
struct GroupedWs {
    int *local_rank;  // [P]
    int *cnt;         // [nblocks][E]
    int *prior;       // [nblocks][E]
    uint8_t *xq;      // [P][H]    E4M3 rows of x in sorted order
    uint8_t *xs;      // [P][H/32] their E8M0 scales
    uint8_t *hq;      // [P][I]    E4M3 rows of h in sorted order
    uint8_t *hs;      // [P][Ip/32], Ip = I rounded up to 128 (tail bytes unused)
    size_t end;       // total bytes
};

__host__ __device__ inline GroupedWs grouped_ws_layout(void *ws, int E, int H, int I, int T, int k) {
    GroupedWs g;
    const size_t P = (size_t)T * k;
    const size_t nblocks = (P + 1023) / 1024;
    char *base = (char *)ws;
    size_t o = 256;
    g.local_rank = (int *)(base + o);  o += align_up(P * 4, 1024);
    g.cnt = (int *)(base + o);         o += align_up(nblocks * E * 4, 1024);
    g.prior = (int *)(base + o);       o += align_up(nblocks * E * 4, 1024);
    g.xq = (uint8_t *)(base + o);      o += align_up(P * H, 1024);
    g.xs = (uint8_t *)(base + o);      o += align_up(P * (H / 32), 1024);
    g.hq = (uint8_t *)(base + o);      o += align_up(P * I, 1024);
    g.hs = (uint8_t *)(base + o);      o += align_up(P * (((size_t)I + 127) / 128 * 4), 1024);
    g.end = o;
    return g;
}

// The two grouped block-scaled GEMMs (gate/up with SwiGLU and MXFP8 epilogue,
// then down), over the sorted rows.
cudaError_t launch_grouped_gemms(const PoolView &v, int T, int k, const int32_t *offsets, const GroupedWs &g,
                                 void *partial, int partial_dtype, StatusWord *st, cudaStream_t stream);

}  // namespace moe
