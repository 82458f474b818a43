// Decode / verify path: 1..32 rows, memory-bound.
//
// One row runs the fused cooperative kernel (decode_fused.cu).  Several rows (the
// verify batch of the four-SSD page, "可选的 Qwen 扩展": one forward pass checks
// several rows) run on the tensor cores through the grouped GEMMs with five-part
// MXFP4 activations (launch_decode_multi in prefill.cu) when I is a multiple of 64;
// otherwise the kernels below read each distinct selected expert from the pool once
// and dequantise its packed 4-bit weights in registers:
//   decode_prep_kernel    union of selected experts, per-expert row lists,
//                         bf16 rows -> f16 with a per-row power-of-two scale
//   decode_gateup_kernel  g = W_g x, u = W_u x, h = silu(g) * u       (fp32 out)
//   decode_down_kernel    y = sum_j w_j (W_d h_j) (+ residual)         (bf16 out)
// Inner products run as packed f16 FMAs over one 32-element scale block (E2M1
// times a scaled f16 input is exact in f16; the 16-term block sum is rounded in
// f16), then the block sum is scaled by its E8M0 factor and accumulated in fp32.
#include "moe_internal.cuh"
#include "prefill_internal.cuh"

namespace moe {
namespace {

constexpr int kThreads = 256;          // 8 warps
constexpr int kDownPairGroup = 32;     // pairs whose h is staged in shared memory at once

struct DecodeWs {
    int *n_union;      // [1]
    int *union_e;      // [P]
    int *union_off;    // [P + 1]
    int *pair_list;    // [P] pair indices sorted by (expert, pair)
    __half *x16;       // [M][H]
    int *x_exp;        // [M]
    float *h;          // [P][I]
    unsigned int *h_amax;  // [P]
};

__host__ __device__ inline DecodeWs decode_ws(void *ws, int H, int I, int M, int k) {
    DecodeWs d;
    const int P = M * k;
    char *p = (char *)ws + 256;
    d.n_union = (int *)p;                 p += 256;
    d.union_e = (int *)p;                 p += align_up((size_t)P * 4, 256);
    d.union_off = (int *)p;               p += align_up((size_t)(P + 1) * 4, 256);
    d.pair_list = (int *)p;               p += align_up((size_t)P * 4, 256);
    d.x16 = (__half *)p;                  p += align_up((size_t)M * H * 2, 256);
    d.x_exp = (int *)p;                   p += align_up((size_t)M * 4, 256);
    d.h = (float *)p;                     p += align_up((size_t)P * I * 4, 256);
    d.h_amax = (unsigned int *)p;         p += align_up((size_t)P * 4, 256);
    return d;
}

__host__ __device__ inline size_t decode_ws_end(int H, int I, int M, int k) {
    DecodeWs d = decode_ws((void *)0, H, I, M, k);
    return (size_t)((char *)d.h_amax - (char *)0) + align_up((size_t)M * k * 4, 256);
}

__device__ __forceinline__ float block_max(float v, float *red) {
    for (int off = 16; off > 0; off >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, off));
    if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = v;
    __syncthreads();
    float r = 0.f;
    for (int w = 0; w < (int)(blockDim.x >> 5); w++) r = fmaxf(r, red[w]);
    __syncthreads();
    return r;
}

// Blocks 0..M-1: row m of x -> f16 scaled by 2^-s, max|x 2^-s| in [128, 256).
// Block M: validate idx, group the pairs by expert, clear h_amax.
__global__ void __launch_bounds__(kThreads) decode_prep_kernel(const uint16_t *__restrict__ x, int M, int H,
                                                               const int32_t *__restrict__ idx, int k, int E,
                                                               DecodeWs d, StatusWord *st) {
    __shared__ float red[32];
    __shared__ int ekey[kMaxDecodeRows * kMaxK];
    __shared__ int sorted_e[kMaxDecodeRows * kMaxK];
    const int tid = threadIdx.x;
    if ((int)blockIdx.x < M) {
        const int m = blockIdx.x;
        const uint16_t *xr = x + (size_t)m * H;
        float a = 0.f;
        for (int h = tid; h < H; h += blockDim.x) a = fmaxf(a, fabsf(bf16_bits_to_float(xr[h])));
        const float amax = block_max(a, red);
        int s = 0;
        if (amax > 0.f) {
            int ex;
            frexpf(amax, &ex);  // amax in [2^(ex-1), 2^ex)
            s = ex - 1 - 7;
        }
        for (int h = tid; h < H; h += blockDim.x)
            d.x16[(size_t)m * H + h] = __float2half_rn(ldexpf(bf16_bits_to_float(xr[h]), -s));
        if (tid == 0) d.x_exp[m] = s;
        return;
    }
    const int P = M * k;
    for (int p = tid; p < P; p += blockDim.x) {
        const int e = idx[p];
        const bool ok = e >= 0 && e < E;
        if (!ok) set_status(st, MOE_ERR_BAD_INDEX, (unsigned)p);
        ekey[p] = ok ? e : 0x7fffffff;
        d.h_amax[p] = 0u;
    }
    __syncthreads();
    // rank of each pair in (expert, pair) order
    for (int a = tid; a < P; a += blockDim.x) {
        const int ea = ekey[a];
        int r = 0;
        for (int b = 0; b < P; b++) {
            const int eb = ekey[b];
            r += (eb < ea) || (eb == ea && b < a);
        }
        d.pair_list[r] = a;
        sorted_e[r] = ea;
    }
    __syncthreads();
    if (tid == 0) {
        int nu = 0;
        for (int r = 0; r < P; r++) {
            const int e = sorted_e[r];
            if (e == 0x7fffffff) break;
            if (r == 0 || e != sorted_e[r - 1]) {
                d.union_e[nu] = e;
                d.union_off[nu] = r;
                nu++;
            }
        }
        int nvalid = 0;
        while (nvalid < P && sorted_e[nvalid] != 0x7fffffff) nvalid++;
        d.union_off[nu] = nvalid;
        *d.n_union = nu;
    }
}

// 32 elements of one row block times the matching f16 input block, summed in f16
// pairs, returned as fp32 (before the E8M0 scale).
__device__ __forceinline__ float block_dot(const uint4 &q, const uint4 *xb) {
    const unsigned int words[4] = {q.x, q.y, q.z, q.w};
    unsigned int acc0 = 0u, acc1 = 0u;
#pragma unroll
    for (int wd = 0; wd < 4; wd++) {
        unsigned int w0, w1, w2, w3;
        e2m1x8_to_f16x2x4(words[wd], w0, w1, w2, w3);
        const uint4 xv = xb[wd];
        acc0 = hfma2_u32(w0, xv.x, acc0);
        acc1 = hfma2_u32(w1, xv.y, acc1);
        acc0 = hfma2_u32(w2, xv.z, acc0);
        acc1 = hfma2_u32(w3, xv.w, acc1);
    }
    return f16x2_sum_to_float(acc0) + f16x2_sum_to_float(acc1);
}

// One warp task = (expert of the union, two intermediate indices i0, i0+1):
// gate rows i0, i0+1 and up rows i0, i0+1 of W_gu, applied to every row routed to
// the expert.
__global__ void __launch_bounds__(kThreads) decode_gateup_kernel(PoolView v, int M, int k, DecodeWs d) {
    const int lane = threadIdx.x & 31;
    const int gwarp = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int nwarps = (gridDim.x * blockDim.x) >> 5;
    const int nu = *d.n_union;
    const int tasks_per_expert = v.I / 2;
    const int ntasks = nu * tasks_per_expert;
    const int nkb = v.H / 32;
    for (int task = gwarp; task < ntasks; task += nwarps) {
        const int ui = task / tasks_per_expert;
        const int i0 = 2 * (task % tasks_per_expert);
        const int e = d.union_e[ui];
        const uint8_t *rec = v.base + (uint64_t)e * v.rec;
        const int rg = 32 * (i0 / kGroupRows) + (i0 % kGroupRows);  // gate row of i0 in W_gu
        const int rows[4] = {rg, rg + 1, rg + kGroupRows, rg + kGroupRows + 1};
        const uint8_t *crow[4];
        const uint8_t *srow[4];
#pragma unroll
        for (int r = 0; r < 4; r++) {
            crow[r] = rec + (uint64_t)rows[r] * v.ld_gu;
            srow[r] = rec + v.off_sgu + (uint64_t)rows[r] * v.lds_gu;
        }
        for (int pi = d.union_off[ui]; pi < d.union_off[ui + 1]; pi++) {
            const int p = d.pair_list[pi];
            const int m = p / k;
            const __half *xrow = d.x16 + (size_t)m * v.H;
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            for (int kb = lane; kb < nkb; kb += 32) {
                uint4 q[4];
                unsigned int sb[4];
#pragma unroll
                for (int r = 0; r < 4; r++) {
                    q[r] = ldg_stream16(crow[r] + kb * 16);
                    sb[r] = ldg_stream_u8(srow[r] + kb);
                }
                uint4 xb[4];
                const uint4 *xp = reinterpret_cast<const uint4 *>(xrow + kb * 32);
#pragma unroll
                for (int wd = 0; wd < 4; wd++) xb[wd] = __ldg(xp + wd);
#pragma unroll
                for (int r = 0; r < 4; r++) acc[r] = fmaf(block_dot(q[r], xb), e8m0_to_float(sb[r]), acc[r]);
            }
#pragma unroll
            for (int r = 0; r < 4; r++)
                for (int off = 16; off > 0; off >>= 1) acc[r] += __shfl_xor_sync(0xffffffffu, acc[r], off);
            if (lane == 0) {
                const int s = d.x_exp[m];
                const float g0 = ldexpf(acc[0], s), g1 = ldexpf(acc[1], s);
                const float u0 = ldexpf(acc[2], s), u1 = ldexpf(acc[3], s);
                const float h0 = g0 / (1.f + expf(-g0)) * u0;
                const float h1 = g1 / (1.f + expf(-g1)) * u1;
                d.h[(size_t)p * v.I + i0] = h0;
                d.h[(size_t)p * v.I + i0 + 1] = h1;
                atomicMax(&d.h_amax[p], __float_as_uint(fmaxf(fabsf(h0), fabsf(h1))));
            }
        }
    }
}

// CTA = `rows` consecutive output rows over all pairs; pairs are staged up to 32
// at a time in shared memory as f16 scaled by a per-pair power of two.
__global__ void __launch_bounds__(kThreads) decode_down_kernel(PoolView v, int M, int k, int rows, int group,
                                                               const float *__restrict__ w,
                                                               const uint16_t *__restrict__ residual,
                                                               uint16_t *__restrict__ y, DecodeWs d,
                                                               const int32_t *__restrict__ idx) {
    extern __shared__ __align__(16) unsigned char smem[];
    __half *hs = reinterpret_cast<__half *>(smem);                                 // [group][Ip]
    float *yacc = reinterpret_cast<float *>(smem + (size_t)group * v.Ip * 2);    // [M][rows]
    __shared__ float pscale[kDownPairGroup];
    __shared__ int pexp[kDownPairGroup];
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const int row0 = blockIdx.x * rows;
    const int P = M * k;
    const int nkb = v.I / 32;
    for (int i = tid; i < M * rows; i += blockDim.x) yacc[i] = 0.f;
    for (int g0 = 0; g0 < P; g0 += group) {
        const int ng = min(group, P - g0);
        __syncthreads();
        if (tid < ng) {
            const int p = g0 + tid;
            const float amax = __uint_as_float(d.h_amax[p]);
            int s = 0;
            if (amax > 0.f && isfinite(amax)) {
                int ex;
                frexpf(amax, &ex);
                s = ex - 1 - 7;
            }
            pexp[tid] = s;
            const int e = idx[p];
            const bool ok = e >= 0 && e < v.E;
            pscale[tid] = ok ? ldexpf(w[p], s) : 0.f;
        }
        __syncthreads();
        for (int i = tid; i < ng * v.Ip; i += blockDim.x) {
            const int pp = i / v.Ip, c = i % v.Ip;
            const float hv = (c < v.I) ? d.h[(size_t)(g0 + pp) * v.I + c] : 0.f;
            hs[i] = __float2half_rn(ldexpf(hv, -pexp[pp]));
        }
        __syncthreads();
        for (int lr = warp; lr < rows; lr += kThreads / 32) {
            const int o = row0 + lr;
            if (o >= v.H) continue;
            for (int pp = 0; pp < ng; pp++) {
                const int p = g0 + pp;
                const int e = idx[p];
                if (e < 0 || e >= v.E) continue;
                const uint8_t *rec = v.base + (uint64_t)e * v.rec;
                const uint8_t *crow = rec + v.off_d + (uint64_t)o * v.ld_d;
                const uint8_t *srow = rec + v.off_sd + (uint64_t)o * v.lds_d;
                float acc = 0.f;
                for (int kb = lane; kb < nkb; kb += 32) {
                    const uint4 q = ldg_stream16(crow + kb * 16);
                    const unsigned int sb = ldg_stream_u8(srow + kb);
                    const uint4 *xb = reinterpret_cast<const uint4 *>(hs + (size_t)pp * v.Ip + kb * 32);
                    acc = fmaf(block_dot(q, xb), e8m0_to_float(sb), acc);
                }
                for (int off = 16; off > 0; off >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, off);
                if (lane == 0) yacc[(p / k) * rows + lr] += pscale[pp] * acc;
            }
        }
    }
    __syncthreads();
    for (int i = tid; i < M * rows; i += blockDim.x) {
        const int m = i / rows, lr = i % rows;
        const int o = row0 + lr;
        if (o >= v.H) continue;
        float val = yacc[i];
        if (residual != nullptr) val += bf16_bits_to_float(residual[(size_t)m * v.H + o]);
        const __nv_bfloat16 b = __float2bfloat16_rn(val);
        y[(size_t)m * v.H + o] = *reinterpret_cast<const uint16_t *>(&b);
    }
}

__global__ void prescale_kernel(const uint16_t *__restrict__ x, int H, uint16_t *__restrict__ out) {
    __shared__ float red[32];
    const uint16_t *xr = x + (size_t)blockIdx.x * H;
    float a = 0.f;
    for (int h = threadIdx.x; h < H; h += blockDim.x) a = fmaxf(a, fabsf(bf16_bits_to_float(xr[h])));
    const float amax = block_max(a, red);
    int p = 0;
    if (amax > 0.f) {
        int ex;
        frexpf(amax, &ex);
        p = ex - 1 - 2;
    }
    for (int h = threadIdx.x; h < H; h += blockDim.x) {
        const __nv_bfloat16 b = __float2bfloat16_rn(ldexpf(bf16_bits_to_float(xr[h]), -p));
        out[(size_t)blockIdx.x * H + h] = *reinterpret_cast<const uint16_t *>(&b);
    }
}

PerDevice g_num_sms(0);

}  // namespace

size_t decode_workspace_bytes(int E, int H, int I, int M, int k) {
    const size_t general = decode_ws_end(H, I, M, k);
    // M = 1: the fused kernel; M > 1: the grouped GEMMs when the shape allows
    const size_t special = M == 1 ? decode_fused_workspace_bytes(I, k) : decode_multi_workspace_bytes(E, H, I, M, k);
    return special > general ? special : general;
}

cudaError_t launch_decode(const PoolView &v, const uint16_t *x, int M, const int32_t *idx, const float *w, int k,
                          const uint16_t *residual, uint16_t *y, void *ws, cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    int num_sms = 0;
    {
        const cudaError_t e = device_attr(cudaDevAttrMultiProcessorCount, g_num_sms, &num_sms);
        if (e != cudaSuccess) return e;
    }
    if (M == 1) {
        const cudaError_t e = launch_decode_fused(v, x, idx, w, k, residual, y, ws, st);
        if (e != cudaErrorNotSupported) return e;
    } else {
        const cudaError_t e = launch_decode_multi(v, x, M, idx, w, k, residual, y, ws, st);
        if (e != cudaErrorNotSupported) return e;
    }
    DecodeWs d = decode_ws(ws, v.H, v.I, M, k);
    StatusWord *stw = reinterpret_cast<StatusWord *>(ws);
    {
        TraceScope trace_scope("decode_prep", st);
        decode_prep_kernel<<<M + 1, kThreads, 0, st>>>(x, M, v.H, idx, k, v.E, d, stw);
    }
    const int P = M * k;
    const int umax = P < v.E ? P : v.E;
    const long long tasks = (long long)umax * (v.I / 2);
    long long blocks = (tasks + 7) / 8;
    const long long cap = (long long)num_sms * 4;
    if (blocks > cap) blocks = cap;
    {
        TraceScope trace_scope("decode_gateup", st);
        decode_gateup_kernel<<<(unsigned)blocks, kThreads, 0, st>>>(v, M, k, d);
    }
    // two CTAs per SM, each a block of consecutive output rows (a multiple of 8)
    int rows = (v.H + 2 * num_sms - 1) / (2 * num_sms);
    rows = (rows + 7) / 8 * 8;
    // pairs staged per pass: at most 32, and at most ~200 KB of f16 rows
    int group = P < kDownPairGroup ? P : kDownPairGroup;
    const int fit = (int)((200 * 1024 - (size_t)M * rows * 4) / ((size_t)v.Ip * 2));
    if (group > fit) group = fit;
    if (group < 1) return cudaErrorInvalidValue;
    const size_t smem = (size_t)group * v.Ip * 2 + (size_t)M * rows * 4;
    static PerDevice smem_down(0);
    cudaError_t e = ensure_dynamic_smem(decode_down_kernel, smem, smem_down);
    if (e != cudaSuccess) return e;
    {
        TraceScope trace_scope("decode_down", st);
        decode_down_kernel<<<(v.H + rows - 1) / rows, kThreads, smem, st>>>(v, M, k, rows, group, w, residual, y, d,
                                                                             idx);
    }
    return cudaGetLastError();
}

cudaError_t launch_prescale(const uint16_t *x, int M, int H, uint16_t *out, cudaStream_t st) {
    if (M == 0) return cudaSuccess;
    {
        TraceScope trace_scope("prescale", st);
        prescale_kernel<<<M, 256, 0, st>>>(x, H, out);
    }
    return cudaGetLastError();
}

}  // namespace moe
