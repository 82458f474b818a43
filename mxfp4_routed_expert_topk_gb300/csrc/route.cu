// Router: logits, exact top-k and softmax over the selected logits.
//
// The pages ("工作原理" on the Apple Silicon page) say the router picks 16 of each
// layer's routed experts per token.  Selection here is EXACT: expert e ranks by
// the real number
//   l_e = sum_h x_h W_r[e,h] (+ skew_e),  ties broken to the lower index,
// and the k winners are returned in descending order.
//
// route_logits_kernel computes l~_e in fp32 with a rigorous bound
// |l~_e - l_e| <= b_e.  A product of two bf16 is exact in fp32, so the only
// errors are the roundings of the additions.  A rounded sum r = fl(a + b) is off
// by at most u |r| (u = 2^-24, round to nearest) when r is normal, and by at most
// 2^-150 when it is subnormal.  The kernel therefore carries, next to every partial
// sum, u times the sum of the magnitudes of all the rounded additions below it (a
// running error bound, accumulated with rounding upwards):
//   |l~ - l| <= u * sum over the additions of |r_i|  +  2^-149 per product,
// the last term for underflowing products and subnormal sums.  For sums of terms
// of mixed sign this is far tighter than the a-priori bound gamma_d * sum |x W|,
// so far fewer tokens need the exact evaluation.
//
// For many tokens (route_tiled_kernel) the logits are a register-tiled fp32 FMA
// product with a bounded summation tree of depth d, and the a-priori bound
//   |l~ - l| <= gamma_d * (sum_h |x_h W_r[e,h]| + |skew_e|),  gamma_d = d u / (1 - d u),
// is used with the sum of |x_h W_r[e,h]| replaced by its Cauchy-Schwarz upper bound
// ||x|| ||W_r[e]||, so each product costs one FMA.
//
// route_select_kernel (one CTA per token) sorts by (l~ desc, index asc) and
// certifies the order with the intervals [l~ - b, l~ + b]: an outsider can only
// enter the top k if its interval reaches the lowest lower bound of the winners,
// and two experts can only swap if their intervals meet.  Clusters of meeting
// intervals that touch the top k are re-evaluated with exact integer arithmetic
// (every term is an integer multiple of 2^-268) and ordered by exact value.
#include "moe_internal.cuh"
#include "sm100_async.cuh"

namespace moe {
namespace {

constexpr int kLogitTokens = 8;    // tokens per CTA in the logit kernel
constexpr int kLogitExperts = 4;   // experts per CTA (two warps each, one per half of H)
constexpr int kMaxE = 4096;
constexpr int kMaxCand = 256;      // experts that may still enter the top k
constexpr int kMaxExact = 64;      // experts evaluated exactly per token
constexpr int kLimbs = 20;         // base-2^32 digits of an exact logit, unit 2^-268
constexpr int kBins = 512;         // exponent bins of the exact evaluation
constexpr int kTiledMinTokens = 64;  // tokens from which the logits take the tiled kernel

struct RouteWs {
    float *logit;  // [M][E]
    float *bound;  // [M][E]
    float *xnorm;  // [M] ||x_m|| (tiled path)
    float *wnorm;  // [E] ||W_r[e]|| (tiled path)
    size_t end;
};

__host__ __device__ inline RouteWs route_ws(void *ws, int M, int E) {
    RouteWs r;
    char *p = (char *)ws;
    size_t o = 256;
    r.logit = (float *)(p + o); o += align_up((size_t)M * E * sizeof(float), 256);
    r.bound = (float *)(p + o); o += align_up((size_t)M * E * sizeof(float), 256);
    r.xnorm = (float *)(p + o); o += align_up((size_t)M * sizeof(float), 256);
    r.wnorm = (float *)(p + o); o += align_up((size_t)E * sizeof(float), 256);
    r.end = o;
    return r;
}

__device__ __forceinline__ void unpack_bf16x8(const uint4 &v, float f[8]) {
    const unsigned int u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
    for (int i = 0; i < 4; i++) {
        f[2 * i] = __uint_as_float(u[i] << 16);
        f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
    }
}

// Block (bx, by): experts 4*bx .. 4*bx+3 for tokens 8*by .. 8*by+7.  Warp w handles
// expert 4*bx + w/2 over one half of H; lanes take 8 consecutive elements per step.
// Used with 256 threads; x rows staged in dynamic shared memory.  NB chunks of
// W_r are loaded per batch (one batch covers H/2 = 4096 with NB = 16).
// With `prescale` (one token): the staged row is replaced by x_hat = x * 2^-p, p =
// floor(log2 max|x|) - 2, rounded to bf16 element by element exactly as
// prescale_kernel does, and the logits are those of x_hat; CTA 0 writes x_hat to
// xhat_out (when not null).
template <int NB>
__device__ void logits_block(const uint16_t *__restrict__ x, int M, int H, const uint16_t *__restrict__ Wr, int E,
                             const float *__restrict__ skew, float *__restrict__ logit,
                             float *__restrict__ bound, bool prescale = false, uint16_t *xhat_out = nullptr) {
    extern __shared__ __align__(16) uint16_t xs[];  // [nt][H]
    __shared__ float red_l[8][kLogitTokens], red_s[8][kLogitTokens];
    const int m0 = blockIdx.y * kLogitTokens;
    const int nt = min(kLogitTokens, M - m0);
    const int nvec = nt * H / 8;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int e = blockIdx.x * kLogitExperts + (warp >> 1);
    const int hmid = ((H / 2) + 7) / 8 * 8;
    const int h0 = (warp & 1) ? hmid : 0, h1 = (warp & 1) ? H : hmid;
    const uint16_t *wrow = Wr + (size_t)(e < E ? e : 0) * H;
    // this warp's first batch of W_r chunks is requested before x is staged, so the
    // two latencies overlap
    uint4 wv[NB];
#pragma unroll
    for (int c = 0; c < NB; c++) {
        const int h = h0 + lane * 8 + 256 * c;
        wv[c] = (e < E && h < h1) ? __ldg(reinterpret_cast<const uint4 *>(wrow + h)) : make_uint4(0u, 0u, 0u, 0u);
    }
    const uint4 *xg = reinterpret_cast<const uint4 *>(x + (size_t)m0 * H);
    for (int i = threadIdx.x; i < nvec; i += blockDim.x) reinterpret_cast<uint4 *>(xs)[i] = xg[i];
    __syncthreads();
    if (prescale) {
        __shared__ float pmax[32];
        float am = 0.f;
        for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
            float f[8];
            unpack_bf16x8(reinterpret_cast<const uint4 *>(xs)[i], f);
#pragma unroll
            for (int j = 0; j < 8; j++) am = fmaxf(am, fabsf(f[j]));
        }
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) am = fmaxf(am, __shfl_xor_sync(0xffffffffu, am, off));
        if ((threadIdx.x & 31) == 0) pmax[threadIdx.x >> 5] = am;
        __syncthreads();
        float amax = 0.f;
        for (int w = 0; w < (int)(blockDim.x >> 5); w++) amax = fmaxf(amax, pmax[w]);
        int p = 0;
        if (amax > 0.f) {
            int ex;
            frexpf(amax, &ex);
            p = ex - 1 - 2;
        }
        for (int i = threadIdx.x; i < nvec; i += blockDim.x) {
            float f[8];
            unpack_bf16x8(reinterpret_cast<const uint4 *>(xs)[i], f);
            uint32_t u[4];
#pragma unroll
            for (int j = 0; j < 4; j++) {
                const __nv_bfloat16 lo = __float2bfloat16_rn(ldexpf(f[2 * j], -p));
                const __nv_bfloat16 hi = __float2bfloat16_rn(ldexpf(f[2 * j + 1], -p));
                u[j] = (uint32_t)(*reinterpret_cast<const uint16_t *>(&lo)) |
                       ((uint32_t)(*reinterpret_cast<const uint16_t *>(&hi)) << 16);
            }
            const uint4 v = make_uint4(u[0], u[1], u[2], u[3]);
            reinterpret_cast<uint4 *>(xs)[i] = v;
            if (xhat_out != nullptr && blockIdx.x == 0) reinterpret_cast<uint4 *>(xhat_out)[i] = v;
        }
        __syncthreads();
    }

    // acc: the partial logit; ea, eb: u times the magnitudes of the additions below
    // it (two chains, rounded upwards)
    constexpr float u = 5.9604645e-8f;  // 2^-24
    float acc[kLogitTokens], ea[kLogitTokens], eb[kLogitTokens];
#pragma unroll
    for (int t = 0; t < kLogitTokens; t++) acc[t] = ea[t] = eb[t] = 0.f;
    if (e < E) {
        // batches of NB chunks: all loads of a batch issued before any arithmetic (the
        // first before x was staged); chunks are summed in increasing h (the order the
        // bound assumes)
        for (int hb = h0 + lane * 8; hb < h1; hb += 256 * NB) {
            if (hb != h0 + lane * 8) {
#pragma unroll
                for (int c = 0; c < NB; c++) {
                    const int h = hb + 256 * c;
                    wv[c] = h < h1 ? __ldg(reinterpret_cast<const uint4 *>(wrow + h)) : make_uint4(0u, 0u, 0u, 0u);
                }
            }
#pragma unroll
            for (int c = 0; c < NB; c++) {
                const int h = hb + 256 * c;
                if (h >= h1) break;
                float wf[8];
                unpack_bf16x8(wv[c], wf);
#pragma unroll
                for (int t = 0; t < kLogitTokens; t++) {
                    if (t < nt) {
                        float xf[8], p[8];
                        unpack_bf16x8(*reinterpret_cast<const uint4 *>(xs + (size_t)t * H + h), xf);
#pragma unroll
                        for (int i = 0; i < 8; i++) p[i] = xf[i] * wf[i];  // exact
                        const float s01 = p[0] + p[1], s23 = p[2] + p[3], s45 = p[4] + p[5], s67 = p[6] + p[7];
                        const float s03 = s01 + s23, s47 = s45 + s67;
                        const float s = s03 + s47;
                        acc[t] += s;
                        ea[t] = __fmaf_ru(fabsf(s01), u, ea[t]);
                        eb[t] = __fmaf_ru(fabsf(s23), u, eb[t]);
                        ea[t] = __fmaf_ru(fabsf(s45), u, ea[t]);
                        eb[t] = __fmaf_ru(fabsf(s67), u, eb[t]);
                        ea[t] = __fmaf_ru(fabsf(s03), u, ea[t]);
                        eb[t] = __fmaf_ru(fabsf(s47), u, eb[t]);
                        ea[t] = __fmaf_ru(fabsf(s), u, ea[t]);
                        eb[t] = __fmaf_ru(fabsf(acc[t]), u, eb[t]);
                    }
                }
            }
        }
    }
#pragma unroll
    for (int t = 0; t < kLogitTokens; t++) {
        float err = __fadd_ru(ea[t], eb[t]);
        // butterfly: both partners form the same sum, and each carries the bounds of
        // both halves plus that of the new addition
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const float o = __shfl_xor_sync(0xffffffffu, acc[t], off);
            const float oe = __shfl_xor_sync(0xffffffffu, err, off);
            acc[t] += o;
            err = __fmaf_ru(fabsf(acc[t]), u, __fadd_ru(err, oe));
        }
        if (lane == 0) {
            red_l[warp][t] = acc[t];
            red_s[warp][t] = err;
        }
    }
    __syncthreads();
    if (threadIdx.x < kLogitExperts * nt) {
        const int q = threadIdx.x / nt, t = threadIdx.x % nt;
        const int eq = blockIdx.x * kLogitExperts + q;
        if (eq < E) {
            float l = red_l[2 * q][t] + red_l[2 * q + 1][t];
            float b = __fmaf_ru(fabsf(l), u, __fadd_ru(red_s[2 * q][t], red_s[2 * q + 1][t]));
            if (skew != nullptr) {
                l = l + skew[eq];
                b = __fmaf_ru(fabsf(l), u, b);
            }
            // underflowing products and subnormal sums: at most 2^-150 each, fewer
            // than 2H of them; 2^-148 per element of H covers both
            b = __fmaf_ru((float)H, 2.8025969e-45f, b);
            logit[(size_t)(m0 + t) * E + eq] = l;
            bound[(size_t)(m0 + t) * E + eq] = b;
        }
    }
}

__global__ void __launch_bounds__(256) route_logits_kernel(const uint16_t *__restrict__ x, int M, int H,
                                                           const uint16_t *__restrict__ Wr, int E,
                                                           const float *__restrict__ skew,
                                                           float *__restrict__ logit, float *__restrict__ bound) {
    // launched early (programmatic dependent launch): wait for the previous kernel,
    // then let the next one launch
    griddep_wait();
    griddep_launch_dependents();
    logits_block<16>(x, M, H, Wr, E, skew, logit, bound);
}

// ------------------------------------------------------- tiled logits (many tokens)
//
// CTA: 64 tokens x 64 experts over one half of H (grid z); 256 threads in four
// K groups of 64, each thread an 8 x 8 block of (token, expert).  Per step of 64
// elements of K the CTA stages x and W_r (bf16 -> fp32, K-major) in shared memory
// and group g takes elements 16g .. 16g+15 of the step.  A thread's products pass
// through at most 31 roundings of an inner FMA chain (two steps, 32 products; the
// first FMA onto 0 is exact), then one addition per 32 products into an outer
// running sum (H/256 of them), then the tree of the four groups (2), the sum of
// the two halves (1) and the skew (1).
constexpr int kTileT = 64, kTileE = 64, kTileKStep = 64, kTiledThreads = 256;
constexpr int kTiledStages = 3;  // bf16 staging buffers in flight
// x and W_r: two fp32 compute buffers (64 KB) and the bf16 staging ring (3 x 16 KB)
constexpr size_t kTiledSmem = 2 * 2 * 4 * 16 * 64 * sizeof(float) + (size_t)kTiledStages * 2 * 64 * 64 * sizeof(uint16_t);

__host__ __device__ inline int tiled_tree_depth(int H) { return 31 + (H + 255) / 256 + 2 + 1 + 1; }

// ||row|| for the M rows of x and the E rows of W_r, one warp per row.  Squares of
// bf16 values are exact in fp32; the computed sum of squares is within a relative
// (H/256 + 8) u of the true one, far inside the 2^-10 margin of the bound that uses
// it, and underflowed squares (at most 2^-149 each) are added back as H 2^-149.
__global__ void route_norms_kernel(const uint16_t *__restrict__ x, int M, int H, const uint16_t *__restrict__ Wr,
                                   int E, float *__restrict__ xnorm, float *__restrict__ wnorm) {
    const int lane = threadIdx.x & 31;
    const int r = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    if (r >= M + E) return;
    const uint16_t *row = r < M ? x + (size_t)r * H : Wr + (size_t)(r - M) * H;
    float ss = 0.f;
    for (int h = lane * 8; h < H; h += 256) {
        float f[8];
        unpack_bf16x8(*reinterpret_cast<const uint4 *>(row + h), f);
#pragma unroll
        for (int i = 0; i < 8; i++) ss = __fmaf_rn(f[i], f[i], ss);
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, off);
    if (lane == 0) {
        const float n = sqrtf(ss + (float)H * 1.4012985e-45f);
        if (r < M)
            xnorm[r] = n;
        else
            wnorm[r - M] = n;
    }
}

// Two fp32 values in one 64-bit register (lo in the low half, as in memory), and the
// packed fp32 arithmetic of sm_100-family cores on such pairs: each half is an
// ordinary, correctly rounded fp32 operation.
__device__ __forceinline__ unsigned long long dup_f32x2(float v) {
    unsigned long long r;
    asm("mov.b64 %0, {%1, %1};" : "=l"(r) : "f"(v));
    return r;
}
__device__ __forceinline__ float unpack_f32x2(unsigned long long v, int hi) {
    float lo_f, hi_f;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(lo_f), "=f"(hi_f) : "l"(v));
    return hi ? hi_f : lo_f;
}
// d = a * b + d (round to nearest, no flush), halfwise
__device__ __forceinline__ void fma_f32x2(unsigned long long &d, unsigned long long a, unsigned long long b) {
    asm("fma.rn.f32x2 %0, %1, %2, %0;" : "+l"(d) : "l"(a), "l"(b));
}
// d = d + a (round to nearest), halfwise
__device__ __forceinline__ void add_f32x2(unsigned long long &d, unsigned long long a) {
    asm("add.rn.f32x2 %0, %0, %1;" : "+l"(d) : "l"(a));
}

// 16-byte asynchronous copy global -> shared (both 16-byte aligned); src_bytes 0
// writes zeros without reading.
__device__ __forceinline__ void cp_async16(void *dst, const void *src, uint32_t src_bytes) {
    asm volatile("cp.async.cg.shared.global [%0], [%1], 16, %2;" ::"r"((uint32_t)__cvta_generic_to_shared(dst)),
                 "l"(src), "r"(src_bytes)
                 : "memory");
}
__device__ __forceinline__ void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
template <int N>
__device__ __forceinline__ void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// Partial logits of one half of H: half 0 into logit[], half 1 into bound[] (the
// finish kernel combines them in place).  Rows past M or E are computed on zeros and
// not stored.
//
// Each step of 64 K elements: x and W_r rows arrive as raw bf16 by cp.async in a ring
// of kTiledStages staging buffers ([row][64] with the 16-byte chunks of row r at
// position chunk ^ (r % 8), so the conversion reads are free of bank conflicts),
// then every thread converts 2 x 16 elements into the fp32 K-major buffer of the
// step (two buffers alternate), and the four K groups compute from it.
__global__ void __launch_bounds__(kTiledThreads, 1)
    route_tiled_kernel(const uint16_t *__restrict__ x, int M, int H, const uint16_t *__restrict__ Wr, int E,
                       float *__restrict__ part0, float *__restrict__ part1) {
    extern __shared__ __align__(16) float tiled_smem[];  // kTiledSmem bytes
    // fp32 compute buffers [2][group][k][64] for x and W_r, then the bf16 staging ring
    auto xs = reinterpret_cast<float(*)[4][16][kTileT]>(tiled_smem);
    auto wsm = reinterpret_cast<float(*)[4][16][kTileE]>(tiled_smem + 2 * 4 * 16 * kTileT);
    uint16_t *stage = reinterpret_cast<uint16_t *>(tiled_smem + 2 * 4 * 16 * (kTileT + kTileE));
    constexpr int kStageElems = 2 * 64 * kTileKStep;  // x rows then W_r rows, bf16
    const int tid = threadIdx.x;
    const int t0 = blockIdx.y * kTileT, e0 = blockIdx.x * kTileE;
    const int half = blockIdx.z;
    const int hlen = H / 2, hbase = half * hlen;
    const int nsteps = hlen / kTileKStep;
    // copies: 2 operands x 64 rows x 8 chunks of 16 bytes, four per thread
    auto issue = [&](int step) {
        uint16_t *st = stage + (size_t)(step % kTiledStages) * kStageElems;
#pragma unroll
        for (int q = 0; q < 4; q++) {
            const int c = tid + q * kTiledThreads;  // 0..1023
            const int op = c >> 9, row = (c >> 3) & 63, ch = c & 7;
            const int grow = (op == 0 ? t0 : e0) + row;
            const bool valid = grow < (op == 0 ? M : E);
            const uint16_t *src = (op == 0 ? x : Wr) + (size_t)(valid ? grow : 0) * H + hbase + step * kTileKStep + ch * 8;
            cp_async16(st + (size_t)op * 64 * kTileKStep + row * kTileKStep + ((ch ^ (row & 7)) * 8), src,
                       valid ? 16u : 0u);
        }
        cp_async_commit();
    };
    // conversion: thread (row = tid % 64, group g = tid / 64) takes elements 16g..16g+15
    // of its x row and its W_r row
    const int crow = tid & 63, cg = tid >> 6;
    auto convert = [&](int step) {
        const uint16_t *st = stage + (size_t)(step % kTiledStages) * kStageElems;
        const int buf = step & 1;
#pragma unroll
        for (int op = 0; op < 2; op++) {
#pragma unroll
            for (int hq = 0; hq < 2; hq++) {
                const int ch = 2 * cg + hq;
                const uint4 v = *reinterpret_cast<const uint4 *>(st + (size_t)op * 64 * kTileKStep + crow * kTileKStep +
                                                                 ((ch ^ (crow & 7)) * 8));
                float f[8];
                unpack_bf16x8(v, f);
#pragma unroll
                for (int j = 0; j < 8; j++) {
                    if (op == 0)
                        xs[buf][cg][8 * hq + j][crow] = f[j];
                    else
                        wsm[buf][cg][8 * hq + j][crow] = f[j];
                }
            }
        }
    };
    // compute: group g = tid / 64; within it ty = (tid % 64) / 8, tx = tid % 8; tokens
    // 4ty..4ty+3 and 32+4ty.., experts 4tx..4tx+3 and 32+4tx..  The accumulators are
    // packed in pairs of adjacent experts (fma.rn.f32x2 / add.rn.f32x2: two independent,
    // correctly rounded fp32 operations per instruction, so every (token, expert) sum
    // takes the same roundings in the same order as scalar fp32 code).
    const int g = tid >> 6, ty = (tid & 63) >> 3, tx = tid & 7;
    unsigned long long inner[8][4], outer[8][4];
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int p = 0; p < 4; p++) inner[i][p] = outer[i][p] = 0ull;  // +0.0f in both halves
#pragma unroll
    for (int p = 0; p < kTiledStages - 1; p++) {
        if (p < nsteps)
            issue(p);
        else
            cp_async_commit();  // empty group: the wait counts stay uniform
    }
    for (int step = 0; step < nsteps; step++) {
        cp_async_wait<kTiledStages - 2>();  // this thread's copies of `step` have landed
        __syncthreads();                     // everyone's; and everyone is done with step - 1's
                                             // compute buffer and step - 1's staging slot
        if (step + kTiledStages - 1 < nsteps)
            issue(step + kTiledStages - 1);
        else
            cp_async_commit();
        convert(step);
        __syncthreads();
        const int buf = step & 1;
#pragma unroll
        for (int k = 0; k < 16; k++) {
            const float4 a0 = *reinterpret_cast<const float4 *>(&xs[buf][g][k][4 * ty]);
            const float4 a1 = *reinterpret_cast<const float4 *>(&xs[buf][g][k][32 + 4 * ty]);
            // experts 4tx.. and 32+4tx.. as pairs (adjacent floats: lo = the lower expert)
            const ulonglong2 b01 = *reinterpret_cast<const ulonglong2 *>(&wsm[buf][g][k][4 * tx]);
            const ulonglong2 b23 = *reinterpret_cast<const ulonglong2 *>(&wsm[buf][g][k][32 + 4 * tx]);
            const float av[8] = {a0.x, a0.y, a0.z, a0.w, a1.x, a1.y, a1.z, a1.w};
            const unsigned long long bp[4] = {b01.x, b01.y, b23.x, b23.y};
#pragma unroll
            for (int i = 0; i < 8; i++) {
                const unsigned long long ap = dup_f32x2(av[i]);
#pragma unroll
                for (int p = 0; p < 4; p++) fma_f32x2(inner[i][p], ap, bp[p]);
            }
        }
        if ((step & 1) || step + 1 == nsteps) {
#pragma unroll
            for (int i = 0; i < 8; i++)
#pragma unroll
                for (int p = 0; p < 4; p++) {
                    add_f32x2(outer[i][p], inner[i][p]);
                    inner[i][p] = 0ull;
                }
        }
    }
    cp_async_wait<0>();
    __syncthreads();
    // the four groups' sums: ((g0 + g1) + (g2 + g3)), through shared memory
    float *red = tiled_smem;  // the two compute buffers: 4 x [64][64] floats
#pragma unroll
    for (int i = 0; i < 8; i++)
#pragma unroll
        for (int j = 0; j < 8; j++) {
            const int tt = (i < 4 ? 4 * ty + i : 32 + 4 * ty + i - 4);
            const int ee = (j < 4 ? 4 * tx + j : 32 + 4 * tx + j - 4);
            red[(size_t)g * 4096 + tt * 64 + ee] = unpack_f32x2(outer[i][j >> 1], j & 1);
        }
    __syncthreads();
    float *part = half == 0 ? part0 : part1;
    for (int o = tid; o < kTileT * kTileE; o += kTiledThreads) {
        const int tt = o / kTileE, ee = o % kTileE;
        if (t0 + tt < M && e0 + ee < E) {
            const float v = __fadd_rn(__fadd_rn(red[o], red[4096 + o]), __fadd_rn(red[8192 + o], red[12288 + o]));
            part[(size_t)(t0 + tt) * E + e0 + ee] = v;
        }
    }
}

// logit = half0 + half1 (+ skew), bound from the tree depth and ||x|| ||W_r[e]||
// (+ |skew|), in place over the two halves.
__global__ void route_finish_kernel(int M, int H, int E, const float *__restrict__ skew,
                                    const float *__restrict__ xnorm, const float *__restrict__ wnorm,
                                    float *__restrict__ logit, float *__restrict__ bound) {
    const size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (i >= (size_t)M * E) return;
    const int m = (int)(i / E), e = (int)(i % E);
    float l = __fadd_rn(logit[i], bound[i]);
    float S = xnorm[m] * wnorm[e];
    if (skew != nullptr) {
        const float sk = skew[e];
        l = __fadd_rn(l, sk);
        S = S + fabsf(sk);
    }
    const int d = tiled_tree_depth(H);
    // as in logits_block: (d+1) u S with the factor 1 + 2^-10 for the roundings of S
    // and of the norms; 2^-148 per product for underflow
    float b = (float)(d + 1) * 5.9604645e-8f * S * (1.0f + 9.765625e-4f);
    b = b + (float)H * 2.8025969e-45f;
    logit[i] = l;
    bound[i] = b;
}

// ------------------------------------------------------------ exact logits

__device__ __forceinline__ bool bf16_parts(uint16_t b, int &neg, unsigned int &m, int &ep) {
    const int E = (b >> 7) & 0xFF;
    neg = (b >> 15) & 1;
    m = (b & 0x7Fu) | (E ? 0x80u : 0u);
    ep = E ? E : 1;
    return E != 0xFF;
}

__device__ void limbs_add_shifted(long long *limbs, __int128 v, int o) {
    const bool neg = v < 0;
    unsigned __int128 mag = neg ? (unsigned __int128)(-v) : (unsigned __int128)v;
    const int li = o / 32, sh = o % 32;
    const unsigned __int128 s = mag << sh;  // |v| < 2^95, so s < 2^127
#pragma unroll
    for (int q = 0; q < 4; q++) {
        const long long c = (long long)((unsigned long long)(s >> (32 * q)) & 0xffffffffull);
        limbs[li + q] += neg ? -c : c;
    }
}

__device__ void limbs_normalise(long long *d) {
    for (int i = 0; i < kLimbs - 1; i++) {
        const long long c = d[i] >> 32;  // floor division by 2^32
        d[i] -= c * (1ll << 32);
        d[i + 1] += c;
    }
}

// -1, 0, +1 for a < b, a == b, a > b (normalised limbs)
__device__ int limbs_cmp(const long long *a, const long long *b) {
    if (a[kLimbs - 1] != b[kLimbs - 1]) return a[kLimbs - 1] < b[kLimbs - 1] ? -1 : 1;
    for (int i = kLimbs - 2; i >= 0; i--)
        if (a[i] != b[i]) return a[i] < b[i] ? -1 : 1;
    return 0;
}

__device__ __forceinline__ __int128 shfl_xor_i128(__int128 v, int off) {
    unsigned long long lo = (unsigned long long)v, hi = (unsigned long long)((unsigned __int128)v >> 64);
    lo = __shfl_xor_sync(0xffffffffu, lo, off);
    hi = __shfl_xor_sync(0xffffffffu, hi, off);
    return (__int128)(((unsigned __int128)hi << 64) | lo);
}

struct ExactScratch {
    long long bins[kBins];
    __int128 part[32];
    int tmax[32];
    int T0;
    int bad;
    int any_bin;          // some term fell below the 128-bit window
    int nnz;              // number of non-empty bins
    short nzl[kBins];     // their exponents
};

// The exact logit of expert e for token row xr, as normalised limbs (thread 0 writes out).
// Terms inside the 64-bit window below the largest exponent are summed in 128-bit
// registers; any term further down goes to a per-exponent bin.  Whole CTA.
__device__ void exact_logit(const uint16_t *xr, const uint16_t *wr, int H, const float *skew_e,
                            ExactScratch &sc, long long *out) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    for (int i = tid; i < kBins; i += blockDim.x) sc.bins[i] = 0;
    if (tid == 0) {
        sc.bad = 0;
        sc.any_bin = 0;
        sc.nnz = 0;
    }
    // skew term: fp32 = m * 2^(E'-150) = m * 2^(E'+118-268)
    int sk_neg = 0, sk_t = -1;
    unsigned int sk_m = 0;
    if (skew_e != nullptr) {
        const unsigned int u = __float_as_uint(*skew_e);
        const int Es = (u >> 23) & 0xFF;
        sk_neg = u >> 31;
        sk_m = (u & 0x7FFFFFu) | (Es ? 0x800000u : 0u);
        sk_t = sk_m ? (Es ? Es : 1) + 118 : -1;
        if (Es == 0xFF && tid == 0) sc.bad = 1;
    }
    // rows read 4 elements (8 bytes) at a time: H % 8 == 0 and the rows start on
    // 16-byte boundaries
    const uint2 *xv = reinterpret_cast<const uint2 *>(xr);
    const uint2 *wv = reinterpret_cast<const uint2 *>(wr);
    const int H4 = H / 4;
    int tmax = (tid == 0) ? sk_t : -1;
    bool bad = false;
    for (int h4 = tid; h4 < H4; h4 += blockDim.x) {
        const uint2 a = xv[h4], b = wv[h4];
        const unsigned int av[4] = {a.x & 0xffffu, a.x >> 16, a.y & 0xffffu, a.y >> 16};
        const unsigned int bv[4] = {b.x & 0xffffu, b.x >> 16, b.y & 0xffffu, b.y >> 16};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            int n1, n2, e1, e2;
            unsigned int m1, m2;
            const bool ok = bf16_parts((uint16_t)av[q], n1, m1, e1) & bf16_parts((uint16_t)bv[q], n2, m2, e2);
            if (!ok) bad = true;
            if (m1 && m2) tmax = max(tmax, e1 + e2);
        }
    }
    if (bad) sc.bad = 1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) tmax = max(tmax, __shfl_xor_sync(0xffffffffu, tmax, off));
    if (lane == 0) sc.tmax[warp] = tmax;
    __syncthreads();
    if (tid == 0) {
        int t = -1;
        for (int w = 0; w < (int)(blockDim.x / 32); w++) t = max(t, sc.tmax[w]);
        sc.T0 = t;
    }
    __syncthreads();
    const int lo = max(sc.T0 - 63, 0);
    __int128 acc = 0;
    bool binned = false;
    for (int h4 = tid; h4 < H4; h4 += blockDim.x) {
        const uint2 a = xv[h4], b = wv[h4];
        const unsigned int av[4] = {a.x & 0xffffu, a.x >> 16, a.y & 0xffffu, a.y >> 16};
        const unsigned int bv[4] = {b.x & 0xffffu, b.x >> 16, b.y & 0xffffu, b.y >> 16};
#pragma unroll
        for (int q = 0; q < 4; q++) {
            int n1, n2, e1, e2;
            unsigned int m1, m2;
            bf16_parts((uint16_t)av[q], n1, m1, e1);
            bf16_parts((uint16_t)bv[q], n2, m2, e2);
            if (!(m1 && m2)) continue;
            const int t = e1 + e2;
            const long long p = (long long)(m1 * m2);
            if (t >= lo) {
                const __int128 v = (__int128)p << (t - lo);
                acc += (n1 ^ n2) ? -v : v;
            } else {
                atomicAdd(reinterpret_cast<unsigned long long *>(&sc.bins[t]),
                          (unsigned long long)((n1 ^ n2) ? -p : p));
                binned = true;
            }
        }
    }
    if (tid == 0 && sk_t >= 0) {
        if (sk_t >= lo) {
            const __int128 v = (__int128)sk_m << (sk_t - lo);
            acc += sk_neg ? -v : v;
        } else {
            atomicAdd(reinterpret_cast<unsigned long long *>(&sc.bins[sk_t]),
                      (unsigned long long)(sk_neg ? -(long long)sk_m : (long long)sk_m));
            binned = true;
        }
    }
    if (binned) sc.any_bin = 1;
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) acc += shfl_xor_i128(acc, off);
    if (lane == 0) sc.part[warp] = acc;
    __syncthreads();
    // the non-empty bins below the window, found in parallel (exact integer sums:
    // the order they are added in does not matter)
    if (sc.any_bin) {
        for (int t = tid; t < lo; t += blockDim.x)
            if (sc.bins[t] != 0) sc.nzl[atomicAdd(&sc.nnz, 1)] = (short)t;
    }
    __syncthreads();
    if (tid == 0) {
        __int128 tot = 0;
        for (int w = 0; w < (int)(blockDim.x / 32); w++) tot += sc.part[w];
        for (int i = 0; i < kLimbs; i++) out[i] = 0;
        if (sc.T0 >= 0) {
            limbs_add_shifted(out, tot, lo);
            for (int q = 0; q < sc.nnz; q++) {
                const int t = sc.nzl[q];
                limbs_add_shifted(out, (__int128)sc.bins[t], t);
            }
        }
        limbs_normalise(out);
    }
    __syncthreads();
}

// ------------------------------------------------------------- selection

constexpr int kRouteThreads = 256;
constexpr int kRouteWarps = kRouteThreads / 32;
// Selection kernels are instantiated for J = 4, 8, 16 keys per thread (E up to
// 1024, 2048, 4096).
static_assert(16 * kRouteThreads == kMaxE, "the largest selection covers kMaxE experts");

__device__ __forceinline__ unsigned int orderable(float f) {
    const unsigned int u = __float_as_uint(f);
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Sort key of expert e: larger logit first, then lower index (keys are unique).
__device__ __forceinline__ unsigned long long route_key(float l, int e) {
    return ((unsigned long long)orderable(l) << 32) | (unsigned long long)(0xFFFFFFFFu - (unsigned)e);
}

__device__ __forceinline__ int key_expert(unsigned long long key) {
    return (int)(0xFFFFFFFFu - (unsigned)(key & 0xFFFFFFFFull));
}

// The warp's k largest keys in descending order into out[0..k) (0 = none): k rounds
// of a warp max; the lane holding the winner drops it and rescans its own keys.
template <int J>
__device__ void warp_topk(unsigned long long (&key)[J], int k, unsigned long long *out) {
    const int lane = threadIdx.x & 31;
    unsigned long long best = 0ull;
#pragma unroll
    for (int j = 0; j < J; j++) best = key[j] > best ? key[j] : best;
    for (int r = 0; r < k; r++) {
        unsigned long long m = best;
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            const unsigned long long o = __shfl_xor_sync(0xffffffffu, m, off);
            m = o > m ? o : m;
        }
        if (lane == 0) out[r] = m;
        if (m != 0ull && best == m) {
            best = 0ull;
#pragma unroll
            for (int j = 0; j < J; j++) {
                if (key[j] == m) key[j] = 0ull;
                best = key[j] > best ? key[j] : best;
            }
        }
    }
}

// Maximum of a 64-bit key over the warp: two single-instruction reductions, the
// high halves first, then the low halves of the lanes holding the highest one.
__device__ __forceinline__ unsigned long long warp_max_u64(unsigned long long v) {
    const unsigned int hi = (unsigned int)(v >> 32);
    const unsigned int mhi = __reduce_max_sync(0xffffffffu, hi);
    const unsigned int lo = hi == mhi ? (unsigned int)v : 0u;
    const unsigned int mlo = __reduce_max_sync(0xffffffffu, lo);
    return ((unsigned long long)mhi << 32) | mlo;
}

__device__ __forceinline__ unsigned long long warp_min_u64(unsigned long long v) {
    const unsigned int hi = (unsigned int)(v >> 32);
    const unsigned int mhi = __reduce_min_sync(0xffffffffu, hi);
    const unsigned int lo = hi == mhi ? (unsigned int)v : 0xffffffffu;
    const unsigned int mlo = __reduce_min_sync(0xffffffffu, lo);
    return ((unsigned long long)mhi << 32) | mlo;
}

constexpr int kMaxTopCand = 512;  // keys at or above the filter threshold ranked directly

struct SelectShared {
    unsigned long long wtop[kRouteWarps][kMaxK];  // each warp's top keys
    unsigned long long top[kMaxK];                // the token's top k by fp32 logit
    float top_l[kMaxK], top_b[kMaxK];             // their fp32 logits and bounds
    float final_l[kMaxK];                         // fp32 logits of the final selection
    unsigned long long ckey[kMaxTopCand];         // keys at or above the threshold
    float cl[kMaxTopCand], cb[kMaxTopCand];
    unsigned long long thr;
    int nc;
    unsigned int Lord;
    int cand[kMaxCand];                           // outsiders that may still enter
    int ncand;
    int nonfinite;
    int uncertain;
    int overflow;
    int nx;
    int aexp[kMaxCand + kMaxK];                   // candidate set ordered by upper bound
    float aup[kMaxCand + kMaxK], alo[kMaxCand + kMaxK];  // its interval ends (staged)
    int comp[kMaxCand + kMaxK];                   // interval-cluster id
    int xlist[kMaxExact];                         // experts evaluated exactly
    long long exact[kMaxExact][kLimbs];
    int final_idx[kMaxK];
    ExactScratch sc;
};

// Exact top-k and softmax of one token (whole CTA of kRouteThreads threads).
// lm / bm: the token's fp32 logits and bounds (read through L2: they may have
// been written by other CTAs of the same kernel).
template <int J>
__device__ void select_token(int m, const uint16_t *__restrict__ x, int H, const uint16_t *__restrict__ Wr, int E,
                             const float *__restrict__ skew, int k, const float *lm, const float *bm,
                             int32_t *__restrict__ idx_out, float *__restrict__ w_out, StatusWord *st,
                             SelectShared &s) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    if (tid == 0) {
        s.ncand = 0;
        s.nonfinite = 0;
        s.uncertain = 0;
        s.overflow = 0;
        s.nx = 0;
        s.Lord = 0xFFFFFFFFu;
    }
    unsigned long long key[J];
    float lv[J], bv[J];
    bool bad = false;
#pragma unroll
    for (int j = 0; j < J; j++) {
        const int e = tid + kRouteThreads * j;
        key[j] = 0ull;
        lv[j] = 0.f;
        bv[j] = 0.f;
        if (e < E) {
            lv[j] = __ldcg(lm + e);
            bv[j] = __ldcg(bm + e);
            if (!isfinite(lv[j]) || !isfinite(bv[j])) bad = true;
            key[j] = route_key(lv[j], e);
        }
    }
    __syncthreads();
    if (bad) s.nonfinite = 1;
    // (1) each warp's top q keys, q = ceil(k / warps): these 8q keys are distinct, so
    // at least k keys lie at or above the smallest of them (0 if a warp has fewer)
    const int q = (k + kRouteWarps - 1) / kRouteWarps;
    {
        unsigned long long best = 0ull;
#pragma unroll
        for (int j = 0; j < J; j++) best = key[j] > best ? key[j] : best;
        for (int r = 0; r < q; r++) {
            const unsigned long long mx = warp_max_u64(best);
            if (lane == 0) s.wtop[warp][r] = mx;
            if (mx != 0ull && best == mx) {
                best = 0ull;
#pragma unroll
                for (int j = 0; j < J; j++) {
                    if (key[j] == mx) key[j] = 0ull;
                    best = key[j] > best ? key[j] : best;
                }
            }
        }
    }
    __syncthreads();
    if (warp == 0) {  // the smallest of the kRouteWarps * q warp maxima (q <= 4)
        const unsigned long long t = lane < kRouteWarps * q ? s.wtop[lane / q][lane % q] : ~0ull;
        const unsigned long long tmin = warp_min_u64(t);
        if (lane == 0) {
            s.thr = tmin;
            s.nc = 0;
        }
    }
    __syncthreads();
    // (2) gather every key at or above the threshold: one slot reservation per warp
    // for all its keys, each key's slot from the ballots
    const unsigned long long thr = s.thr;
    {
        unsigned int bal[J];
        int cnt = 0;
#pragma unroll
        for (int j = 0; j < J; j++) {
            const int e = tid + kRouteThreads * j;
            key[j] = e < E ? route_key(lv[j], e) : 0ull;  // restore what (1) cleared
            bal[j] = __ballot_sync(0xffffffffu, key[j] != 0ull && key[j] >= thr);
            cnt += __popc(bal[j]);
        }
        if (cnt != 0) {  // warp-uniform
            int base = 0;
            if (lane == 0) base = atomicAdd(&s.nc, cnt);
            base = __shfl_sync(0xffffffffu, base, 0);
#pragma unroll
            for (int j = 0; j < J; j++) {
                const int slot = base + __popc(bal[j] & ((1u << lane) - 1u));
                if (((bal[j] >> lane) & 1u) && slot < kMaxTopCand) {
                    s.ckey[slot] = key[j];
                    s.cl[slot] = lv[j];
                    s.cb[slot] = bv[j];
                }
                base += __popc(bal[j]);
            }
        }
    }
    __syncthreads();
    const int nc = s.nc;
    if (nc <= kMaxTopCand) {
        // (3) a candidate's place is the number of larger candidates (keys are unique)
        for (int c = tid; c < nc; c += kRouteThreads) {
            const unsigned long long kc = s.ckey[c];
            int r = 0;
#pragma unroll 8
            for (int d = 0; d < nc; d++) r += s.ckey[d] > kc;
            if (r < k) {
                s.top[r] = kc;
                s.top_l[r] = s.cl[c];
                s.top_b[r] = s.cb[c];
            }
        }
    } else {
        // many keys at the threshold: k rounds of warp maxima, then over the warps
        warp_topk<J>(key, k, s.wtop[warp]);
        __syncthreads();
        if (warp == 0) {
            constexpr int JW = kRouteWarps * kMaxK / 32;
            unsigned long long wk[JW];
#pragma unroll
            for (int j = 0; j < JW; j++) {
                const int qq = lane + 32 * j;
                const int ww = qq / kMaxK, r = qq % kMaxK;
                wk[j] = (r < k) ? s.wtop[ww][r] : 0ull;
            }
            warp_topk<JW>(wk, k, s.top);
        }
        __syncthreads();
        if (tid < k) {
            const int e = key_expert(s.top[tid]);
            s.top_l[tid] = __ldcg(lm + e);
            s.top_b[tid] = __ldcg(bm + e);
        }
    }
    __syncthreads();
    const unsigned long long kth = s.top[k - 1];
    // lowest lower bound among the k winners
    if (tid < k) atomicMin(&s.Lord, orderable(__fsub_rd(s.top_l[tid], s.top_b[tid])));
    __syncthreads();
    const unsigned int Lo = s.Lord;
    // outsiders whose upper bound reaches it; adjacent winners whose intervals meet
#pragma unroll
    for (int j = 0; j < J; j++) {
        const int e = tid + kRouteThreads * j;
        if (e < E && route_key(lv[j], e) < kth && orderable(__fadd_ru(lv[j], bv[j])) >= Lo) {
            const int slot = atomicAdd(&s.ncand, 1);
            if (slot < kMaxCand) s.cand[slot] = e;
            else s.overflow = 1;
        }
    }
    if (tid + 1 < k) {
        if (!(__fsub_rd(s.top_l[tid], s.top_b[tid]) > __fadd_ru(s.top_l[tid + 1], s.top_b[tid + 1]))) s.uncertain = 1;
    }
    __syncthreads();
    auto L_ = [&](int e) { return __ldcg(lm + e); };
    auto B_ = [&](int e) { return __ldcg(bm + e); };
    if (s.nonfinite) {
        if (tid == 0) set_status(st, MOE_ERR_NONFINITE, (unsigned)m);
        if (tid < k) {
            s.final_idx[tid] = key_expert(s.top[tid]);
            s.final_l[tid] = s.top_l[tid];
        }
        __syncthreads();
    } else if (s.ncand == 0 && !s.uncertain) {
        if (tid < k) {
            s.final_idx[tid] = key_expert(s.top[tid]);
            s.final_l[tid] = s.top_l[tid];
        }
        __syncthreads();
    } else {
        // ---- slow path: interval clusters, exact evaluation where needed
        if (tid == 0) {
            atomicAdd(&st->exact_fallbacks, 1u);
            const int nc = min(s.ncand, kMaxCand);
            int n = 0;
            for (int p = 0; p < k; p++) s.aexp[n++] = key_expert(s.top[p]);
            for (int c = 0; c < nc; c++) s.aexp[n++] = s.cand[c];
            s.ncand = n;  // from here on the size of aexp
        }
        __syncthreads();
        // every candidate's interval ends, staged in shared memory by all threads
        for (int i = tid; i < s.ncand; i += kRouteThreads) {
            const int e = s.aexp[i];
            s.aup[i] = __fadd_ru(L_(e), B_(e));
            s.alo[i] = __fsub_rd(L_(e), B_(e));
        }
        __syncthreads();
        if (tid == 0) {
            const int n = s.ncand;
            // insertion sort by upper bound descending (ties: lower index first)
            for (int i = 1; i < n; i++) {
                const int e = s.aexp[i];
                const float ue = s.aup[i], le = s.alo[i];
                int j = i - 1;
                while (j >= 0) {
                    const int f = s.aexp[j];
                    const float uf = s.aup[j];
                    if (uf > ue || (uf == ue && f < e)) break;
                    s.aexp[j + 1] = f;
                    s.aup[j + 1] = uf;
                    s.alo[j + 1] = s.alo[j];
                    j--;
                }
                s.aexp[j + 1] = e;
                s.aup[j + 1] = ue;
                s.alo[j + 1] = le;
            }
            // connected components of the interval graph, in order
            int cid = 0;
            float run_lo = s.alo[0];
            s.comp[0] = 0;
            for (int i = 1; i < n; i++) {
                if (s.aup[i] >= run_lo) {
                    run_lo = fminf(run_lo, s.alo[i]);
                } else {
                    cid++;
                    run_lo = s.alo[i];
                }
                s.comp[i] = cid;
            }
            // members of multi-expert components that start inside the top k
            int pos = 0, nx = 0;
            for (int i = 0; i < n && pos < k;) {
                int j = i;
                while (j < n && s.comp[j] == s.comp[i]) j++;
                if (j - i > 1) {
                    for (int q = i; q < j; q++) {
                        if (nx < kMaxExact) s.xlist[nx++] = s.aexp[q];
                        else s.overflow = 1;
                    }
                }
                pos += j - i;
                i = j;
            }
            s.nx = nx;
        }
        __syncthreads();
        const uint16_t *xr = x + (size_t)m * H;
        for (int q = 0; q < s.nx; q++) {
            const int e = s.xlist[q];
            exact_logit(xr, Wr + (size_t)e * H, H, skew ? skew + e : nullptr, s.sc, s.exact[q]);
            if (tid == 0 && s.sc.bad) s.nonfinite = 1;
            __syncthreads();
        }
        if (tid == 0) {
            if (s.nonfinite) set_status(st, MOE_ERR_NONFINITE, (unsigned)m);
            if (s.overflow) set_status(st, MOE_ERR_UNSUPPORTED_SHAPE, (unsigned)m);
            const int n = s.ncand;
            int pos = 0;
            for (int i = 0; i < n && pos < k;) {
                int j = i;
                while (j < n && s.comp[j] == s.comp[i]) j++;
                if (j - i == 1) {
                    s.final_idx[pos++] = s.aexp[i];
                } else {
                    // order the component by exact value (desc), ties to the lower index
                    int order[kMaxCand + kMaxK];
                    int cnt = 0;
                    for (int q = i; q < j; q++) order[cnt++] = s.aexp[q];
                    auto xi = [&](int e) {
                        for (int q = 0; q < s.nx; q++)
                            if (s.xlist[q] == e) return q;
                        return -1;
                    };
                    for (int a = 1; a < cnt; a++) {
                        const int e = order[a];
                        const int qe = xi(e);
                        int b = a - 1;
                        while (b >= 0) {
                            const int f = order[b];
                            const int qf = xi(f);
                            int c;
                            if (qe >= 0 && qf >= 0) c = limbs_cmp(s.exact[qf], s.exact[qe]);
                            else c = (L_(f) > L_(e)) ? 1 : ((L_(f) < L_(e)) ? -1 : 0);  // only on overflow
                            if (c > 0 || (c == 0 && f < e)) break;
                            order[b + 1] = f;
                            b--;
                        }
                        order[b + 1] = e;
                    }
                    for (int q = 0; q < cnt && pos < k; q++) s.final_idx[pos++] = order[q];
                }
                i = j;
            }
        }
        __syncthreads();
        if (tid < k) s.final_l[tid] = L_(s.final_idx[tid]);
        __syncthreads();
    }
    // softmax over the k selected fp32 logits
    if (tid < 32) {
        const int j = tid;
        const float l = (j < k) ? s.final_l[j] : -__int_as_float(0x7f800000);
        float mx = l;
        for (int off = 16; off > 0; off >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        const float ex = (j < k) ? expf(l - mx) : 0.f;
        float z = ex;
        for (int off = 16; off > 0; off >>= 1) z += __shfl_xor_sync(0xffffffffu, z, off);
        if (j < k) {
            idx_out[(size_t)m * k + j] = s.final_idx[j];
            w_out[(size_t)m * k + j] = ex / z;
        }
    }
}

// One CTA per token.
template <int J>
__global__ void __launch_bounds__(kRouteThreads) route_select_kernel(
    const uint16_t *__restrict__ x, int H, const uint16_t *__restrict__ Wr, int E, const float *__restrict__ skew,
    int k, const float *__restrict__ logit, const float *__restrict__ bound, int32_t *__restrict__ idx_out,
    float *__restrict__ w_out, StatusWord *st) {
    // launched early (programmatic dependent launch): wait for the previous kernel,
    // then let the next one launch
    griddep_wait();
    griddep_launch_dependents();
    __shared__ SelectShared s;
    const int m = blockIdx.x;
    select_token<J>(m, x, H, Wr, E, skew, k, logit + (size_t)m * E, bound + (size_t)m * E, idx_out, w_out, st, s);
}

// Single token: logits of 4 experts per CTA as in route_logits_kernel, then the
// last CTA to finish (ticket in the status word, reset after use) selects.
template <int J>
__global__ void __launch_bounds__(kRouteThreads) route_single_kernel(
    const uint16_t *__restrict__ x, int H, const uint16_t *__restrict__ Wr, int E, const float *__restrict__ skew,
    int k, float *__restrict__ logit, float *__restrict__ bound, int32_t *__restrict__ idx_out,
    float *__restrict__ w_out, StatusWord *st, uint16_t *xhat) {
    __shared__ SelectShared s;
    __shared__ int last;
    extern __shared__ __align__(16) uint16_t xrow[];  // the (pre-scaled) token staged by logits_block
    griddep_wait();  // launched early: the previous kernel (e.g. the layer below) has completed
    logits_block<16>(x, 1, H, Wr, E, skew, logit, bound, xhat != nullptr, xhat);
    __syncthreads();
    if (threadIdx.x == 0) {
        // release: this CTA's logits (ordered by the CTA barrier) before the
        // ticket; acquire: every earlier CTA's logits after it
        unsigned int t;
        asm volatile("atom.acq_rel.gpu.global.add.u32 %0, [%1], 1;" : "=r"(t) : "l"(&st->pad[kStRouteTicket]) : "memory");
        last = (t == gridDim.x - 1);
    }
    __syncthreads();
    if (!last) return;
    // every other CTA has exited: the next kernel (the expert forward) may launch and
    // set itself up while this CTA selects; it reads idx and w only after this grid
    // has completed
    griddep_launch_dependents();
    // the exact fallback reads the token this CTA staged (x_hat when pre-scaled)
    select_token<J>(0, xhat != nullptr ? xrow : x, H, Wr, E, skew, k, logit, bound, idx_out, w_out, st, s);
    if (threadIdx.x == 0) st->pad[kStRouteTicket] = 0u;
}

template <int J>
cudaError_t launch_route_j(const uint16_t *x, int M, int H, const uint16_t *Wr, int E, const float *skew, int k,
                           int32_t *idx, float *w, const RouteWs &r, size_t smem1, StatusWord *stw, cudaStream_t st,
                           uint16_t *xhat) {
    static PerDevice smem_single(0);
    dim3 g1((E + kLogitExperts - 1) / kLogitExperts, (M + kLogitTokens - 1) / kLogitTokens);
    if (M == 1) {
        cudaError_t e = ensure_dynamic_smem(route_single_kernel<J>, smem1, smem_single);
        if (e != cudaSuccess) return e;
        TraceScope trace_scope("route_single", st);
        // programmatic dependent launch: the CTAs start while the previous kernel of the
        // stream finishes and wait for it before reading anything
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(g1.x);
        cfg.blockDim = dim3(kRouteThreads);
        cfg.dynamicSmemBytes = smem1;
        cfg.stream = st;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attr[0].val.programmaticStreamSerializationAllowed = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        e = cudaLaunchKernelEx(&cfg, route_single_kernel<J>, x, H, Wr, E, skew, k, r.logit, r.bound, idx, w, stw, xhat);
        if (e != cudaSuccess) return e;
        return cudaGetLastError();
    }
    if (M >= kTiledMinTokens && H % 128 == 0) {
        static PerDevice smem_tiled(0);
        cudaError_t e = ensure_dynamic_smem(route_tiled_kernel, kTiledSmem, smem_tiled);
        if (e != cudaSuccess) return e;
        TraceScope trace_scope("route_logits", st);
        route_norms_kernel<<<(M + E + 7) / 8, 256, 0, st>>>(x, M, H, Wr, E, r.xnorm, r.wnorm);
        route_tiled_kernel<<<dim3((E + kTileE - 1) / kTileE, (M + kTileT - 1) / kTileT, 2), kTiledThreads, kTiledSmem,
                             st>>>(
            x, M, H, Wr, E, r.logit, r.bound);
        const size_t n = (size_t)M * E;
        route_finish_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(M, H, E, skew, r.xnorm, r.wnorm, r.logit,
                                                                        r.bound);
    } else {
        TraceScope trace_scope("route_logits", st);
        cudaError_t e = launch_pdl(route_logits_kernel, g1, dim3(256), smem1, st, x, M, H, Wr, E, skew, r.logit, r.bound);
        if (e != cudaSuccess) return e;
    }
    {
        TraceScope trace_scope("route_select", st);
        cudaError_t e = launch_pdl(route_select_kernel<J>, dim3(M), dim3(kRouteThreads), 0, st, x, H, Wr, E, skew, k,
                                   r.logit, r.bound, idx, w, stw);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

}  // namespace

size_t route_workspace_bytes(int E, int M, int k) {
    (void)k;
    return route_ws(nullptr, M, E).end;
}

cudaError_t launch_route(const uint16_t *x, int M, int H, const uint16_t *Wr, int E, const float *skew, int k,
                         int32_t *idx, float *w, void *ws, cudaStream_t st, uint16_t *xhat) {
    if (M == 0) return cudaSuccess;
    RouteWs r = route_ws(ws, M, E);
    const int nt = M < kLogitTokens ? M : kLogitTokens;
    if ((size_t)nt * H * sizeof(uint16_t) > 200 * 1024) return cudaErrorInvalidValue;
    const size_t smem1 = (size_t)nt * H * sizeof(uint16_t);
    static PerDevice smem_logits(0);
    cudaError_t e = ensure_dynamic_smem(route_logits_kernel, smem1, smem_logits);
    if (e != cudaSuccess) return e;
    StatusWord *stw = reinterpret_cast<StatusWord *>(ws);
    // pre-scaled routing: one token folds the pre-scale into the router's own staging
    // of x; several tokens pre-scale first and route x_hat
    uint16_t *fused_xhat = nullptr;
    if (xhat != nullptr) {
        if (M == 1) {
            fused_xhat = xhat;
        } else {
            if ((e = launch_prescale(x, M, H, xhat, st)) != cudaSuccess) return e;
            x = xhat;
        }
    }
    if (E <= 4 * kRouteThreads)
        return launch_route_j<4>(x, M, H, Wr, E, skew, k, idx, w, r, smem1, stw, st, fused_xhat);
    if (E <= 8 * kRouteThreads)
        return launch_route_j<8>(x, M, H, Wr, E, skew, k, idx, w, r, smem1, stw, st, fused_xhat);
    return launch_route_j<16>(x, M, H, Wr, E, skew, k, idx, w, r, smem1, stw, st, fused_xhat);
}

}  // namespace moe
