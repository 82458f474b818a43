// Single-token decode of the routed-expert layer in one cooperative persistent
// kernel, one CTA per SM (the memory-bound path of the layer: each of the 16
// selected experts' packed MXFP4 weights is streamed from HBM exactly once).
//
//   phase A  g = W_g x, u = W_u x, h = silu(g) * u for every (slot, index) item;
//            each CTA owns a contiguous range of units of 8 items (one stage each)
//   grid barrier (h complete in global memory)
//   phase B  y[o] = sum_j w_j (W_d,j h_j)[o] (+ residual) for this CTA's block of
//            output rows, summed in a fixed order (deterministic, no atomics)
//
// A producer warp streams weight rows and their scale rows with bulk copies into a
// ring of shared-memory slots (evict-first in L2); W_d rows of phase B are fetched
// while phase A finishes and while CTAs wait at the grid barrier.  Consumer warps
// dequantise in registers: E2M1 pairs -> f16x2 (cvt), packed f16 FMAs over one
// 32-element scale block against the token (f16 in shared memory, scaled by a
// power of two; in phase B the warp's h in registers), then the block sum is
// scaled by its E8M0 factor in fp32.  Phase A gives each (gate row, up row) item
// to a pair of warps, phase B each selected expert to one warp.
#include <algorithm>

#include "moe_internal.cuh"
#include "sm100_async.cuh"

namespace moe {
namespace {

constexpr int kCW = 16;                       // consumer warps
constexpr int kItems = 8;                     // phase-A items per stage (a warp pair each)
constexpr int kThreadsF = (kCW + 1) * 32;     // + one producer warp
constexpr int kSlots = 3;
constexpr int kMaxJ = 7;                      // H <= 32 lanes * 32 elements * 7
constexpr int kMaxKF = 16;                    // one pair per consumer warp in phase B
constexpr int kMaxR = 4;                      // output rows per phase-B stage
constexpr int kMaxRowsCta = 64;               // output rows per CTA

struct FusedArgs {
    PoolView v;
    int k;
    int G;
    const uint16_t *x;
    const int32_t *idx;
    const float *w;
    const uint16_t *residual;
    uint16_t *y;
    float *h;            // [k][8][I/32] float4 workspace (see h_slot)
    StatusWord *st;      // grid barrier and exit counters
    unsigned int barrier_count;  // arrivals the grid barrier waits for: G (more only under
                                 // moe_debug_set_barrier_extra, to make the wait run out)
    uint32_t slot_bytes;
    int R;
    uint32_t sb_stride;  // bytes per pair of phase-B scale rows in a slot
    uint32_t sp_stride;  // != 0: all of a CTA's W_d scale rows are preloaded once, this
                         // many bytes per pair (else each phase-B stage carries its own)
    uint32_t tail_bytes; // the token / preloaded-scale region (a multiple of 16)
};

// 32 E2M1 elements (16 bytes) times the matching f16x2 input block: 16 packed f16
// FMAs in one chain, then the two halves summed in fp32.
__device__ __forceinline__ float block_dot1(const uint4 &q, const uint4 *xb) {
    const unsigned int words[4] = {q.x, q.y, q.z, q.w};
    unsigned int acc = 0u;
#pragma unroll
    for (int wd = 0; wd < 4; wd++) {
        unsigned int w0, w1, w2, w3;
        e2m1x8_to_f16x2x4(words[wd], w0, w1, w2, w3);
        const uint4 xv = xb[wd];
        acc = hfma2_u32(w0, xv.x, acc);
        acc = hfma2_u32(w1, xv.y, acc);
        acc = hfma2_u32(w2, xv.z, acc);
        acc = hfma2_u32(w3, xv.w, acc);
    }
    return f16x2_sum_to_float(acc);
}

// Position of h[p][i] in the workspace: float4 (p, e8, kb) at (p*8 + e8)*(I/32) + kb
// for 32-block kb = i/32 and eighth e8 = (i%32)/4, so that in phase B the lanes of
// a warp, one 32-block each, read 512 contiguous bytes per load instruction.
__device__ __forceinline__ size_t h_slot(int p, int i, int nkbd) {
    return ((size_t)(p * 8 + ((i & 31) >> 2)) * nkbd + (i >> 5)) * 4 + (i & 3);
}

// E8M0 byte -> 2^(b-127) with one shift: byte 0 gives 0 instead of 2^-127 (far
// below anything it scales), byte 255 (NaN) gives +inf (non-finite either way).
__device__ __forceinline__ float e8m0_fast(unsigned int b) { return __uint_as_float(b << 23); }

// f * 2^n for n in [-126, 254], exact unless the result is subnormal (then one
// rounding, as a single multiplication by 2^n would give): a scale-up above 2^127
// is split into two exact steps.
__device__ __forceinline__ float mul_pow2(float f, int n) {
    if (n > 127) {
        f *= __uint_as_float((uint32_t)(n - 127 + 127) << 23);
        n = 127;
    }
    return f * __uint_as_float((uint32_t)(n + 127) << 23);
}

__device__ __forceinline__ unsigned int pack_half2(float lo, float hi) {
    const __half2 h = __floats2half2_rn(lo, hi);
    return *reinterpret_cast<const unsigned int *>(&h);
}

__global__ void __launch_bounds__(kThreadsF, 1) decode_fused_kernel(const FusedArgs a) {
    extern __shared__ __align__(1024) unsigned char smem[];
    const PoolView &v = a.v;
    uint8_t *slots = smem;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + (size_t)kSlots * a.slot_bytes);
    uint64_t *empty = full + kSlots;
    uint64_t *fullS = empty + kSlots;  // the preloaded W_d scale rows (8 barriers: 64 bytes)
    // (slots are a multiple of 128 bytes; every region below starts 16-byte aligned)
    float *red = reinterpret_cast<float *>(full + 8);                   // [kCW][kMaxRowsCta]
    // phase A: the token, f16 [4][H/32] x 8; phase B (once the last phase-A stage has
    // been released): the preloaded W_d scale rows, [pair][sp_stride]
    uint8_t *tail = reinterpret_cast<uint8_t *>(red + kCW * kMaxRowsCta);
    uint4 *xsm = reinterpret_cast<uint4 *>(tail);
    const uint8_t *spre = tail;
    float2 *pairsum = reinterpret_cast<float2 *>(tail + a.tail_bytes);  // [2][kItems][2] half sums
    int *sidx = reinterpret_cast<int *>(pairsum + 2 * kItems * 2);      // [kMaxKF]
    int *abort_flag = sidx + kMaxKF;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int b = blockIdx.x, G = a.G, k = a.k;
    // I % 32 == 0: a unit of 8 items never straddles a pair or a 16-row group
    const int nunits = k * v.I / kItems;
    const int u_lo = (int)((long long)b * nunits / G), u_hi = (int)((long long)(b + 1) * nunits / G);
    const int nstageA = u_hi - u_lo;
    const int o_lo = (int)((long long)b * v.H / G), o_hi = (int)((long long)(b + 1) * v.H / G);
    const int rows = o_hi - o_lo;
    const int nstageB = (rows + a.R - 1) / a.R;
    const int nkb = v.H / 32, nkbd = v.I / 32;
    const int ldg = v.ld_gu, lsg = v.lds_gu;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kSlots; s++) {
            mbar_init(&full[s], 1);
            mbar_init(&empty[s], kCW);
        }
        mbar_init(fullS, 1);
        *abort_flag = 0;
        fence_mbar_init();
    }
    // launched early (programmatic dependent launch): nothing global is read before the
    // previous kernel of the stream (typically the router) has completed
    griddep_wait();
    if (threadIdx.x < k) {
        const int e = a.idx[threadIdx.x];
        const bool ok = e >= 0 && e < v.E;
        sidx[threadIdx.x] = ok ? e : -1;
        if (!ok && b == 0) set_status(a.st, MOE_ERR_BAD_INDEX, (unsigned)threadIdx.x);
    }
    __syncthreads();

    if (warp == kCW) {
        // -------------------------------------------------------------- producer
        // Lane 0 waits for a free slot and posts the stage's byte count; the copies
        // of the stage are then issued by several lanes at once (one per run in
        // phase A, one per pair in phase B).
        const uint64_t pol = policy_evict_first();
        int issued = 0;
        bool run = true;
        // phase A: one unit (8 gate rows, 8 up rows, their scale runs) per stage
        for (int s = 0; s < nstageA; s++) {
            const int slot = s % kSlots;
            const uint32_t ph = (uint32_t)(s / kSlots) & 1u;
            int go = 1;
            if (lane == 0) {
                if (!mbar_wait_or_abort(&empty[slot], ph ^ 1u, a.st, 0x100u + slot, abort_flag)) {
                    *abort_flag = 1;
                    go = 0;
                } else {
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(kItems * 2 * (ldg + lsg)));
                }
            }
            if (__shfl_sync(0xffffffffu, go, 0) == 0) {
                run = false;
                break;
            }
            if (lane < 4) {
                // 8 consecutive gate rows (lane 0), the matching up rows (1) and
                // their scale runs (2, 3)
                uint8_t *dst = slots + (size_t)slot * a.slot_bytes;
                const int n0 = (u_lo + s) * kItems;
                const int p = n0 / v.I, i = n0 % v.I;
                const int e = max(sidx[p], 0);  // invalid pairs: read expert 0, result discarded
                const uint8_t *rec = v.base + (uint64_t)e * v.rec;
                const int rg = 32 * (i / kGroupRows) + (i % kGroupRows) + (lane & 1) * kGroupRows;
                if (lane < 2)
                    bulk_g2s(dst + (size_t)(lane & 1) * kItems * ldg, rec + (uint64_t)rg * ldg,
                             (uint32_t)(kItems * ldg), &full[slot], pol);
                else
                    bulk_g2s(dst + (size_t)2 * kItems * ldg + (size_t)(lane & 1) * kItems * lsg,
                             rec + v.off_sgu + (uint64_t)rg * lsg, (uint32_t)(kItems * lsg), &full[slot], pol);
            }
            issued = s + 1;
        }
        // phase B: R rows of W_d of every pair per stage.  The scale rows of all this
        // CTA's output rows are preloaded with stage 2 (or the last one if there are
        // fewer): by then the last phase-A stage, the last reader of the token
        // region they overwrite, has been released.
        const int spre_at = a.sp_stride != 0 ? min(2, nstageB - 1) : -1;
        const uint64_t p_lo = (uint64_t)o_lo * v.lds_d / 16 * 16;
        const uint32_t pbytes = (uint32_t)(((uint64_t)o_hi * v.lds_d + 15) / 16 * 16 - p_lo);
        for (int sb = 0; run && sb < nstageB; sb++) {
            const int s = nstageA + sb;
            const int slot = s % kSlots;
            const uint32_t ph = (uint32_t)(s / kSlots) & 1u;
            const int r0 = sb * a.R, nr = min(a.R, rows - r0);
            // per-stage scale rows: the 16-byte aligned span covering rows o_lo+r0 .. +nr
            const uint64_t s_lo = (uint64_t)(o_lo + r0) * v.lds_d / 16 * 16;
            const uint64_t s_hi = ((uint64_t)(o_lo + r0 + nr) * v.lds_d + 15) / 16 * 16;
            const uint32_t sbytes = a.sp_stride != 0 ? 0u : (uint32_t)(s_hi - s_lo);
            const bool pre = sb == spre_at;
            int go = 1;
            if (lane == 0) {
                bool okw = mbar_wait_or_abort(&empty[slot], ph ^ 1u, a.st, 0x100u + slot, abort_flag);
                if (okw && pre && nstageA > 0) {
                    const int sl = nstageA - 1;  // nothing has reused its slot yet
                    okw = mbar_wait_or_abort(&empty[sl % kSlots], (uint32_t)(sl / kSlots) & 1u, a.st, 0x140u, abort_flag);
                }
                if (!okw) {
                    *abort_flag = 1;
                    go = 0;
                } else {
                    if (pre) mbar_arrive_expect_tx(fullS, (uint32_t)k * pbytes);
                    mbar_arrive_expect_tx(&full[slot], (uint32_t)(k * (nr * v.ld_d + sbytes)));
                }
            }
            if (__shfl_sync(0xffffffffu, go, 0) == 0) break;
            if (lane < k) {
                const int p = lane;
                const int e = max(sidx[p], 0);
                const uint8_t *rec = v.base + (uint64_t)e * v.rec;
                if (pre) bulk_g2s(tail + (size_t)p * a.sp_stride, rec + v.off_sd + p_lo, pbytes, fullS, pol);
                uint8_t *dst = slots + (size_t)slot * a.slot_bytes;
                bulk_g2s(dst + (size_t)p * a.R * v.ld_d, rec + v.off_d + (uint64_t)(o_lo + r0) * v.ld_d,
                         (uint32_t)(nr * v.ld_d), &full[slot], pol);
                if (sbytes != 0)
                    bulk_g2s(dst + (size_t)k * a.R * v.ld_d + (size_t)p * a.sb_stride, rec + v.off_sd + s_lo, sbytes,
                             &full[slot], pol);
            }
            issued = s + 1;
        }
        // copies still in flight must land before this CTA can exit
        if (lane == 0) {
            for (int t = max(0, issued - kSlots); t < issued; t++)
                mbar_wait(&full[t % kSlots], (uint32_t)(t / kSlots) & 1u, a.st, 0x180u);
            if (a.sp_stride != 0 && nstageB > 0 && issued - nstageA > min(2, nstageB - 1))
                mbar_wait(fullS, 0u, a.st, 0x1a0u);
        }
        __syncwarp();
        return;
    }

    // ------------------------------------------------------------------ consumers
    // the token (at most two 16-byte chunks per consumer thread) and its max |x|
    uint4 xraw[2];
    float xa = 0.f;
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int c = threadIdx.x + r * kCW * 32;
        xraw[r] = c < v.H / 8 ? __ldg(reinterpret_cast<const uint4 *>(a.x) + c) : make_uint4(0u, 0u, 0u, 0u);
        const unsigned int u[4] = {xraw[r].x, xraw[r].y, xraw[r].z, xraw[r].w};
#pragma unroll
        for (int t = 0; t < 4; t++)
            xa = fmaxf(xa, fmaxf(fabsf(__uint_as_float(u[t] << 16)), fabsf(__uint_as_float(u[t] & 0xffff0000u))));
    }
#pragma unroll
    for (int off = 16; off > 0; off >>= 1) xa = fmaxf(xa, __shfl_xor_sync(0xffffffffu, xa, off));
    if (lane == 0) red[warp] = xa;
    named_barrier(1, kCW * 32);
    float amax_x = 0.f;
    for (int ww = 0; ww < kCW; ww++) amax_x = fmaxf(amax_x, red[ww]);
    // the token as f16 scaled by 2^-sx, max|x 2^-sx| in [128, 256) (exact for bf16),
    // staged in shared memory for all consumer warps
    int sx = 0;
    if (amax_x > 0.f) {
        int ex;
        frexpf(amax_x, &ex);
        sx = ex - 1 - 7;
    }
#pragma unroll
    for (int r = 0; r < 2; r++) {
        const int c = threadIdx.x + r * kCW * 32;
        if (c < v.H / 8) {
            const unsigned int u[4] = {xraw[r].x, xraw[r].y, xraw[r].z, xraw[r].w};
            unsigned int hw[4];
#pragma unroll
            for (int t = 0; t < 4; t++)
                hw[t] = pack_half2(mul_pow2(__uint_as_float(u[t] << 16), -sx),
                                   mul_pow2(__uint_as_float(u[t] & 0xffff0000u), -sx));
            // eighth q of 32-block kb at [q][kb]: a warp's lanes read consecutive 16 bytes
            xsm[(c & 3) * nkb + (c >> 2)] = make_uint4(hw[0], hw[1], hw[2], hw[3]);
        }
    }
    named_barrier(1, kCW * 32);  // also orders the reads of red[] before its reuse in phase B

    bool ok = true;
    int s = 0;
    // ---- phase A: item j of a stage (gate row + up row) is shared by warps 2j and
    // 2j+1, which take alternate 32-block columns of the row.  Warp w issues on
    // scheduler w mod 4; which warp of the pair takes the even columns (one more
    // when the row has an odd number of columns) alternates every two items, so
    // the four schedulers get equal work.
    const int item = warp >> 1, half = (warp & 1) ^ ((item >> 1) & 1);
    for (; s < nstageA; s++) {
        const int slot = s % kSlots;
        const uint32_t ph = (uint32_t)(s / kSlots) & 1u;
        const int n = (u_lo + s) * kItems + item;
        const int p = n / v.I, i = n % v.I;
        const bool valid = sidx[p] >= 0;
        ok = mbar_wait_or_abort(&full[slot], ph, a.st, 0x200u + slot, abort_flag);
        if (!ok) *abort_flag = 1;
        float ag = 0.f, au = 0.f;
        if (ok && valid) {
            const uint8_t *base = slots + (size_t)slot * a.slot_bytes;
            const uint8_t *cg = base + (size_t)item * ldg;
            const uint8_t *cu = base + (size_t)(kItems + item) * ldg;
            const uint8_t *sgp = base + (size_t)2 * kItems * ldg + (size_t)item * lsg;
            const uint8_t *sup = base + (size_t)2 * kItems * ldg + (size_t)(kItems + item) * lsg;
#pragma unroll
            for (int jj = 0; jj < (kMaxJ + 1) / 2; jj++) {
                const int j = 2 * jj + half;
                const int kb = lane + 32 * j;
                if (j < kMaxJ && kb < nkb) {
                    uint4 xb[4];
#pragma unroll
                    for (int q = 0; q < 4; q++) xb[q] = xsm[q * nkb + kb];
                    const uint4 qg = *reinterpret_cast<const uint4 *>(cg + kb * 16);
                    const uint4 qu = *reinterpret_cast<const uint4 *>(cu + kb * 16);
                    ag = fmaf(block_dot1(qg, xb), e8m0_fast(sgp[kb]), ag);
                    au = fmaf(block_dot1(qu, xb), e8m0_fast(sup[kb]), au);
                }
            }
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[slot]);
#pragma unroll
        for (int off = 16; off > 0; off >>= 1) {
            ag += __shfl_xor_sync(0xffffffffu, ag, off);
            au += __shfl_xor_sync(0xffffffffu, au, off);
        }
        float2 *ps = pairsum + (size_t)(s & 1) * kItems * 2;
        if (lane == 0) ps[item * 2 + half] = make_float2(ag, au);
        named_barrier(2 + item, 64);  // the two warps of this item
        if (ok && valid && half == 0 && lane == 0) {
            const float2 lo = ps[item * 2], hi = ps[item * 2 + 1];
            const float gv = ldexpf(lo.x + hi.x, sx), uv = ldexpf(lo.y + hi.y, sx);
            // fast exponential and division (a few ulp): the accurate forms cost this
            // lane's warp, and the warp pair waiting for it, about 15 % of a stage
            const float hval = __fdividef(gv, 1.f + __expf(-gv)) * uv;
            a.h[h_slot(p, i, nkbd)] = hval;
        }
    }
    // every consumer warp takes part, aborted or not, so the named barriers match
    ok = grid_barrier(&a.st->pad[kStGridBarrier], a.barrier_count, 1, kCW * 32, a.st, 0x300u, abort_flag);
    // phase B remains: the next kernel of the stream (the next router) may launch; it
    // waits for this grid to complete before it reads anything
    if (threadIdx.x == 0) griddep_launch_dependents();

    // ---- phase B: each lane owns up to two (pair, 32-block) combinations of h, in
    // registers as f16 scaled by a power of two per combination (from the max |h| of
    // its 32 elements), and for every output row of a stage adds
    //   w_pair * (W_d,pair row block . h block) * scale
    // for each.  Combination 0: pair = warp, block = lane (blocks 0..31).
    // Combination 1: the tail blocks 32..I/32-1 of every pair, packed densely into
    // the lanes of as few warps as possible, starting after the warps of
    // combination 0, so that no warp instruction runs with idle lanes it could
    // have avoided.
    const int T1 = nkbd > 32 ? nkbd - 32 : 0;
    const int g = warp * 32 + lane;
    const int c1 = (g - (k * 32) % (kCW * 32) + kCW * 32) % (kCW * 32);
    const int pb[2] = {warp, T1 > 0 ? c1 / T1 : 0};
    const int kbs[2] = {lane, T1 > 0 ? 32 + c1 % T1 : 0};
    const bool pv[2] = {ok && warp < k && lane < nkbd && sidx[warp] >= 0,
                        ok && T1 > 0 && c1 < k * T1 && sidx[pb[1]] >= 0};
    uint4 hr[2][4];
    float wsc[2] = {0.f, 0.f};
    // the lanes' h blocks first (their latency overlaps the rest of the setup)
    float4 hv[2][4][2];
    {
#pragma unroll
        for (int u = 0; u < 2; u++) {
            const float4 *hp =
                reinterpret_cast<const float4 *>(a.h) + (size_t)(pv[u] ? pb[u] : 0) * 8 * nkbd + (pv[u] ? kbs[u] : 0);
#pragma unroll
            for (int q = 0; q < 8; q++) {
                const float4 z = make_float4(0.f, 0.f, 0.f, 0.f);
                hv[u][q >> 1][q & 1] = pv[u] ? __ldcg(hp + (size_t)q * nkbd) : z;
            }
        }
    }
    if (ok) {
#pragma unroll
        for (int u = 0; u < 2; u++) {
            float hm = 0.f;
#pragma unroll
            for (int q = 0; q < 4; q++)
#pragma unroll
                for (int h2 = 0; h2 < 2; h2++) {
                    const float4 f = hv[u][q][h2];
                    hm = fmaxf(hm, fmaxf(fmaxf(fabsf(f.x), fabsf(f.y)), fmaxf(fabsf(f.z), fabsf(f.w))));
                }
            // max |h 2^-sp| in [128, 256); sp in [-126, 120], so 2^-sp and 2^sp are
            // normal floats and the scaling is exact
            int sp = 0;
            if (hm > 0.f && isfinite(hm)) sp = max((int)((__float_as_uint(hm) >> 23) & 0xffu) - 127 - 7, -126);
            const float dn = __uint_as_float((uint32_t)(127 - sp) << 23);
            if (pv[u]) wsc[u] = __ldg(a.w + pb[u]) * __uint_as_float((uint32_t)(127 + sp) << 23);
#pragma unroll
            for (int q = 0; q < 4; q++) {
                const float4 f0 = hv[u][q][0], f1 = hv[u][q][1];
                hr[u][q] = make_uint4(pack_half2(f0.x * dn, f0.y * dn), pack_half2(f0.z * dn, f0.w * dn),
                                      pack_half2(f1.x * dn, f1.y * dn), pack_half2(f1.z * dn, f1.w * dn));
            }
        }
        // the preloaded scale rows (one wait per launch)
        if (a.sp_stride != 0 && nstageB > 0) {
            ok = mbar_wait_or_abort(fullS, 0u, a.st, 0x3a0u, abort_flag);
            if (!ok) *abort_flag = 1;
        }
        const int soffP = (int)((uint64_t)o_lo * v.lds_d % 16);
        for (int sb = 0; sb < nstageB; sb++, s++) {  // every lane runs every stage (warp shuffles below)
            const int slot = s % kSlots;
            const uint32_t ph = (uint32_t)(s / kSlots) & 1u;
            const int r0 = sb * a.R, nr = min(a.R, rows - r0);
            const int soff = (int)((uint64_t)(o_lo + r0) * v.lds_d % 16);  // first scale row in the span
            ok = mbar_wait_or_abort(&full[slot], ph, a.st, 0x400u + slot, abort_flag);
            if (!ok) *abort_flag = 1;
            float part[kMaxR] = {0.f, 0.f, 0.f, 0.f};
            if (ok) {
                const uint8_t *base = slots + (size_t)slot * a.slot_bytes;
#pragma unroll
                for (int u = 0; u < 2; u++) {
                    if (!pv[u]) continue;
                    const uint8_t *row = base + (size_t)pb[u] * a.R * v.ld_d + kbs[u] * 16;
                    const uint8_t *srow = a.sp_stride != 0
                                              ? spre + (size_t)pb[u] * a.sp_stride + soffP + (size_t)r0 * v.lds_d + kbs[u]
                                              : base + (size_t)k * a.R * v.ld_d + (size_t)pb[u] * a.sb_stride + soff + kbs[u];
#pragma unroll
                    for (int r = 0; r < kMaxR; r++) {
                        if (r >= nr) continue;
                        const uint4 q = *reinterpret_cast<const uint4 *>(row + (size_t)r * v.ld_d);
                        part[r] = fmaf(wsc[u] * block_dot1(q, hr[u]), e8m0_fast(srow[(size_t)r * v.lds_d]), part[r]);
                    }
                }
            }
            __syncwarp();
            if (lane == 0) mbar_arrive(&empty[slot]);
#pragma unroll
            for (int r = 0; r < kMaxR; r++) {
                float t = part[r];
#pragma unroll
                for (int off = 16; off > 0; off >>= 1) t += __shfl_xor_sync(0xffffffffu, t, off);
                if (lane == 0 && r < nr) red[warp * kMaxRowsCta + r0 + r] = t;
            }
        }
    }
    named_barrier(1, kCW * 32);
    if (ok && !*(volatile int *)abort_flag) {
        for (int t = threadIdx.x; t < rows; t += kCW * 32) {
            float acc = 0.f;
            for (int ww = 0; ww < kCW; ww++) acc += red[ww * kMaxRowsCta + t];
            const int o = o_lo + t;
            if (a.residual != nullptr) acc += bf16_bits_to_float(a.residual[o]);
            const __nv_bfloat16 bv = __float2bfloat16_rn(acc);
            a.y[o] = *reinterpret_cast<const uint16_t *>(&bv);
        }
    }
    // every CTA is past the grid barrier: the last one here resets both counters
    if (threadIdx.x == 0) {
        __threadfence();
        if (atomicAdd(&a.st->pad[kStExitCount], 1u) == (unsigned)G - 1u) {
            atomicExch(&a.st->pad[kStGridBarrier], 0u);
            atomicExch(&a.st->pad[kStExitCount], 0u);
        }
    }
}

PerDevice g_sms(0);
PerDevice g_smem_max(0);
PerDevice g_grid(-1);  // co-resident CTAs of the fused kernel (0: unusable), per device
PerDevice g_smem_set(0);
unsigned int g_barrier_extra = 0;  // test hook: arrivals the grid barrier waits for beyond G

}  // namespace

cudaError_t set_wait_limit_decode_fused(uint64_t ns) { return set_wait_limit_here(ns); }

void set_barrier_extra(unsigned int extra) { g_barrier_extra = extra; }

// Launch the fused kernel if the shape allows it; cudaErrorNotSupported otherwise
// (the caller then uses the general decode kernels).
cudaError_t launch_decode_fused(const PoolView &v, const uint16_t *x, const int32_t *idx, const float *w, int k,
                                const uint16_t *residual, uint16_t *y, void *ws, cudaStream_t st) {
    if (!(k <= kMaxKF && v.H <= 32 * 32 * kMaxJ && v.H % 512 == 0 && v.I <= 64 * 32))
        return cudaErrorNotSupported;
    int dev = 0, sms = 0, smem_max = 0;
    cudaError_t e = current_device(&dev);
    if (e != cudaSuccess) return e;
    if ((e = device_attr(cudaDevAttrMultiProcessorCount, g_sms, &sms)) != cudaSuccess) return e;
    if ((e = device_attr(cudaDevAttrMaxSharedMemoryPerBlockOptin, g_smem_max, &smem_max)) != cudaSuccess) return e;
    FusedArgs fa;
    fa.v = v;
    fa.k = k;
    fa.x = x;
    fa.idx = idx;
    fa.w = w;
    fa.residual = residual;
    fa.y = y;
    fa.h = reinterpret_cast<float *>((char *)ws + 256);
    fa.st = reinterpret_cast<StatusWord *>(ws);
    const uint32_t slotA = (uint32_t)(2 * kItems * (v.ld_gu + v.lds_gu));
    // phase-B stage: R rows of W_d per pair plus a 16-byte aligned span of their scale rows
    auto sb_of = [&](int r) { return (uint32_t)((r * v.lds_d + 15) / 16 * 16 + 32); };
    auto stageB = [&](int r) { return (uint32_t)k * ((uint32_t)r * v.ld_d + sb_of(r)); };
    int R = kMaxR;
    while (R > 1 && stageB(R) > slotA) R--;
    fa.R = R;
    fa.sb_stride = sb_of(R);
    const uint32_t slot_need = slotA > stageB(R) ? slotA : stageB(R);
    fa.slot_bytes = (slot_need + 127) / 128 * 128;
    // everything but the token / preloaded-scale region
    const size_t head = (size_t)kSlots * fa.slot_bytes + 8 * sizeof(uint64_t) + (size_t)kCW * kMaxRowsCta * sizeof(float) +
                        2 * kItems * 2 * sizeof(float2) + (kMaxKF + 4) * sizeof(int);
    // the W_d scale rows of a CTA's output rows (at most ceil(H / SMs) of them), one
    // 16-byte aligned span per pair, if they fit in shared memory
    const int rows_max = (v.H + sms - 1) / sms;
    const uint32_t sp = (uint32_t)((rows_max * v.lds_d + 15) / 16 * 16 + 32);
    const size_t tok = (size_t)v.H * 2;
    fa.sp_stride = head + std::max(tok, (size_t)k * sp) <= (size_t)smem_max ? sp : 0u;
    fa.tail_bytes = (uint32_t)std::max(tok, (size_t)k * fa.sp_stride);
    const size_t smem = head + fa.tail_bytes;
    e = ensure_dynamic_smem(decode_fused_kernel, smem, g_smem_set);
    if (e != cudaSuccess) return e;
    int grid = g_grid.v[dev].load(std::memory_order_relaxed);
    if (grid < 0) {
        int per_sm = 0;
        e = cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_fused_kernel, kThreadsF, smem);
        if (e != cudaSuccess) return e;
        grid = per_sm >= 1 ? sms : 0;
        g_grid.v[dev].store(grid, std::memory_order_relaxed);
    }
    fa.G = grid;
    fa.barrier_count = (unsigned int)grid + g_barrier_extra;
    if (fa.G <= 0 || fa.G > kMaxFusedGrid || (v.H + fa.G - 1) / fa.G > kMaxRowsCta) return cudaErrorNotSupported;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(fa.G);
    cfg.blockDim = dim3(kThreadsF);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs co-resident: the grid barrier needs it
    attr[0].val.cooperative = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlap the launch with the
    attr[1].val.programmaticStreamSerializationAllowed = 1;          // previous kernel's tail
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    TraceScope trace_scope("decode_fused", st);
    e = cudaLaunchKernelEx(&cfg, decode_fused_kernel, fa);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

}  // namespace moe
