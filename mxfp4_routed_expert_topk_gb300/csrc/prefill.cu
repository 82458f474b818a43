// Expert-major prefill path ("作者仍需帮助的事项" on the four-SSD page: read each
// expert once per layer and process all of its routed rows together).
//
//   sort_rank_kernel / sort_scan_kernel / sort_scatter_kernel
//        stable counting sort of the pairs p = t*k + j by expert (bit-exact perm)
//   gather_quant_kernel
//        rows of x in sorted order, quantised to MXFP8 (E4M3 + E8M0 per 32), the
//        scales written in the tile order of the GEMMs
//   grouped GEMMs (tcgen05, block-scaled)               -- gemm.cu
//   combine_kernel
//        y[t] = sum_j w[t,j] partial[inv_perm[t*k+j]] (+ residual), slot order
// The multi-token decode (launch_decode_multi) uses the same pieces with a one-CTA
// sort (sort_small_kernel) and five-part MXFP4 activations (gather_split5_f4_kernel).
#include <algorithm>

#include "moe_internal.cuh"
#include "prefill_internal.cuh"

namespace moe {
namespace {

constexpr int kSortBlock = 1024;  // pairs per block of the counting sort
constexpr int kGatherChunk = 1024; // elements of a token row per gather warp (a multiple of 256)

// Block b: local rank of each of its pairs among the block's pairs of the same
// expert (in pair order), and the block's per-expert counts cnt[b][e].
__global__ void __launch_bounds__(kSortBlock) sort_rank_kernel(const int32_t *__restrict__ idx, int P, int E,
                                                               int *__restrict__ local_rank, int *__restrict__ cnt,
                                                               StatusWord *st) {
    __shared__ int es[kSortBlock];
    __shared__ int hist[kMaxSortE];
    const int b = blockIdx.x, tid = threadIdx.x;
    const int p = b * kSortBlock + tid;
    for (int e = tid; e < E; e += blockDim.x) hist[e] = 0;
    int e = -1;
    if (p < P) {
        e = idx[p];
        if (e < 0 || e >= E) {
            set_status(st, MOE_ERR_BAD_INDEX, (unsigned)p);
            e = -1;
        }
    }
    es[tid] = e;
    __syncthreads();
    if (e >= 0) {
        int r = 0;
        for (int q = 0; q < tid; q++) r += (es[q] == e);
        local_rank[p] = r;
        atomicAdd(&hist[e], 1);
    }
    __syncthreads();
    for (int x = tid; x < E; x += blockDim.x) cnt[(size_t)b * E + x] = hist[x];
}

// Exclusive scan over the 1024 threads of a CTA (total in *total); warp_sum is
// shared scratch of 32 ints.
__device__ int block_exclusive_scan(int s, int *warp_sum, int *total) {
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    int incl = s;
    for (int off = 1; off < 32; off <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, off);
        if (lane >= off) incl += v;
    }
    __syncthreads();
    if (lane == 31) warp_sum[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int w = warp_sum[lane];
        for (int off = 1; off < 32; off <<= 1) {
            const int v = __shfl_up_sync(0xffffffffu, w, off);
            if (lane >= off) w += v;
        }
        warp_sum[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    *total = warp_sum[31];
    return incl - s + (warp > 0 ? warp_sum[warp - 1] : 0);
}

// From the per-expert totals tot[0..E) (shared): offsets = their exclusive scan,
// uexp / n_union = the experts with a non-zero total, ascending, and tile_off = the
// exclusive scan of each expert's column tiles ceil(nparts * tot[e] / BN).  1024 threads.
__device__ void offsets_and_union(const int *tot, int E, int *warp_sum, int32_t *offsets, int32_t *uexp,
                                  int32_t *n_union, int32_t *tile_off, int BN, int nparts) {
    const int tid = threadIdx.x;
    const int per = (E + blockDim.x - 1) / blockDim.x;
    const int lo = tid * per, hi = min(E, lo + per);
    int s = 0, nz = 0, nt = 0;
    for (int e = lo; e < hi; e++) {
        s += tot[e];
        nz += tot[e] > 0;
        nt += (nparts * tot[e] + BN - 1) / BN;
    }
    int total;
    int base = block_exclusive_scan(s, warp_sum, &total);
    for (int e = lo; e < hi; e++) {
        offsets[e] = base;
        base += tot[e];
    }
    if (tid == 0) offsets[E] = total;
    int nu;
    int ub = block_exclusive_scan(nz, warp_sum, &nu);
    for (int e = lo; e < hi; e++)
        if (tot[e] > 0) uexp[ub++] = e;
    if (tid == 0) *n_union = nu;
    int ntiles;
    int tb = block_exclusive_scan(nt, warp_sum, &ntiles);
    for (int e = lo; e < hi; e++) {
        tile_off[e] = tb;
        tb += (nparts * tot[e] + BN - 1) / BN;
    }
    if (tid == 0) tile_off[E] = ntiles;
}

// One CTA: prior[b][e] = sum_{b'<b} cnt[b'][e]; offsets = exclusive scan of totals;
// the list of experts that have pairs.
__global__ void __launch_bounds__(1024) sort_scan_kernel(int nblocks, int E, const int *__restrict__ cnt,
                                                         int *__restrict__ prior, int32_t *__restrict__ offsets,
                                                         int32_t *__restrict__ uexp, int32_t *__restrict__ n_union,
                                                         int32_t *__restrict__ tile_off, int BN, int nparts) {
    __shared__ int tot[kMaxSortE];
    __shared__ int warp_sum[32];
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) {
        int run = 0;
        for (int b = 0; b < nblocks; b++) {
            prior[(size_t)b * E + e] = run;
            run += cnt[(size_t)b * E + e];
        }
        tot[e] = run;
    }
    __syncthreads();
    offsets_and_union(tot, E, warp_sum, offsets, uexp, n_union, tile_off, BN, nparts);
}

// The whole sort in one CTA of 1024 threads for P <= 1024 pairs (multi-token
// decode): per-expert counts, offsets, the list of experts with pairs, and the
// stable scatter (a pair's place among its expert's pairs is the number of earlier
// pairs of the same expert).
__global__ void __launch_bounds__(1024) sort_small_kernel(const int32_t *__restrict__ idx, int P, int E,
                                                          int32_t *__restrict__ offsets, int32_t *__restrict__ uexp,
                                                          int32_t *__restrict__ n_union, int32_t *__restrict__ perm,
                                                          int32_t *__restrict__ inv_perm, int32_t *__restrict__ tile_off,
                                                          int BN, int nparts, int maxcnt, StatusWord *st) {
    // launched early (programmatic dependent launch) on the multi-row decode path:
    // wait for the previous kernel, then let the next one launch
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int tot[kMaxSortE];
    __shared__ int es[1024];
    __shared__ int warp_sum[32];
    const int tid = threadIdx.x;
    for (int e = tid; e < E; e += blockDim.x) tot[e] = 0;
    int e = -1;
    if (tid < P) {
        e = idx[tid];
        if (e < 0 || e >= E) {
            set_status(st, MOE_ERR_BAD_INDEX, (unsigned)tid);
            e = -1;
        }
    }
    es[tid] = e;
    __syncthreads();
    if (e >= 0) atomicAdd(&tot[e], 1);
    __syncthreads();
    // (maxcnt > 0) an expert named more than maxcnt times, which distinct indices per
    // row cannot give, is reported: the GEMMs reserve room for that many pairs only
    if (maxcnt > 0 && e >= 0 && tot[e] > maxcnt) set_status(st, MOE_ERR_BAD_INDEX, (unsigned)tid);
    offsets_and_union(tot, E, warp_sum, offsets, uexp, n_union, tile_off, BN, nparts);
    __syncthreads();  // offsets[] of this CTA's threads are visible to the others
    if (tid < P) {
        if (e < 0) {
            inv_perm[tid] = -1;
        } else {
            int r = 0;
            for (int q = 0; q < tid; q++) r += (es[q] == e);
            const int pos = offsets[e] + r;
            perm[pos] = tid;
            inv_perm[tid] = pos;
        }
    }
}

__global__ void sort_scatter_kernel(const int32_t *__restrict__ idx, int P, int E, const int *__restrict__ local_rank,
                                    const int *__restrict__ prior, const int32_t *__restrict__ offsets,
                                    int32_t *__restrict__ perm, int32_t *__restrict__ inv_perm) {
    const int p = blockIdx.x * blockDim.x + threadIdx.x;
    if (p >= P) return;
    const int e = idx[p];
    if (e < 0 || e >= E) {
        inv_perm[p] = -1;
        return;
    }
    const int b = p / kSortBlock;
    const int pos = offsets[e] + prior[(size_t)b * E + e] + local_rank[p];
    perm[pos] = p;
    inv_perm[p] = pos;
}

// Where the scale words of one activation row go: the tile-ordered block of its
// expert's column tile (sf_tile_word), and the row's column in that tile.
struct RowTile {
    int tile, col;
};
__device__ __forceinline__ RowTile row_tile(int e, int local_row, const int32_t *tile_off, int BN) {
    return RowTile{tile_off[e] + local_row / BN, local_row % BN};
}

// The scale words of h's padding blocks (I/32 .. Ip/32 - 1, all in the last K tile)
// for one activation row: 0, which the gate/up epilogue overwrites for the blocks
// below I/32.  The matching codes are zero in both operands.
__device__ __forceinline__ void zero_h_pad(uint8_t *hs, int I, int nsfb, RowTile rt) {
    const int ip = (I + 127) / 128 * 128;
    if (ip != I)
        *reinterpret_cast<uint32_t *>(hs + sf_tile_word(rt.tile, ip / 128, nsfb, ip / 128 - 1, rt.col)) = 0u;
}

// Token t, a chunk of kGatherChunk elements per warp: MXFP8(x[t]) once, written to the
// sorted row of each of its k pairs (inv_perm; a pair whose expert index was invalid
// has none).  Shared
// exponent X = floor(log2 amax) - 8 per 32-block (clamped to [-127, 127]); codes are
// RNE(x / 2^X) to E4M3 with saturation.  x / 2^X is exact for bf16 input.  Each lane
// takes 8 consecutive elements (a 32-block is 4 lanes, a 128-element K tile 16), so a
// warp step covers 256 elements; scales go to the tile-ordered blocks, one 4-byte word
// per K tile.
__global__ void gather_quant_kernel(const uint16_t *__restrict__ x, int T, int H, int I, int k,
                                    const int32_t *__restrict__ idx, const int32_t *__restrict__ inv_perm,
                                    const int32_t *__restrict__ offsets, const int32_t *__restrict__ tile_off, int BN,
                                    int nsfb, uint8_t *__restrict__ xq, uint8_t *__restrict__ xs,
                                    uint8_t *__restrict__ hs) {
    const int lane = threadIdx.x & 31;
    const int nchunk = (H + kGatherChunk - 1) / kGatherChunk;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int t = gw / nchunk, chunk = gw % nchunk;
    if (t >= T) return;
    // lane j < k: slot j's sorted row and its place in the tile-ordered scales
    int myrow = -1;
    RowTile myrt{0, 0};
    if (lane < k) {
        const int p = t * k + lane;
        myrow = inv_perm[p];
        if (myrow >= 0) {
            const int e = idx[p];
            myrt = row_tile(e, myrow - offsets[e], tile_off, BN);
        }
    }
    const uint16_t *xr = x + (size_t)t * H;
    const int b_end = min(H, (chunk + 1) * kGatherChunk);
    for (int b0 = chunk * kGatherChunk; b0 < b_end; b0 += 256) {
        // H is a multiple of 128: the upper half-warp may have nothing in the last step
        const bool on = b0 + lane * 8 < b_end;
        float f[8];
        if (on) {
            const uint4 v = *reinterpret_cast<const uint4 *>(xr + b0 + lane * 8);
            const unsigned int u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                f[2 * i] = __uint_as_float(u[i] << 16);
                f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) f[i] = 0.f;
        }
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 8; i++) a = fmaxf(a, fabsf(f[i]));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        int X = -127;
        if (a > 0.f) {
            int ex;
            frexpf(a, &ex);
            X = max(-127, min(127, ex - 1 - 8));
        }
        uint32_t q[2] = {0u, 0u};
#pragma unroll
        for (int i = 0; i < 4; i++) {
            unsigned short pair;
            asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;"
                : "=h"(pair)
                : "f"(ldexpf(f[2 * i + 1], -X)), "f"(ldexpf(f[2 * i], -X)));
            q[i >> 1] |= (uint32_t)pair << (16 * (i & 1));
        }
        // scale word of each K tile: the bytes of lanes 16h, 16h+4, 16h+8, 16h+12
        const uint32_t sb = (uint32_t)(X + 127);
        const uint32_t b1 = __shfl_down_sync(0xffffffffu, sb, 4);
        const uint32_t b2 = __shfl_down_sync(0xffffffffu, sb, 8);
        const uint32_t b3 = __shfl_down_sync(0xffffffffu, sb, 12);
        const uint32_t word = sb | (b1 << 8) | (b2 << 16) | (b3 << 24);
        const int kt = (b0 + lane * 8) >> 7;
        for (int j = 0; j < k; j++) {
            const int r = __shfl_sync(0xffffffffu, myrow, j);
            if (r < 0) continue;  // warp-uniform
            const int tile = __shfl_sync(0xffffffffu, myrt.tile, j);
            const int col = __shfl_sync(0xffffffffu, myrt.col, j);
            if (on) {
                *reinterpret_cast<uint2 *>(xq + (size_t)r * H + b0 + lane * 8) = make_uint2(q[0], q[1]);
                if ((lane & 15) == 0)
                    *reinterpret_cast<uint32_t *>(xs + sf_tile_word(tile, H / 128, nsfb, kt, col)) = word;
            }
        }
    }
    if (chunk == 0 && myrow >= 0) zero_h_pad(hs, I, nsfb, myrt);
}

// gather_quant_kernel with MXFP4 rows: shared exponent X = floor(log2 amax) - 2 per
// 32-block (E2M1 emax 2), codes RNE(x / 2^X) to E2M1 with saturation, two per byte
// (rows of H/2 bytes: a lane's 8 elements are one 4-byte word).  The scale words go
// to the same tile-ordered blocks.
__global__ void gather_quant4_kernel(const uint16_t *__restrict__ x, int T, int H, int I, int k,
                                     const int32_t *__restrict__ idx, const int32_t *__restrict__ inv_perm,
                                     const int32_t *__restrict__ offsets, const int32_t *__restrict__ tile_off, int BN,
                                     int nsfb, uint8_t *__restrict__ xq, uint8_t *__restrict__ xs,
                                     uint8_t *__restrict__ hs) {
    const int lane = threadIdx.x & 31;
    const int nchunk = (H + kGatherChunk - 1) / kGatherChunk;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int t = gw / nchunk, chunk = gw % nchunk;
    if (t >= T) return;
    int myrow = -1;
    RowTile myrt{0, 0};
    if (lane < k) {
        const int p = t * k + lane;
        myrow = inv_perm[p];
        if (myrow >= 0) {
            const int e = idx[p];
            myrt = row_tile(e, myrow - offsets[e], tile_off, BN);
        }
    }
    const uint16_t *xr = x + (size_t)t * H;
    const int b_end = min(H, (chunk + 1) * kGatherChunk);
    for (int b0 = chunk * kGatherChunk; b0 < b_end; b0 += 256) {
        const bool on = b0 + lane * 8 < b_end;
        float f[8];
        if (on) {
            const uint4 v = *reinterpret_cast<const uint4 *>(xr + b0 + lane * 8);
            const unsigned int u[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                f[2 * i] = __uint_as_float(u[i] << 16);
                f[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) f[i] = 0.f;
        }
        float a = 0.f;
#pragma unroll
        for (int i = 0; i < 8; i++) a = fmaxf(a, fabsf(f[i]));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
        a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
        int X = -127;
        if (a > 0.f) {
            int ex;
            frexpf(a, &ex);
            X = max(-127, min(127, ex - 1 - 2));
        }
#pragma unroll
        for (int i = 0; i < 8; i++) f[i] = ldexpf(f[i], -X);
        const uint32_t q = e2m1x8_rn(f);
        const uint32_t sb = (uint32_t)(X + 127);
        const uint32_t b1 = __shfl_down_sync(0xffffffffu, sb, 4);
        const uint32_t b2 = __shfl_down_sync(0xffffffffu, sb, 8);
        const uint32_t b3 = __shfl_down_sync(0xffffffffu, sb, 12);
        const uint32_t word = sb | (b1 << 8) | (b2 << 16) | (b3 << 24);
        const int kt = (b0 + lane * 8) >> 7;
        for (int j = 0; j < k; j++) {
            const int r = __shfl_sync(0xffffffffu, myrow, j);
            if (r < 0) continue;  // warp-uniform
            const int tile = __shfl_sync(0xffffffffu, myrt.tile, j);
            const int col = __shfl_sync(0xffffffffu, myrt.col, j);
            if (on) {
                *reinterpret_cast<uint32_t *>(xq + (size_t)r * (H / 2) + (b0 + lane * 8) / 2) = q;
                if ((lane & 15) == 0)
                    *reinterpret_cast<uint32_t *>(xs + sf_tile_word(tile, H / 128, nsfb, kt, col)) = word;
            }
        }
    }
    if (chunk == 0 && myrow >= 0) zero_h_pad(hs, I, nsfb, myrt);
}

// Row r of the sorted pairs: x[perm[r] / k] as five MXFP4 parts (rows 5r .. 5r+4, two
// codes per byte, H/2 bytes per row) for the kind::mxf4 multi-token decode, with one
// E8M0 scale per part and 32-block in the tile-ordered blocks.  One warp per (row,
// 256-element step): a lane takes 8 consecutive elements (16-byte loads), a 32-block is
// 4 lanes and a 128-element K tile 16.  Part q takes the remainder's
// shared exponent floor(log2 amax) - 2 and its E2M1 codes (RNE, saturating), and the
// remainder drops what the codes represent (exact in fp32: a code keeps the leading
// bits of the remainder, and a saturated code lies below it within a factor of two).
// Each part shrinks the block's largest remainder about fourfold; five keep the layer's
// outputs within about 3e-4 of RMS of the unquantised result.
__global__ void gather_split5_f4_kernel(const uint16_t *__restrict__ x, int H, int I, int k, int E,
                                        const int32_t *__restrict__ idx, const int32_t *__restrict__ perm,
                                        const int32_t *__restrict__ offsets, const int32_t *__restrict__ tile_off,
                                        int BN, int nsfb, uint8_t *__restrict__ xq, uint8_t *__restrict__ xs,
                                        uint8_t *__restrict__ hs) {
    // launched early (programmatic dependent launch) on the multi-row decode path:
    // wait for the previous kernel, then let the next one launch
    griddep_wait();
    griddep_launch_dependents();
    constexpr int NP = kDecodeParts;
    constexpr int kChunk = 256;  // elements per warp: one step (few rows, so many warps)
    const int lane = threadIdx.x & 31;
    const int nchunk = (H + kChunk - 1) / kChunk;
    const int gw = (blockIdx.x * blockDim.x + threadIdx.x) >> 5;
    const int r = gw / nchunk, chunk = gw % nchunk;
    if (r >= offsets[E]) return;
    const int p = perm[r];
    const int t = p / k, e = idx[p];
    RowTile rt[NP];
#pragma unroll
    for (int q = 0; q < NP; q++) rt[q] = row_tile(e, NP * (r - offsets[e]) + q, tile_off, BN);
    const uint16_t *xr = x + (size_t)t * H;
    {
        const int b0 = chunk * kChunk;
        const bool on = b0 + lane * 8 < H;  // H is a multiple of 128: the upper half-warp may be off
        float v[8];
        if (on) {
            const uint4 u4 = *reinterpret_cast<const uint4 *>(xr + b0 + lane * 8);
            const unsigned int u[4] = {u4.x, u4.y, u4.z, u4.w};
#pragma unroll
            for (int i = 0; i < 4; i++) {
                v[2 * i] = __uint_as_float(u[i] << 16);
                v[2 * i + 1] = __uint_as_float(u[i] & 0xffff0000u);
            }
        } else {
#pragma unroll
            for (int i = 0; i < 8; i++) v[i] = 0.f;
        }
        const int kt = (b0 + lane * 8) >> 7;
#pragma unroll
        for (int q = 0; q < NP; q++) {
            float a = 0.f;
#pragma unroll
            for (int i = 0; i < 8; i++) a = fmaxf(a, fabsf(v[i]));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
            a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
            const int X = mx4_exp(a);
            // 2^-X and 2^X as floats (exact scalings; 2^-127 for X = -127 is subnormal)
            const float down = __uint_as_float((uint32_t)(127 - X) << 23);
            const float up = X > -127 ? __uint_as_float((uint32_t)(X + 127) << 23) : 5.877471754e-39f;
            float sc[8];
#pragma unroll
            for (int i = 0; i < 8; i++) sc[i] = v[i] * down;
            const uint32_t c = e2m1x8_rn(sc);
#pragma unroll
            for (int i = 0; i < 8; i++) v[i] -= e2m1_nibble_value(c >> (4 * i)) * up;
            const uint32_t sb = (uint32_t)(X + 127);
            const uint32_t b1 = __shfl_down_sync(0xffffffffu, sb, 4);
            const uint32_t b2 = __shfl_down_sync(0xffffffffu, sb, 8);
            const uint32_t b3 = __shfl_down_sync(0xffffffffu, sb, 12);
            if (on) {
                *reinterpret_cast<uint32_t *>(xq + ((size_t)NP * r + q) * (H / 2) + (b0 + lane * 8) / 2) = c;
                if ((lane & 15) == 0)
                    *reinterpret_cast<uint32_t *>(xs + sf_tile_word(rt[q].tile, H / 128, nsfb, kt, rt[q].col)) =
                        sb | (b1 << 8) | (b2 << 16) | (b3 << 24);
            }
        }
    }
    if (lane == 0 && chunk == 0) {
#pragma unroll
        for (int q = 0; q < NP; q++) zero_h_pad(hs, I, nsfb, rt[q]);
    }
}

template <typename PT>
__device__ __forceinline__ float load_partial(const PT *p);
template <>
__device__ __forceinline__ float load_partial<float>(const float *p) { return *p; }
template <>
__device__ __forceinline__ float load_partial<__nv_bfloat16>(const __nv_bfloat16 *p) { return __bfloat162float(*p); }

// Block per token; threads over the hidden dimension.  Slot order j, fp32.
template <typename PT>
__global__ void combine_kernel(const PT *__restrict__ partial, const int32_t *__restrict__ inv_perm,
                               const float *__restrict__ w, int k, int H, const uint16_t *__restrict__ residual,
                               uint16_t *__restrict__ y, int chunk) {
    // launched early (programmatic dependent launch) on the multi-row decode path:
    // wait for the previous kernel, then let the next one launch
    griddep_wait();
    griddep_launch_dependents();
    __shared__ int rows[kMaxK];
    __shared__ float ws[kMaxK];
    const int t = blockIdx.x;
    const int o_lo = blockIdx.y * chunk, o_hi = min(H, o_lo + chunk);
    if (threadIdx.x < k) {
        rows[threadIdx.x] = inv_perm[(size_t)t * k + threadIdx.x];
        ws[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
    }
    __syncthreads();
    for (int o = o_lo + threadIdx.x; o < o_hi; o += blockDim.x) {
        float acc = 0.f;
        for (int j = 0; j < k; j++) {
            const int r = rows[j];
            if (r >= 0) acc = fmaf(ws[j], load_partial<PT>(partial + (size_t)r * H + o), acc);
        }
        if (residual != nullptr) acc += bf16_bits_to_float(residual[(size_t)t * H + o]);
        const __nv_bfloat16 b = __float2bfloat16_rn(acc);
        y[(size_t)t * H + o] = *reinterpret_cast<const uint16_t *>(&b);
    }
}

// Four consecutive partial elements as fp32 (16-byte or 8-byte loads).
__device__ __forceinline__ void load_partial4(const float *p, float (&v)[4]) {
    const float4 q = *reinterpret_cast<const float4 *>(p);
    v[0] = q.x;
    v[1] = q.y;
    v[2] = q.z;
    v[3] = q.w;
}
__device__ __forceinline__ void load_partial4(const __nv_bfloat16 *p, float (&v)[4]) {
    const uint2 q = *reinterpret_cast<const uint2 *>(p);
    v[0] = __uint_as_float(q.x << 16);
    v[1] = __uint_as_float(q.x & 0xffff0000u);
    v[2] = __uint_as_float(q.y << 16);
    v[3] = __uint_as_float(q.y & 0xffff0000u);
}

// combine_kernel with four consecutive outputs per thread (H a multiple of 4, rows
// 16-byte aligned): the same slot-order fp32 sums, so the same bits.
template <typename PT>
__global__ void combine4_kernel(const PT *__restrict__ partial, const int32_t *__restrict__ inv_perm,
                                const float *__restrict__ w, int k, int H, const uint16_t *__restrict__ residual,
                                uint16_t *__restrict__ y, int chunk) {
    __shared__ int rows[kMaxK];
    __shared__ float ws[kMaxK];
    const int t = blockIdx.x;
    const int o_lo = blockIdx.y * chunk, o_hi = min(H, o_lo + chunk);
    if (threadIdx.x < k) {
        rows[threadIdx.x] = inv_perm[(size_t)t * k + threadIdx.x];
        ws[threadIdx.x] = w[(size_t)t * k + threadIdx.x];
    }
    __syncthreads();
    for (int o = o_lo + 4 * threadIdx.x; o < o_hi; o += 4 * blockDim.x) {
        float acc[4] = {0.f, 0.f, 0.f, 0.f};
        for (int j = 0; j < k; j++) {
            const int r = rows[j];
            if (r >= 0) {
                float v[4];
                load_partial4(partial + (size_t)r * H + o, v);
#pragma unroll
                for (int i = 0; i < 4; i++) acc[i] = fmaf(ws[j], v[i], acc[i]);
            }
        }
        if (residual != nullptr) {
            const uint2 rv = *reinterpret_cast<const uint2 *>(residual + (size_t)t * H + o);
            acc[0] += __uint_as_float(rv.x << 16);
            acc[1] += __uint_as_float(rv.x & 0xffff0000u);
            acc[2] += __uint_as_float(rv.y << 16);
            acc[3] += __uint_as_float(rv.y & 0xffff0000u);
        }
        uint16_t b[4];
#pragma unroll
        for (int i = 0; i < 4; i++) {
            const __nv_bfloat16 bv = __float2bfloat16_rn(acc[i]);
            b[i] = *reinterpret_cast<const uint16_t *>(&bv);
        }
        *reinterpret_cast<uint2 *>(y + (size_t)t * H + o) =
            make_uint2((uint32_t)b[0] | ((uint32_t)b[1] << 16), (uint32_t)b[2] | ((uint32_t)b[3] << 16));
    }
}

// The four-wide combine's loads and stores are aligned: H % 4 == 0 and the row bases
// aligned to a whole vector.
bool combine4_ok(const void *partial, int partial_dtype, int H, const uint16_t *residual, const uint16_t *y) {
    const size_t pv = partial_dtype == MOE_PARTIAL_F32 ? 16 : 8;
    return H % 4 == 0 && (uintptr_t)partial % pv == 0 && (uintptr_t)y % 8 == 0 &&
           (residual == nullptr || (uintptr_t)residual % 8 == 0);
}

// Diagnostics: the MX-quantised h of sorted row r and 32-block b as the gate/up
// epilogue wrote it (codes, one per byte of the output, and the scale byte from the
// tile-ordered blocks).  One thread per (row, block); the row's expert is the last e
// with offsets[e] <= r.
__global__ void read_h_kernel(int E, int I, const int32_t *__restrict__ offsets, const int32_t *__restrict__ tile_off,
                              int BN, int nsfb, bool fp4, const uint8_t *__restrict__ hq_ws,
                              const uint8_t *__restrict__ hs_ws, uint8_t *__restrict__ hq, uint8_t *__restrict__ hs) {
    const int nb = I / 32;
    const size_t gid = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    const int P = offsets[E];
    if (gid >= (size_t)P * nb) return;
    const int r = (int)(gid / nb), b = (int)(gid % nb);
    int lo = 0, hi = E - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) / 2;
        if (offsets[mid] <= r) lo = mid;
        else hi = mid - 1;
    }
    const RowTile rt = row_tile(lo, r - offsets[lo], tile_off, BN);
    const int ip = (I + 127) / 128 * 128;
    hs[(size_t)r * nb + b] = hs_ws[sf_tile_word(rt.tile, ip / 128, nsfb, b >> 2, rt.col) + (b & 3)];
    if (fp4) {
        const uint8_t *src = hq_ws + (size_t)r * (I / 2) + 16 * b;
        for (int j = 0; j < 16; j++) {
            hq[(size_t)r * I + 32 * b + 2 * j] = src[j] & 15;
            hq[(size_t)r * I + 32 * b + 2 * j + 1] = src[j] >> 4;
        }
        return;
    }
    const uint4 *src = reinterpret_cast<const uint4 *>(hq_ws + (size_t)r * I + 32 * b);
    uint4 *dst = reinterpret_cast<uint4 *>(hq + (size_t)r * I + 32 * b);
    dst[0] = src[0];
    dst[1] = src[1];
}

}  // namespace

cudaError_t launch_read_h(const PoolView &v, int T, int k, int act_mode, const int32_t *offsets, const void *ws,
                          uint8_t *hq, uint8_t *hs, cudaStream_t st) {
    const bool fp4 = act_mode == MOE_ACT_MXFP4;
    const GroupedWs g = grouped_ws_layout(const_cast<void *>(ws), v.E, v.H, v.I, T, k, 1, fp4);
    const size_t n = (size_t)T * k * (v.I / 32);
    if (n == 0) return cudaSuccess;
    read_h_kernel<<<(unsigned)((n + 255) / 256), 256, 0, st>>>(v.E, v.I, offsets, g.tile_off, g.BN, g.nsfb, fp4, g.hq,
                                                               g.hs, hq, hs);
    return cudaGetLastError();
}

size_t grouped_workspace_bytes(int E, int H, int I, int T, int k) {
    // either activation format (MXFP4 tiles are narrower, so more of them)
    return std::max(grouped_ws_layout(nullptr, E, H, I, T, k, 1, false).end,
                    grouped_ws_layout(nullptr, E, H, I, T, k, 1, true).end);
}

cudaError_t launch_grouped(const PoolView &v, const uint16_t *x, int T, const int32_t *idx, int k, int act_mode,
                           int32_t *perm, int32_t *inv_perm, int32_t *offsets, void *partial, int partial_dtype,
                           void *ws, cudaStream_t st) {
    if (v.E > kMaxSortE) return cudaErrorNotSupported;
    const bool fp4 = act_mode == MOE_ACT_MXFP4;
    const GroupedWs g = grouped_ws_layout(ws, v.E, v.H, v.I, T, k, 1, fp4);
    StatusWord *stw = reinterpret_cast<StatusWord *>(ws);
    const int P = T * k;
    if (P == 0) {
        cudaMemsetAsync(offsets, 0, (size_t)(v.E + 1) * sizeof(int32_t), st);
        return cudaGetLastError();
    }
    const int nblocks = (P + kSortBlock - 1) / kSortBlock;
    {
        TraceScope trace_scope("sort_rank", st);
        sort_rank_kernel<<<nblocks, kSortBlock, 0, st>>>(idx, P, v.E, g.local_rank, g.cnt, stw);
    }
    {
        TraceScope trace_scope("sort_scan", st);
        sort_scan_kernel<<<1, 1024, 0, st>>>(nblocks, v.E, g.cnt, g.prior, offsets, g.uexp, g.n_union, g.tile_off, g.BN,
                                             1);
    }
    {
        TraceScope trace_scope("sort_scatter", st);
        sort_scatter_kernel<<<(P + 255) / 256, 256, 0, st>>>(idx, P, v.E, g.local_rank, g.prior, offsets, perm, inv_perm);
    }
    {
        TraceScope trace_scope("gather_quant", st);
        const int nchunk = (v.H + kGatherChunk - 1) / kGatherChunk;
        const unsigned nblk = (unsigned)(((size_t)T * nchunk * 32 + 255) / 256);
        if (fp4)
            gather_quant4_kernel<<<nblk, 256, 0, st>>>(x, T, v.H, v.I, k, idx, inv_perm, offsets, g.tile_off, g.BN,
                                                       g.nsfb, g.xq, g.xs, g.hs);
        else
            gather_quant_kernel<<<nblk, 256, 0, st>>>(x, T, v.H, v.I, k, idx, inv_perm, offsets, g.tile_off, g.BN,
                                                      g.nsfb, g.xq, g.xs, g.hs);
    }
    cudaError_t e = launch_grouped_gemms(v, T, k, offsets, g, partial, partial_dtype, stw, st, 1, fp4);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

size_t decode_multi_workspace_bytes(int E, int H, int I, int M, int k) {
    return decode_multi_ws_layout((void *)0, E, H, I, M, k).end;
}

cudaError_t launch_decode_multi(const PoolView &v, const uint16_t *x, int M, const int32_t *idx, const float *w, int k,
                                const uint16_t *residual, uint16_t *y, void *ws, cudaStream_t st) {
    if (v.E > kMaxSortE || v.I % 64 != 0 || v.H % 128 != 0 || M > kMaxDecodeRows) return cudaErrorNotSupported;
    const DecodeMultiWs d = decode_multi_ws_layout(ws, v.E, v.H, v.I, M, k);
    StatusWord *stw = reinterpret_cast<StatusWord *>(ws);
    const int P = M * k;
    if (P > 1024) return cudaErrorNotSupported;
    // with the k indices of a row distinct, an expert has at most M pairs, 5 M columns:
    // when that is below a tile, the GEMM stages reserve only those B rows (more stages
    // fit), and the sort reports an expert with more pairs than fit
    int bsr = (kDecodeParts * M + 15) / 16 * 16;
    if (bsr >= d.g.BN) bsr = 0;  // whole tiles (an expert with more pairs takes further tiles)
    {
        TraceScope trace_scope("sort_small", st);
        const cudaError_t e = launch_pdl(sort_small_kernel, dim3(1), dim3(1024), 0, st, idx, P, v.E, d.offsets, d.g.uexp,
                                         d.g.n_union, d.perm, d.inv_perm, d.g.tile_off, d.g.BN, kDecodeParts,
                                         bsr / kDecodeParts, stw);
        if (e != cudaSuccess) return e;
    }
    {
        TraceScope trace_scope("gather_split", st);
        const int nchunk5 = (v.H + 255) / 256;  // the five-part split takes one 256-element step per warp
        const cudaError_t e = launch_pdl(gather_split5_f4_kernel, dim3((P * nchunk5 * 32 + 255) / 256), dim3(256), 0, st,
                                         x, v.H, v.I, k, v.E, idx, d.perm, d.offsets, d.g.tile_off, d.g.BN, d.g.nsfb,
                                         d.g.xq, d.g.xs, d.g.hs);
        if (e != cudaSuccess) return e;
    }
    cudaError_t e = launch_grouped_gemms(v, M, k, d.offsets, d.g, d.partial, MOE_PARTIAL_F32, stw, st, kDecodeParts,
                                         true, bsr);
    if (e != cudaSuccess) return e;
    {
        TraceScope trace_scope("combine", st);
        // few rows: a (row, 256-element chunk) grid, one output per thread (more warps in
        // flight than four outputs per thread, which is faster at this size)
        e = launch_pdl(combine_kernel<float>, dim3(M, (v.H + 255) / 256), dim3(256), 0, st, (const float *)d.partial,
                       (const int32_t *)d.inv_perm, w, k, v.H, residual, y, 256);
        if (e != cudaSuccess) return e;
    }
    return cudaGetLastError();
}

cudaError_t launch_combine(const void *partial, int partial_dtype, const int32_t *inv_perm, const float *w, int T, int k,
                           int H, const uint16_t *residual, uint16_t *y, cudaStream_t st) {
    if (T == 0) return cudaSuccess;
    TraceScope trace_scope("combine", st);
    // one CTA per row over all of H, four outputs per thread when the rows are aligned
    // for it; or, when there are few rows, (row, 256-element chunk) CTAs with one output
    // per thread (more warps in flight)
    const bool v4 = T >= 152 && combine4_ok(partial, partial_dtype, H, residual, y);
    const int chunk = T < 152 ? 256 : H;
    const dim3 grid(T, (H + chunk - 1) / chunk);
    const int nthr = 256;
    if (partial_dtype == MOE_PARTIAL_F32) {
        if (v4)
            combine4_kernel<float><<<grid, nthr, 0, st>>>((const float *)partial, inv_perm, w, k, H, residual, y, chunk);
        else
            combine_kernel<float><<<grid, 256, 0, st>>>((const float *)partial, inv_perm, w, k, H, residual, y, chunk);
    } else {
        if (v4)
            combine4_kernel<__nv_bfloat16><<<grid, nthr, 0, st>>>((const __nv_bfloat16 *)partial, inv_perm, w, k, H,
                                                                 residual, y, chunk);
        else
            combine_kernel<__nv_bfloat16><<<grid, 256, 0, st>>>((const __nv_bfloat16 *)partial, inv_perm, w, k, H,
                                                                residual, y, chunk);
    }
    return cudaGetLastError();
}

}  // namespace moe
