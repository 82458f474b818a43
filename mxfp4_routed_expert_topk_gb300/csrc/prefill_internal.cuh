// Internal declarations of the expert-major prefill path.
#pragma once

#include <cuda_fp16.h>

#include "moe_internal.cuh"

namespace moe {

constexpr int kMaxSortE = 4096;  // experts supported by the grouped path

constexpr int kMaxBN = 192;      // accumulator columns of a grouped-GEMM tile
constexpr int kMaxBN4 = 192;     // ... with MXFP4 activations

// Accumulator columns per tile (BN) of the grouped GEMMs for P pairs over E experts,
// T rows, nparts activation rows per pair; 0 when the shape is not supported.
// nparts = 1: 1.5 times the mean rows per expert rounded up to 32, 32..192 (an expert
// with more rows takes several tiles; narrow tiles let the GEMMs run two CTAs per SM);
// the same rule with MXFP4 activations (fp4).
// nparts = 5: tiles of 16 pairs.
__host__ __device__ inline int grouped_bn(int P, int E, int T, int nparts, bool fp4 = false) {
    if (nparts == 5) return 80;  // five MXFP4 parts: one group of 16 pairs per tile (an expert
                                 // with more rows takes further tiles); one scale atom
    const int cap = fp4 ? kMaxBN4 : kMaxBN;
    const int mean = (P + E - 1) / E;
    int bn = (3 * mean / 2 + 31) / 32 * 32;
    return bn < 32 ? 32 : (bn > cap ? cap : bn);
}

// Scale factors of the activation operand (B) in the layout the MMA consumes, one
// block per (expert, column tile): tile T_e + t of expert e (T_e = tile_off[e]) holds,
// for each K tile kt of 128 elements, nsfb = ceil(BN / 128) atoms of 512 bytes.  Column
// c of the tile (activation row nparts * offsets[e] + t * BN + c) belongs to atom c / 128
// and keeps the 4 scale bytes of its K tile (scale block 4kt+j at byte j of the word)
// in row c % 32 of the atom (16 bytes, word (c / 32) % 4): the 32 x 16-byte layout that
// tcgen05.cp copies into TMEM.  With two atoms, their rows are interleaved by groups of
// 8 (row group g of atom a at byte g * 256 + a * 128): each atom is then one 32x128b
// copy whose row groups are 256 bytes apart; with one atom this is the plain atom.
// Bytes of columns past the tile's rows are never read by a result that is kept.  Byte
// offset of the word of (tile, kt, c):
__host__ __device__ inline size_t sf_tile_word(int tile, int nkt, int nsfb, int kt, int c) {
    return ((size_t)tile * nkt + kt) * (size_t)nsfb * 512 + (size_t)((c & 31) >> 3) * (size_t)nsfb * 128 +
           (size_t)(c >> 7) * 128 + (size_t)(c & 7) * 16 + (size_t)((c >> 5) & 3) * 4;
}

// Bytes of B's scale factors per 128-K tile in shared memory: the atom, or the
// interleaved 1 KB two-atom block (each atom reaches all four TMEM lane quadrants
// through its own .warpx4 copy, so nothing is replicated in shared memory).
__host__ __device__ inline uint32_t sfb_stage_bytes(int nsfb) { return nsfb == 1 ? 512u : 1024u; }

// Activation rows of the grouped GEMMs.  nparts = 1: one MXFP8 row per pair (OCP
// rule, the prefill path), or with fp4 one MXFP4 row (two E2M1 codes per byte,
// element 2j in the low nibble: rows of H/2 and I/2 bytes).  nparts = 5: the value
// is the sum of five MXFP4 parts, each with its own E8M0 scales (the multi-token
// decode path); row 5r+q holds part q of pair r.
struct GroupedWs {
    int *local_rank;  // [P]
    int *cnt;         // [nblocks][E]
    int *prior;       // [nblocks][E]
    int32_t *uexp;    // [E] the experts with at least one pair, ascending
    int32_t *n_union; // [1] their number
    int32_t *tile_off;// [E+1] first column tile of each expert (exclusive scan of its tiles)
    int BN, nsfb;     // columns per tile, 512-byte scale atoms per tile and K tile
    int max_tiles;    // bound on the column tiles of all experts
    uint8_t *xq;      // [nparts*P][H]    E4M3 rows of x in sorted order ([P][H/2] E2M1 pairs with fp4)
    uint8_t *xs;      // [max_tiles][H/128][nsfb][512]  their E8M0 scales (sf_tile_word)
    uint8_t *hq;      // [nparts*P][I]    E4M3 rows of h in sorted order ([P][I/2] with fp4)
    uint8_t *hs;      // [max_tiles][Ip/128][nsfb][512] Ip = I rounded up to 128; the
                      //                   scale bytes of blocks I/32.. are 0 (2^-127)
    size_t end;       // total bytes
};

__host__ __device__ inline GroupedWs grouped_ws_layout(void *ws, int E, int H, int I, int T, int k, int nparts = 1,
                                                       bool fp4 = false) {
    GroupedWs g;
    const size_t P = (size_t)T * k;
    const size_t R = P * (size_t)nparts;
    const size_t nblocks = (P + 1023) / 1024;
    const int bn = grouped_bn((int)P, E, T, nparts, fp4);
    g.BN = bn > 0 ? bn : 48;  // (an unsupported shape is refused at launch)
    g.nsfb = (g.BN + 127) / 128;
    // sum over experts of ceil(rows_e / BN) <= R / BN + (experts with rows)
    g.max_tiles = (int)((R + g.BN - 1) / g.BN + (P < (size_t)E ? P : (size_t)E));
    const size_t ip = ((size_t)I + 127) / 128 * 128;
    char *base = (char *)ws;
    size_t o = 256;
    g.local_rank = (int *)(base + o);  o += align_up(P * 4, 1024);
    g.cnt = (int *)(base + o);         o += align_up(nblocks * E * 4, 1024);
    g.prior = (int *)(base + o);       o += align_up(nblocks * E * 4, 1024);
    g.uexp = (int32_t *)(base + o);    o += align_up((size_t)E * 4, 256);
    g.n_union = (int32_t *)(base + o); o += 256;
    g.tile_off = (int32_t *)(base + o); o += align_up(((size_t)E + 1) * 4, 256);
    g.xq = (uint8_t *)(base + o);      o += align_up(R * H, 1024);
    g.xs = (uint8_t *)(base + o);      o += align_up((size_t)g.max_tiles * (H / 128) * g.nsfb * 512, 1024);
    g.hq = (uint8_t *)(base + o);      o += align_up(R * I, 1024);
    g.hs = (uint8_t *)(base + o);      o += align_up((size_t)g.max_tiles * (ip / 128) * g.nsfb * 512, 1024);
    g.end = o;
    return g;
}

// The multi-token decode through the grouped GEMMs: the grouped workspace with five
// MXFP4 activation parts, then the sort's outputs and the fp32 expert output rows.
struct DecodeMultiWs {
    GroupedWs g;
    int32_t *perm;      // [P]
    int32_t *inv_perm;  // [P]
    int32_t *offsets;   // [E+1]
    float *partial;     // [P][H]
    size_t end;
};

// The multi-token decode writes each row and h as five MXFP4 parts (kind::mxf4).
constexpr int kDecodeParts = 5;

__host__ __device__ inline DecodeMultiWs decode_multi_ws_layout(void *ws, int E, int H, int I, int M, int k) {
    DecodeMultiWs d;
    d.g = grouped_ws_layout(ws, E, H, I, M, k, kDecodeParts, true);
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

// MXFP4 shared exponent of a block with max |v| = amax (finite, non-negative):
// floor(log2 amax) - 2, or -127 for zero and values below 2^-125 (OCP MX rule).
__device__ __forceinline__ int mx4_exp(float amax) { return max(-127, (int)(__float_as_uint(amax) >> 23) - 129); }

// Value of an E2M1 code (the low 4 bits of `nib`): sign bit 3, exponent bits 2..1
// (bias 1), mantissa bit 0.
__device__ __forceinline__ float e2m1_nibble_value(uint32_t nib) {
    const uint32_t m = nib & 7u, e = m >> 1, f = m & 1u;
    const float mag = e == 0u ? 0.5f * (float)f : __uint_as_float((126u + e) << 23) * (1.f + 0.5f * (float)f);
    return (nib & 8u) ? -mag : mag;
}

// Eight values -> eight E2M1 codes (round to nearest even, saturating at +-6), two
// per byte with element 2j in the low nibble: bytes 0..3 of the result.
__device__ __forceinline__ uint32_t e2m1x8_rn(const float (&f)[8]) {
    uint32_t r;
    asm("{\n\t.reg .b8 q0, q1, q2, q3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q0, %2, %1;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q1, %4, %3;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q2, %6, %5;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q3, %8, %7;\n\t"
        "mov.b32 %0, {q0, q1, q2, q3};\n\t}"
        : "=r"(r)
        : "f"(f[0]), "f"(f[1]), "f"(f[2]), "f"(f[3]), "f"(f[4]), "f"(f[5]), "f"(f[6]), "f"(f[7]));
    return r;
}

// Two values -> one byte of E2M1 codes (lo in the low nibble).
__device__ __forceinline__ uint8_t e2m1x2_rn(float lo, float hi) {
    uint32_t r;
    asm("{\n\t.reg .b8 q;\n\t"
        "cvt.rn.satfinite.e2m1x2.f32 q, %1, %2;\n\t"
        "mov.b32 %0, {q, q, q, q};\n\t}"
        : "=r"(r)
        : "f"(hi), "f"(lo));
    return (uint8_t)(r & 0xFFu);
}

// The two grouped block-scaled GEMMs (gate/up with SwiGLU and the MX quantisation of
// h, then down), over the sorted rows.  max_cols > 0 (five-part rows only): no tile
// has more columns than this (the sort reports an expert with more pairs as a bad
// index), so each pipeline stage reserves only that many B rows.
cudaError_t launch_grouped_gemms(const PoolView &v, int T, int k, const int32_t *offsets, const GroupedWs &g,
                                 void *partial, int partial_dtype, StatusWord *st, cudaStream_t stream,
                                 int nparts = 1, bool fp4 = false, int max_cols = 0);

// Multi-token decode (M > 1) through the grouped GEMMs with five-part MXFP4
// activations; cudaErrorNotSupported for shapes the GEMMs do not take.
cudaError_t launch_decode_multi(const PoolView &v, const uint16_t *x, int M, const int32_t *idx, const float *w, int k,
                                const uint16_t *residual, uint16_t *y, void *ws, cudaStream_t st);
size_t decode_multi_workspace_bytes(int E, int H, int I, int M, int k);

}  // namespace moe
