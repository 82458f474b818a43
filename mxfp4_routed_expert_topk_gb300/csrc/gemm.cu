// Grouped block-scaled GEMMs of the expert-major prefill path on the 5th-generation
// tensor cores (tcgen05): weights are the MMA's A operand (E2M1, one E8M0 scale per
// 32 along K, 128 rows per tile), the expert's sorted token rows are B (up to BN rows
// per tile), fp32 accumulators in TMEM.  Two activation formats:
//   MXFP8 rows: kind::mxf8f6f4 (E2M1 x E4M3, the FP8 rate), K = 32 per MMA; A arrives
//          unpacked by the tensor copy (16 E2M1 values per 16 bytes), 128 K per stage;
//   MXFP4 rows (FP4 template): kind::mxf4, scale_vec::2X (E2M1 x E2M1, the FP4 rate),
//          K = 64 per MMA; both operands stay packed (two codes per byte), 256 K per
//          stage, two scale atoms per operand and stage.
//
//   GEMM 1 (gate/up): A = W_gu (2I rows, K = H), B = MXFP8 x rows; epilogue
//            h = silu(g) * u from the interleaved gate/up rows, quantised to MXFP8
//            along I (the same rule as x) -> hq, hs
//   GEMM 2 (down):    A = W_d (H rows, K = I, zero padded to 128), B = MXFP8 h rows;
//            epilogue writes the unweighted expert output rows (fp32 or bf16)
//
// Persistent: CTAs walk the (expert with pairs, row tiles of A) items with a stride of
// the grid, with as many pipeline stages as their share of shared memory holds (the
// stream of K steps runs on across items).  Warp 0 issues a stage's four copies (the
// tensor copies of A and B, and one bulk copy each of their scale factors, which both
// operands keep in memory already in the 32x16-byte layout tcgen05.cp expects: the
// pool's tensor-core scale planes and the tile-ordered activation scales); warp 1 owns
// TMEM and issues the scale copies and MMAs into one of two accumulators; the epilogue
// warps drain the other accumulator, so a tile's epilogue overlaps the next tile's
// MMAs.  Two shapes (GemmShape): one CTA of 12 warps per SM (two epilogue warpgroups)
// or two CTAs of 6 warps per SM (one), chosen per launch by the tile width.  Wide
// one-part tiles can also run on CTA pairs (grouped_gemm_pair_kernel: a cluster of two
// CTAs on two SMs, tcgen05 MMAs of cta_group::2 with M = 256 issued by the even CTA;
// each CTA copies its 128 weight rows and half of the tile's activation rows, and its
// tensor copies count on the even CTA's barrier).  With five-part MXFP4 activations
// (nparts = 5, the multi-token decode) each sorted pair has five B rows whose columns
// the epilogue sums.  Every wait is bounded (MOE_ERR_TIMEOUT), and nothing exits with
// copies or MMAs in flight.
#include <algorithm>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "prefill_internal.cuh"
#include "sm100_async.cuh"

namespace moe {
namespace {

constexpr int kMaxStages = 12;
constexpr int kTileM = 128;
constexpr int kTileK = 128;   // elements (bytes in shared memory for both operands)

// Two shapes of the kernel (template parameter NT = threads per CTA):
//   NT = 384, one CTA per SM: warp 0 copies, warp 1 MMAs, warps 4-7 and 8-11 two
//             epilogue warpgroups taking alternate column groups (2, 3 idle);
//   NT = 192, two CTAs per SM: warp 0 copies, warp 1 MMAs, warps 2-5 one epilogue
//             warpgroup.  Two CTAs give each SM two independent copy and MMA streams,
//             which overlap the fixed per-instruction time of narrow (small N) MMAs.
// An epilogue warp w reads TMEM lanes 32 (w % 4) ...
constexpr int kEpiWarps = 8;  // the most epilogue warps (shared-memory sizing)
template <int NT>
struct GemmShape {
    static constexpr int kEpiFirst = NT == 192 ? 2 : 4;          // first epilogue warp
    static constexpr int kEpiWarps = NT / 32 - kEpiFirst;         // 4 or 8
    static constexpr int kWarpGroups = kEpiWarps / 4;             // 1 or 2
    static constexpr int kCtasPerSm = NT == 192 ? 2 : 1;
};

struct GemmArgs {
    int mode;            // 1: gate/up + SwiGLU + MX quantisation of h, 2: down
    int E;
    int nkt;             // pipeline stages along K (128 K each, 256 with FP4 rows)
    int nkt_sf;          // K tiles of 128 (the unit of the scale-factor blocks)
    uint64_t a_sf_off;   // offset in a record of A's scale factors in tensor-core order [nkt][nmt][512]
    const uint8_t *pool;
    uint64_t rec;
    const int32_t *offsets;
    const int32_t *tile_off;  // first column tile of each expert
    const int32_t *uexp;      // experts with pairs
    const int32_t *n_union;
    const uint8_t *bscale;    // xs or hs in tile order (sf_tile_word), nkt K tiles
    int BN;              // columns of the accumulator tile (multiple of 16)
    int bbox;            // rows per tensor copy of B: BN (one copy per stage), or 16 (as many
                         // copies as the tile's MMA width needs: narrow tiles)
    int bsr;             // B rows reserved per pipeline stage in shared memory: BN, or fewer
                         // (a multiple of 16, with bbox = 16) when no tile has more columns
    int nsfb;            // 512-byte scale atoms of B per K tile = ceil(BN / 128)
    int ns;              // pipeline stages
    int nmt;             // 128-row tiles of A per expert
    int tpi;             // 128-row tiles per work item (1, or 2: one 256-row tensor copy of A)
    int nacc;            // accumulator buffers in TMEM: 2 (a tile's epilogue overlaps the next
                         // tile's MMAs) or 1 (when TMEM is short; two CTAs per SM overlap instead)
    uint32_t tmem_cols;
    // epilogue outputs
    int I;               // intermediate size (gate/up epilogue)
    int H;               // hidden size (down epilogue)
    uint8_t *hq;         // [P][I]
    uint8_t *hs;         // tile order, nkt_h K tiles
    int nkt_h;           // Ip / 128
    void *partial;       // [P][H]
    int partial_dtype;
    int nparts;          // activation rows per pair (1, or 5: the MXFP4 parts of the multi-token decode)
    int pair;            // 1: CTA pairs (cta_group::2), an item is two 128-row tiles of A, one per CTA,
                         // and each CTA holds bsr = BN / 2 rows of B per stage
    StatusWord *st;
};

// ---------------------------------------------------------------- PTX helpers

__device__ __forceinline__ void tma_load_3d(void *dst, const CUtensorMap *map, int c0, int c1, int c2, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
        : "memory");
}

__device__ __forceinline__ void tma_load_2d(void *dst, const CUtensorMap *map, int c0, int c1, uint64_t *bar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];" ::"r"(
            smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(smem_u32(bar))
        : "memory");
}

// A pair's tensor copies: into this CTA's shared memory, completion counted on the even
// CTA's barrier (`mbar`, its address in the cluster window), so that barrier's phase
// covers the copies of both CTAs.
__device__ __forceinline__ void tma_load_3d_pair(void *dst, const CUtensorMap *map, int c0, int c1, int c2,
                                                 uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, %3, "
        "%4}], [%5];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(mbar)
        : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair(void *dst, const CUtensorMap *map, int c0, int c1, uint32_t mbar) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cta.global.tile.mbarrier::complete_tx::bytes.cta_group::2 [%0], [%1, {%2, "
        "%3}], [%4];" ::"r"(smem_u32(dst)),
        "l"(map), "r"(c0), "r"(c1), "r"(mbar)
        : "memory");
}

// Shared-memory matrix descriptor of tcgen05: start address, leading / stride
// byte offsets (16-byte units), fixed version bits 46..48 = 0b001, swizzle mode.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
    uint64_t d = 0;
    d |= (uint64_t)((addr & 0x3FFFFu) >> 4);
    d |= (uint64_t)((lbo >> 4) & 0x3FFFu) << 16;
    d |= (uint64_t)((sbo >> 4) & 0x3FFFu) << 32;
    d |= (uint64_t)1 << 46;
    d |= (uint64_t)(swizzle & 7u) << 61;
    return d;
}
constexpr uint32_t kSwizzle128B = 2;
constexpr uint32_t kSwizzleNone = 0;

// Instruction descriptor of kind::mxf8f6f4: A = E2M1 (5), B = E4M3 (0), both
// K-major, M = m (128, or 256 for a CTA pair), N = n, E8M0 scales, scale-factor ids
// for A and B.
// idesc_mxf8f6f4(n, k) = idesc_mxf8f6f4(n, 0) + k * kIdescSfStep for k in 0..3
constexpr uint32_t kIdescSfStep = (1u << 4) | (1u << 29);

__device__ __forceinline__ uint32_t idesc_mxf8f6f4(int n, int sf_id, int m = kTileM) {
    uint32_t d = 0;
    d |= (uint32_t)(sf_id & 3) << 4;     // B scale factor id
    d |= 5u << 7;                        // A format: E2M1
    d |= 0u << 10;                       // B format: E4M3
    d |= (uint32_t)(n >> 3) << 17;       // N / 8
    d |= 1u << 23;                       // scale format: UE8M0
    d |= (uint32_t)(m >> 4) << 24;       // M / 16
    d |= (uint32_t)(sf_id & 3) << 29;    // A scale factor id
    return d;
}

__device__ __forceinline__ void tmem_alloc(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// Bulk copy global -> shared without a cache hint (16-byte aligned, size a
// multiple of 16), completion counted in bytes on `bar`.
__device__ __forceinline__ void bulk_g2s_l2(void *dst, const void *src, uint32_t bytes, uint64_t *bar) {
    asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(
                     smem_u32(dst)),
                 "l"(src), "r"(bytes), "r"(smem_u32(bar))
                 : "memory");
}

// True in one lane of the converged warp (the lowest active lane, lane 0 in the
// roles below, so a thread's tcgen05 operations and their commits stay together).
__device__ __forceinline__ bool elect_one() {
    uint32_t p;
    asm volatile("{\n\t.reg .pred e;\n\telect.sync _|e, 0xffffffff;\n\tselp.u32 %0, 1, 0, e;\n\t}" : "=r"(p));
    return p != 0;
}

// One 512-byte scale atom (32 rows x 16 bytes) into 4 TMEM columns of all four lane
// quadrants.  Each copy occupies the tensor pipe for about 100 clocks whatever its size
// (a 4 KB 128x256b copy costs the same), in order with the MMAs.
__device__ __forceinline__ void tc_cp_sf(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_mma(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa,
                                       uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// Instruction descriptor of kind::mxf4: A and B E2M1 (format 1 of this kind), both
// K-major, M = m (128, or 256 for a CTA pair), N = n, E8M0 scales.  With
// scale_vec::2X an MMA (K = 64) takes the scale bytes sf_id, sf_id + 1 (sf_id 0 or 2)
// of a 32-bit TMEM column: add kIdescSf2 for sf_id 2 (A and B alike).
constexpr uint32_t kIdescSf2 = (2u << 4) | (2u << 29);

__device__ __forceinline__ uint32_t idesc_mxf4(int n, int m = kTileM) {
    uint32_t d = 0;
    d |= 1u << 7;                        // A format: E2M1
    d |= 1u << 10;                       // B format: E2M1
    d |= (uint32_t)(n >> 3) << 17;       // N / 8
    d |= 1u << 23;                       // scale format: UE8M0
    d |= (uint32_t)(m >> 4) << 24;       // M / 16
    return d;
}

__device__ __forceinline__ void tc_mma_f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_commit(uint64_t *bar) {
    asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
                 : "memory");
}

// ---- CTA pairs (cta_group::2).  A cluster of two CTAs on two SMs: the even CTA issues
// MMAs of M = 256 whose A rows (128 per CTA) and B columns (N / 2 per CTA, the even CTA
// the first half) come from both CTAs' shared memory at the same offsets; each CTA's
// TMEM holds its own 128 accumulator rows, and the scale factors of its A rows and of
// all N columns of B.  Scale copies, MMAs and commits are issued by the even CTA and act
// on both; a commit arrives on the barrier at the same offset in both CTAs.
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}

// All threads of both CTAs (release / acquire at cluster scope).
__device__ __forceinline__ void cluster_sync() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address in the cluster's shared window of the object at the same offset in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void *p, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
    return r;
}

// `count` arrivals on a barrier of the other CTA (release at cluster scope).
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t cluster_addr, uint32_t count) {
    asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr), "r"(count)
                 : "memory");
}

// try_wait with acquire at cluster scope: for phases completed by the other CTA's arrivals.
__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// mbar_wait_or_abort for such phases.
__device__ __forceinline__ bool mbar_wait_cluster_or_abort(uint64_t *bar, uint32_t parity, StatusWord *st,
                                                           unsigned where, const int *abort_flag) {
    if (mbar_try_wait_cluster(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns(), lim = g_wait_limit_ns;
    for (uint32_t it = 0;; it++) {
        if (mbar_try_wait_cluster(bar, parity)) return true;
        if (*(const volatile int *)abort_flag) return false;
        if ((it & 63u) == 63u && global_timer_ns() - t0 > lim) {
            set_status(st, MOE_ERR_TIMEOUT, where);
            return false;
        }
    }
}

// TMEM of both CTAs: one warp of each CTA takes part.
__device__ __forceinline__ void tmem_alloc_pair(uint32_t *dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
                 "r"(ncols)
                 : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}

__device__ __forceinline__ void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}

__device__ __forceinline__ void tc_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
    asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

__device__ __forceinline__ void tc_mma_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                            uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

__device__ __forceinline__ void tc_mma_f4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t sfa, uint32_t sfb, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %6, 0;\n\t"
        "tcgen05.mma.cta_group::2.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
            d_tmem),
        "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
        : "memory");
}

// Commit of the pair's MMAs: arrives on `bar` in both CTAs.
__device__ __forceinline__ void tc_commit_pair(uint64_t *bar) {
    asm volatile(
        "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
            smem_u32(bar)),
        "h"((uint16_t)3)
        : "memory");
}

// 16 accumulator columns of this warp's 32 TMEM lanes; the wait is in the same
// statement, so no use of the registers can be scheduled before the data is there.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
    uint32_t r[16];
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, "
        "%15}, [%16];\n\t"
        "tcgen05.wait::ld.sync.aligned;"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
          "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
        : "r"(taddr)
        : "memory");
#pragma unroll
    for (int i = 0; i < 16; i++) v[i] = __uint_as_float(r[i]);
}

// ------------------------------------------------------------------- kernel

// MXFP8 shared exponent of a 32-block from the bits of its max |h| (a finite
// non-negative float): floor(log2 amax) - 8, or -127 for zero and values below
// 2^-119 (the clamp; subnormals have exponent field 0).  Equal to the frexp form.
__device__ __forceinline__ int mx_exp_from_bits(uint32_t amax_bits) { return max(-127, (int)(amax_bits >> 23) - 135); }

// MXFP4 shared exponent from the bits of the block's max |h|: floor(log2 amax) - 2,
// or -127 for zero and values below 2^-125.
__device__ __forceinline__ int mx4_exp_from_bits(uint32_t amax_bits) { return max(-127, (int)(amax_bits >> 23) - 129); }

// 2^-X as a float for X in [-127, 125] (always a normal number).
__device__ __forceinline__ float pow2_neg(int X) { return __uint_as_float((uint32_t)(127 - X) << 23); }

// Epilogue of the five-part MXFP4 activations (the multi-token decode on kind::mxf4):
// 16 pairs (80 accumulator columns) at a time, each pair's value the sum of its five
// columns in part order.  Gate/up: h = silu(g) * u, written as five MXFP4 parts per
// 32-block along I (the split of gather_split5_f4_kernel; lanes 2m and 2m+1 pack one
// byte); down: the unweighted expert output row in fp32.
__device__ __forceinline__ void epilogue_split5_f4(const GemmArgs &a, uint32_t lane_base, bool ok, int nn, int nmma,
                                                   int mt, int row0, int n0, int tile, int warp, int wg, int nwg,
                                                   int lane, float *amax_x) {
    constexpr int NP = 5;
    const int bar = 2 + 2 * wg + (warp >> 1);  // the warp pair's barrier
    for (int c0 = 16 * NP * wg; c0 < nmma; c0 += 16 * NP * nwg) {
        float v[NP][16];
#pragma unroll
        for (int q = 0; q < NP; q++)
#pragma unroll
            for (int j = 0; j < 16; j++) v[q][j] = 0.f;
        if (ok) {
#pragma unroll
            for (int q = 0; q < NP; q++) tmem_ld16(lane_base + (uint32_t)(c0 + 16 * q), v[q]);
        }
        float pv[16];
#pragma unroll
        for (int j = 0; j < 16; j++) {
            float acc = 0.f;
#pragma unroll
            for (int q = 0; q < NP; q++) {
                const int c = NP * j + q;  // column c of the group: register c % 16 of load c / 16
                acc = q == 0 ? v[c >> 4][c & 15] : acc + v[c >> 4][c & 15];
            }
            pv[j] = acc;
        }
        const int pair0 = (row0 + n0 + c0) / NP;
        const int npair = min(16, (nn - c0) / NP);  // pairs of this group with all their columns
        if (a.mode == 1) {
            // lanes 0-15: gate rows, 16-31: up rows of the same 16 intermediate indices
            const int i = (4 * mt + warp) * 16 + (lane & 15);
            float hv[16];
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const float u = __shfl_down_sync(0xffffffffu, pv[j], 16);
                hv[j] = (lane < 16) ? __fdividef(pv[j], 1.f + __expf(-pv[j])) * u : 0.f;
            }
#pragma unroll 1
            for (int q = 0; q < NP; q++) {
                // max |remainder| of each pair's 32-block along I (warps 2w and 2w+1)
                float am[16];
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    float m = fabsf(hv[j]);
#pragma unroll
                    for (int off = 8; off > 0; off >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, off));
                    am[j] = m;
                }
                if (lane == 0) {
#pragma unroll
                    for (int j = 0; j < 16; j++) amax_x[warp * 16 + j] = am[j];
                }
                named_barrier(bar, 64);
#pragma unroll
                for (int j = 0; j < 16; j++) {
                    const int X = mx4_exp(fmaxf(amax_x[warp * 16 + j], amax_x[(warp ^ 1) * 16 + j]));
                    const float hs = hv[j] * pow2_neg(X);
                    const float hn = __shfl_down_sync(0xffffffffu, hs, 1);
                    const uint8_t byte = e2m1x2_rn(hs, hn);  // this lane's code in the low nibble
                    hv[j] -= e2m1_nibble_value(byte) * __uint_as_float((uint32_t)(X + 127) << 23);
                    if (ok && j < npair && lane < 16 && (lane & 1) == 0) {
                        const uint64_t r = (uint64_t)NP * (pair0 + j) + q;
                        a.hq[r * (a.I / 2) + (i >> 1)] = byte;
                        if (lane == 0 && (warp & 1) == 0)
                            a.hs[sf_tile_word(tile, a.nkt_h, a.nsfb, i >> 7, c0 + NP * j + q) + ((i >> 5) & 3)] =
                                (uint8_t)(X + 127);
                    }
                }
                named_barrier(bar, 64);
            }
        } else {
            const int o = mt * kTileM + 32 * warp + lane;
#pragma unroll
            for (int j = 0; j < 16; j++)
                if (ok && j < npair && o < a.H)
                    reinterpret_cast<float *>(a.partial)[(uint64_t)(pair0 + j) * a.H + o] = pv[j];
        }
    }
}

// One-part (MXFP8) epilogue of a tile's 16-column groups: gate/up -> h = silu(g) * u
// quantised to MXFP8 along I (OCP rule); down -> expert output rows.  ew = warp
// index within the epilogue warpgroup (TMEM lanes 32ew..32ew+31); warpgroup wg of nwg
// takes the column groups c0 = 16 wg, 16 (wg + nwg), ...  Warps 2p and 2p+1 of a warpgroup
// hold the two halves of the same 32-blocks of I and exchange their maxima through
// shared memory under a 64-thread barrier of their own (id 2 + 2 wg + p).
template <bool FP4>
__device__ __forceinline__ void epilogue_mx1(const GemmArgs &a, uint32_t lane_base, bool ok, int nn, int nmma, int mt,
                                             int row0, int n0, int tile, int ew, int wg, int nwg, int lane,
                                             float *amax_x) {
    uint32_t *amax_u = reinterpret_cast<uint32_t *>(amax_x);
    const int bar = 2 + 2 * wg + (ew >> 1);  // the warp pair's barrier
    for (int c0 = 16 * wg; c0 < nmma; c0 += 16 * nwg) {
        float v[16];
#pragma unroll
        for (int j = 0; j < 16; j++) v[j] = 0.f;
        if (ok) tmem_ld16(lane_base + (uint32_t)c0, v);
        if (a.mode == 1) {
            // lanes 0-15: gate rows, 16-31: up rows of the same 16 intermediate indices
            const int i = (4 * mt + ew) * 16 + (lane & 15);
            float hv[16];
            uint32_t am[16];
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const float u = __shfl_down_sync(0xffffffffu, v[j], 16);
                const float g = v[j];
                // fast exp and divide: a few ulps, far inside the tolerance of h
                hv[j] = (lane < 16) ? __fdividef(g, 1.f + __expf(-g)) * u : 0.f;
                // the bits of non-negative floats order as their values
                am[j] = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(hv[j])));
            }
            if (lane == 0) {
#pragma unroll
                for (int j = 0; j < 16; j++) amax_u[ew * 16 + j] = am[j];
            }
            named_barrier(bar, 64);
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int n = c0 + j;
                const uint32_t amb = max(am[j], amax_u[(ew ^ 1) * 16 + j]);
                const int X = FP4 ? mx4_exp_from_bits(amb) : mx_exp_from_bits(amb);
                // h * 2^-X is exact (a power-of-two scaling that stays normal or rounds
                // as ldexp does)
                const float hsc = hv[j] * pow2_neg(X);
                if (FP4) {
                    // lanes 2m and 2m+1 hold intermediate indices i, i+1: one byte
                    const float hnext = __shfl_down_sync(0xffffffffu, hsc, 1);
                    if (ok && n < nn && lane < 16 && (lane & 1) == 0) {
                        const uint64_t r = (uint64_t)(row0 + n0 + n);
                        a.hq[r * (a.I / 2) + (i >> 1)] = e2m1x2_rn(hsc, hnext);
                        if (lane == 0 && (ew & 1) == 0)
                            a.hs[sf_tile_word(tile, a.nkt_h, a.nsfb, i >> 7, n) + ((i >> 5) & 3)] = (uint8_t)(X + 127);
                    }
                } else if (ok && n < nn && lane < 16) {
                    const uint64_t r = (uint64_t)(row0 + n0 + n);
                    unsigned short pair;
                    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(pair) : "f"(0.f), "f"(hsc));
                    a.hq[r * a.I + i] = (uint8_t)(pair & 0xFF);
                    if (lane == 0 && (ew & 1) == 0)
                        a.hs[sf_tile_word(tile, a.nkt_h, a.nsfb, i >> 7, n) + ((i >> 5) & 3)] = (uint8_t)(X + 127);
                }
            }
            named_barrier(bar, 64);
        } else {
            const int o = mt * kTileM + 32 * ew + lane;
#pragma unroll
            for (int j = 0; j < 16; j++) {
                const int n = c0 + j;
                if (ok && n < nn && o < a.H) {
                    const uint64_t r = (uint64_t)(row0 + n0 + n);
                    if (a.partial_dtype == MOE_PARTIAL_F32)
                        reinterpret_cast<float *>(a.partial)[r * a.H + o] = v[j];
                    else
                        reinterpret_cast<__nv_bfloat16 *>(a.partial)[r * a.H + o] = __float2bfloat16_rn(v[j]);
                }
            }
        }
    }
}

// Shared memory of the persistent kernel for BN accumulator columns and ns stages.
// With FP4 rows a stage holds the scale factors of two 128-K tiles (K = 256).
struct GemmSmemLayout {
    uint32_t a, b, sfa, sfb, bars, misc, total, sfa_stage, sfb_stage;
    __host__ __device__ GemmSmemLayout(int BN, int ns, int tpi, bool fp4, int bsr) {
        const uint32_t nsfb = (uint32_t)((BN + 127) / 128);
        sfa_stage = (uint32_t)tpi * (fp4 ? 1024u : 512u);
        sfb_stage = fp4 ? 2u * sfb_stage_bytes((int)nsfb) : sfb_stage_bytes((int)nsfb);
        a = 0;                                            // ns x tpi x 16 KB (1024-aligned)
        b = a + (uint32_t)(ns * tpi) * kTileM * kTileK;   // ns x bsr*128
        sfa = b + (uint32_t)ns * (uint32_t)bsr * kTileK;  // ns x sfa_stage
        sfb = sfa + (uint32_t)ns * sfa_stage;             // ns x sfb_stage
        bars = sfb + (uint32_t)ns * sfb_stage;            // full[], empty[], acc_full[2], acc_empty[2], mma_done
        misc = bars + (2 * kMaxStages + 5) * 8;           // tmem addr, abort, amax[4][16]
        total = misc + 16 + kEpiWarps * 16 * 4;
    }
};

// The work of a CTA: items i = blockIdx.x, +gridDim.x, ... of the n_union * nmt
// (expert of the union, 128-row tile of A) items; each item's columns in tiles of
// BN.  Every role walks this same sequence.
struct JobIter {
    const GemmArgs &a;
    int nu, i, nt, ntile, e, mt, row0, nrows, tile0;
    __device__ JobIter(const GemmArgs &args, int nu_) : a(args), nu(nu_), i((int)blockIdx.x), nt(0), ntile(0) { load(); }
    __device__ void load() {
        ntile = 0;
        const int nwi = (a.nmt + a.tpi - 1) / a.tpi;  // items per expert
        while (i < nu * nwi) {
            const int u = i / nwi;
            mt = (i % nwi) * a.tpi;  // first 128-row tile of the item
            e = a.uexp[u];
            row0 = a.nparts * a.offsets[e];
            nrows = a.nparts * (a.offsets[e + 1] - a.offsets[e]);
            ntile = (nrows + a.BN - 1) / a.BN;
            tile0 = a.tile_off[e];
            if (ntile > 0) break;
            i += (int)gridDim.x;
        }
        nt = 0;
    }
    __device__ bool valid() const { return i < nu * ((a.nmt + a.tpi - 1) / a.tpi) && ntile > 0; }
    __device__ int n0() const { return nt * a.BN; }
    __device__ int tile() const { return tile0 + nt; }
    // columns of the current tile (at most bsr: a tile with more is reported by the
    // sort as a bad index and computed only in part)
    __device__ int nn() const { return min(a.bsr, nrows - nt * a.BN); }
    __device__ void next() {
        if (++nt >= ntile) {
            i += (int)gridDim.x;
            load();
        }
    }
};

template <int NT, bool FP4>
__global__ void __launch_bounds__(NT, GemmShape<NT>::kCtasPerSm)
    grouped_gemm_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                        const GemmArgs a) {
    // launched early (programmatic dependent launch) on the multi-row decode path:
    // wait for the previous kernel, then let the next one launch
    griddep_wait();
    griddep_launch_dependents();
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the tensor copies with 128-byte swizzling need 1024-byte aligned tiles
    unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int ns = a.ns;
    const int tpi = a.tpi;
    const GemmSmemLayout L(a.BN, ns, tpi, FP4, a.bsr);
    uint8_t *sA = smem + L.a, *sB = smem + L.b, *sSFA = smem + L.sfa, *sSFB = smem + L.sfb;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + kMaxStages;
    uint64_t *acc_full = empty + kMaxStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.misc);
    int *abort_flag = reinterpret_cast<int *>(smem + L.misc + 4);
    float *amax_x = reinterpret_cast<float *>(smem + L.misc + 16);  // [8 epilogue warps][16 columns]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int nu = *a.n_union;
    if ((int)blockIdx.x >= nu * ((a.nmt + tpi - 1) / tpi)) return;  // the whole CTA, before any barrier
    const int nsfb = a.nsfb;

    // The unpacked E2M1 copies write 8 of every 16 bytes of an A tile; keep the
    // other 8 (which the MMA format pads with) zero for the whole kernel.  The
    // scale-factor areas start at zero too (the second tile of an item past the
    // expert's last row tile gets no copy and reads whatever is there).
    using Shape = GemmShape<NT>;
    for (int i = threadIdx.x; i < ns * tpi * kTileM * kTileK / 16; i += NT)
        reinterpret_cast<uint4 *>(sA)[i] = make_uint4(0u, 0u, 0u, 0u);
    for (int i = threadIdx.x; i < ns * (int)(L.sfa_stage + L.sfb_stage) / 16; i += NT)
        reinterpret_cast<uint4 *>(sSFA)[i] = make_uint4(0u, 0u, 0u, 0u);  // sSFB follows sSFA
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; s++) {
            mbar_init(&full[s], 1);   // producer's expect-tx arrival
            mbar_init(&empty[s], 1);  // MMA commit
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 1);   // MMA commit after a tile's last K step
            mbar_init(&acc_empty[b], Shape::kEpiWarps);  // the epilogue warps
        }
        mbar_init(mma_done, 1);  // the MMA warp's last commit
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc(tmem_slot, a.tmem_cols);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sf_col0 = (uint32_t)(a.nacc * tpi * a.BN);  // scale factors after the accumulators
    // TMEM columns per stage: 4 per 512-byte scale atom (two atoms per operand with FP4)
    const uint32_t sf_stage = FP4 ? 8u * (uint32_t)tpi + 8u * (uint32_t)nsfb : 4u * (uint32_t)tpi + 4u * (uint32_t)nsfb;

    int it_issued = 0;  // producer: stages issued
    // The copy and MMA roles run their loops with the whole warp converged (waits
    // polled by lane 0, or lanes 0-3 with a vote, and broadcast), so the addresses,
    // coordinates and descriptors are warp-uniform values; one elected lane issues
    // the asynchronous operations.
    if (warp == 0) {
        // ------------------------------------------------------- tensor copies
        int it = 0, s = 0;  // stages issued; slot of stage it
        uint32_t ph = 0;    // phase parity of slot s's use by stage it
        bool run = true;
        for (JobIter J(a, nu); run && J.valid(); J.next()) {
            for (int kt = 0; kt < a.nkt; kt++, it++) {
                int okl = 1;
                if (lane == 0) okl = mbar_wait_or_abort(&empty[s], ph ^ 1u, a.st, 0x500u + s, abort_flag);
                if (!__shfl_sync(0xffffffffu, okl, 0)) {
                    if (lane == 0) *abort_flag = 1;
                    run = false;
                    break;
                }
                // A arrives unpacked (16 E2M1 values in each 16 bytes, 8 of them data) and
                // counts its packed bytes; B counts one byte per element
                // B: one copy of BN rows (rows past this tile's nmma belong to other
                // experts or are out of range and zero; the MMA does not read them)
                // scale factors: the item's row tiles of A (adjacent in the plane) and
                // the column tile's atoms of B, each one contiguous block
                const uint32_t a_tiles = (uint32_t)min(tpi, a.nmt - J.mt);
                const int brow = J.row0 + J.n0();
                if (FP4) {
                    // packed operands, 256 K (128 bytes) per stage: both boxes arrive whole
                    // (parts past the end of K are zero-filled and counted); one or two
                    // 128-K scale tiles (the last stage of an odd count has one)
                    const int n2 = min(2, a.nkt_sf - 2 * kt);
                    const uint32_t sfbk = sfb_stage_bytes(nsfb);  // per 128-K tile
                    const int brows = a.bbox == a.BN ? a.BN : (J.nn() + 15) / 16 * 16;  // B rows copied
                    const uint32_t tx =
                        (uint32_t)(tpi * kTileM * kTileK + brows * kTileK) + (uint32_t)n2 * (512u + sfbk);
                    const uint8_t *sfa_src =
                        a.pool + (uint64_t)J.e * a.rec + a.a_sf_off + ((uint64_t)(2 * kt) * a.nmt + J.mt) * 512;
                    const uint8_t *sfb_src = a.bscale + sf_tile_word(J.tile(), a.nkt_sf, nsfb, 2 * kt, 0);
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&full[s], tx);
                        tma_load_3d(sA + (size_t)s * kTileM * kTileK, &tmA, kt * kTileK, J.mt * kTileM, J.e, &full[s]);
                        for (int c = 0; c < brows; c += a.bbox)
                            tma_load_2d(sB + (size_t)s * a.bsr * kTileK + (size_t)c * kTileK, &tmB, kt * kTileK,
                                        brow + c, &full[s]);
                        for (int j = 0; j < n2; j++)  // the two K tiles' A blocks are nmt blocks apart
                            bulk_g2s_l2(sSFA + (size_t)s * 1024 + 512 * j, sfa_src + (size_t)j * a.nmt * 512, 512u,
                                        &full[s]);
                        // the n2 K tiles' atoms (or interleaved 1 KB two-atom blocks) are adjacent
                        bulk_g2s_l2(sSFB + (size_t)s * 2 * sfbk, sfb_src, (uint32_t)n2 * sfbk, &full[s]);
                    }
                } else {
                    const int brows = a.bbox == a.BN ? a.BN : (J.nn() + 15) / 16 * 16;  // B rows copied
                    const uint32_t tx =
                        (uint32_t)(tpi * kTileM * kTileK / 2 + brows * kTileK) + a_tiles * 512u + sfb_stage_bytes(nsfb);
                    const uint8_t *sfa_src =
                        a.pool + (uint64_t)J.e * a.rec + a.a_sf_off + ((uint64_t)kt * a.nmt + J.mt) * 512;
                    const uint8_t *sfb_src = a.bscale + sf_tile_word(J.tile(), a.nkt, nsfb, kt, 0);
                    if (elect_one()) {
                        mbar_arrive_expect_tx(&full[s], tx);
                        tma_load_3d(sA + (size_t)s * tpi * kTileM * kTileK, &tmA, kt * kTileK, J.mt * kTileM, J.e,
                                    &full[s]);
                        for (int c = 0; c < brows; c += a.bbox)
                            tma_load_2d(sB + (size_t)s * a.bsr * kTileK + (size_t)c * kTileK, &tmB, kt * kTileK,
                                        brow + c, &full[s]);
                        bulk_g2s_l2(sSFA + (size_t)s * tpi * 512, sfa_src, a_tiles * 512u, &full[s]);
                        bulk_g2s_l2(sSFB + (size_t)s * sfb_stage_bytes(nsfb), sfb_src, sfb_stage_bytes(nsfb), &full[s]);
                    }
                }
                __syncwarp();
                it_issued = it + 1;
                if (++s == ns) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1) {
        // ------------------------------------------------------- MMA issue
        // The issue of a stage is a chain of dependent steps (wait, broadcast, scale
        // copies, MMAs, commit), so the warp first asks which of the next few stages
        // have landed (lane i polls stage kt + i, one vote) and issues all of those in
        // one go; the abort flag is read only while a stage is still outstanding.
        int jb = 0, s = 0;  // tiles; slot of the next stage
        uint32_t ph = 0;    // its phase parity
        bool run = true;
        // Descriptors of slot 0, built once: a stage's descriptors add the stage's
        // offset in 16-byte units to the start-address field (shared addresses stay
        // below 2^18, so the 14-bit field never carries into the next one).
        const uint32_t a_stage16 = (uint32_t)(tpi * kTileM * kTileK) >> 4, b_stage16 = (uint32_t)(a.bsr * kTileK) >> 4;
        const uint32_t sfa_stage16 = L.sfa_stage >> 4, sfb_stage16 = L.sfb_stage >> 4;
        const uint64_t adesc0 = smem_desc(smem_u32(sA), 16, 1024, kSwizzle128B);
        const uint64_t bdesc0 = smem_desc(smem_u32(sB), 16, 1024, kSwizzle128B);
        const uint64_t sfadesc0 = smem_desc(smem_u32(sSFA), 128, 128, kSwizzleNone);
        // core matrices of 8 rows x 16 bytes: an atom's row groups are 128 bytes apart, or
        // 256 in a two-atom block (the other atom's rows in between)
        const uint32_t sfb_rg = nsfb == 1 ? 128u : 256u;
        const uint64_t sfbdesc0 = smem_desc(smem_u32(sSFB), sfb_rg, sfb_rg, kSwizzleNone);
        const int nlook = min(4, ns);  // stages polled at once (never past the ring)
        for (JobIter J(a, nu); run && J.valid(); J.next(), jb++) {
            const int nmma = (J.nn() + 15) / 16 * 16;
            // mxf8f6f4: + ks * kIdescSfStep for K step ks; mxf4: + kIdescSf2 for odd ks
            const uint32_t idesc0 = FP4 ? idesc_mxf4(nmma) : idesc_mxf8f6f4(nmma, 0);
            // accumulator buffer of tile jb and its use count
            const int buf = a.nacc == 2 ? (jb & 1) : 0;
            const uint32_t use = a.nacc == 2 ? (uint32_t)(jb >> 1) : (uint32_t)jb;
            // the epilogue has finished with this accumulator (nacc tiles ago)
            int okl = 1;
            if (lane == 0) okl = mbar_wait_or_abort(&acc_empty[buf], (use & 1u) ^ 1u, a.st, 0x680u + buf,
                                                    abort_flag);
            if (!__shfl_sync(0xffffffffu, okl, 0)) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t acc = tmem + (uint32_t)(buf * tpi * a.BN);
            for (int kt = 0; kt < a.nkt;) {
                // stages kt .. kt + r - 1 have landed
                const int want = min(nlook, a.nkt - kt);
                bool rl = false;
                if (lane < want) {
                    const int q = s + lane;
                    rl = mbar_try_wait(&full[q % ns], ph ^ ((uint32_t)(q / ns) & 1u));
                }
                const uint32_t ready = __ballot_sync(0xffffffffu, rl);
                int r = min(__ffs(~ready) - 1, want);
                if (r == 0) {
                    okl = 1;
                    if (lane == 0) okl = mbar_wait_or_abort(&full[s], ph, a.st, 0x700u + s, abort_flag);
                    if (!__shfl_sync(0xffffffffu, okl, 0)) {
                        if (lane == 0) *abort_flag = 1;
                        run = false;
                        break;
                    }
                    r = 1;
                }
                tc_fence_after();
                if (elect_one()) {
                    int sq = s;
                    for (int q = 0; q < r; q++) {
                        const uint32_t sfa_t = tmem + sf_col0 + (uint32_t)sq * sf_stage;  // + 4t for tile t
                        const uint32_t sfb_t = sfa_t + 4u * (uint32_t)tpi;
                        const uint64_t sfad = sfadesc0 + (uint64_t)((uint32_t)sq * sfa_stage16);
                        const uint64_t sfbd = sfbdesc0 + (uint64_t)((uint32_t)sq * sfb_stage16);
                        const uint64_t ad0 = adesc0 + (uint64_t)((uint32_t)sq * a_stage16);
                        const uint64_t bd0 = bdesc0 + (uint64_t)((uint32_t)sq * b_stage16);
                        if constexpr (FP4) {
                            // two 128-K scale atoms per operand (one in the last stage of an
                            // odd count): K step ks (64 K) reads atom ks / 2, bytes 2 (ks % 2)..
                            // B: one atom (4 columns) or one two-atom block (8 columns) per K tile
                            const int n2 = min(2, a.nkt_sf - 2 * (kt + q));
                            const uint32_t sfb_t4 = sfa_t + 8u, bw = 4u * (uint32_t)nsfb;
                            for (int j = 0; j < n2; j++) {
                                tc_cp_sf(sfa_t + 4u * j, sfad + (uint64_t)(32 * j));
                                if (nsfb == 1) {
                                    tc_cp_sf(sfb_t4 + 4u * j, sfbd + (uint64_t)(32 * j));
                                } else {
                                    // the two atoms of the 1 KB block: rows 128 bytes apart in it
                                    tc_cp_sf(sfb_t4 + 8u * j, sfbd + (uint64_t)(64 * j));
                                    tc_cp_sf(sfb_t4 + 8u * j + 4u, sfbd + (uint64_t)(64 * j + 8));
                                }
                            }
                            for (int ks = 0; ks < 2 * n2; ks++)
                                tc_mma_f4(acc, ad0 + (uint64_t)(2 * ks), bd0 + (uint64_t)(2 * ks),
                                          idesc0 + ((ks & 1) ? kIdescSf2 : 0u), sfa_t + 4u * (ks >> 1),
                                          sfb_t4 + bw * (ks >> 1), (kt + q > 0 || ks > 0) ? 1u : 0u);
                        } else {
                            for (int t = 0; t < tpi; t++)
                                tc_cp_sf(sfa_t + 4u * t, sfad + (uint64_t)(32 * t));  // 512 B apart
                            tc_cp_sf(sfb_t, sfbd);
                            if (nsfb == 2) tc_cp_sf(sfb_t + 4u, sfbd + 8u);  // the block's second atom
                            for (int t = 0; t < tpi; t++) {
                                // tile t: rows 128t.. of the stage's A (16 KB apart), accumulator columns t*BN..
                                const uint64_t adt = ad0 + (uint64_t)(1024 * t);
#pragma unroll
                                for (int ks = 0; ks < kTileK / 32; ks++) {
                                    // K step ks: 32 bytes further along both operands' rows
                                    tc_mma(acc + (uint32_t)(t * a.BN), adt + (uint64_t)(2 * ks),
                                           bd0 + (uint64_t)(2 * ks), idesc0 + (uint32_t)ks * kIdescSfStep,
                                           sfa_t + 4u * t, sfb_t, (kt + q > 0 || ks > 0) ? 1u : 0u);
                                }
                            }
                        }
                        tc_commit(&empty[sq]);  // frees the stage when these MMAs have read it
                        if (++sq == ns) sq = 0;
                    }
                }
                __syncwarp();
                kt += r;
                s += r;
                if (s >= ns) {
                    s -= ns;
                    ph ^= 1u;
                }
            }
            if (elect_one()) tc_commit(&acc_full[buf]);  // the accumulator is complete (or as far as it got)
            __syncwarp();
        }
        // every MMA this warp issued has finished before TMEM can be released (also
        // after an abort, when the epilogue may not wait for the last accumulator)
        if (elect_one()) tc_commit(mma_done);
        __syncwarp();
        if (lane == 0) mbar_wait(mma_done, 0u, a.st, 0x6c0u);
        __syncwarp();
    } else if (warp >= Shape::kEpiFirst) {
        // ------------------------------------------------------- epilogue
        const int ew = warp & 3, wg = (warp - Shape::kEpiFirst) >> 2;
        float *amax_g = amax_x + 64 * wg;
        int jb = 0;
        for (JobIter J(a, nu); J.valid(); J.next(), jb++) {
            const int buf = a.nacc == 2 ? (jb & 1) : 0;
            const uint32_t use = a.nacc == 2 ? (uint32_t)(jb >> 1) : (uint32_t)jb;
            const int nn = J.nn(), nmma = (nn + 15) / 16 * 16;
            bool okl = !*(volatile int *)abort_flag && mbar_wait(&acc_full[buf], use & 1u, a.st, 0x800u + buf);
            if (!okl) *abort_flag = 1;
            const bool ok = __all_sync(0xffffffffu, okl);  // warp-uniform for the .sync.aligned loads
            tc_fence_after();
            for (int t = 0; t < tpi; t++) {
                if (J.mt + t >= a.nmt) break;  // a half item past the expert's A rows (uniform)
                const uint32_t lane_base =
                    tmem + (uint32_t)((buf * tpi + t) * a.BN) + ((uint32_t)(32 * ew) << 16);
                if (FP4 && a.nparts == 5)
                    epilogue_split5_f4(a, lane_base, ok, nn, nmma, J.mt + t, J.row0, J.n0(), J.tile(), ew, wg,
                                       Shape::kWarpGroups, lane, amax_g);
                else
                    epilogue_mx1<FP4>(a, lane_base, ok, nn, nmma, J.mt + t, J.row0, J.n0(), J.tile(), ew, wg,
                                      Shape::kWarpGroups, lane, amax_g);
            }
            tc_fence_before();
            __syncwarp();
            if (lane == 0) mbar_arrive(&acc_empty[buf]);
            // no early exit: after an abort the waits are skipped, and both warps of
            // each pair run the same sequence of named barriers to the end
        }
    }
    // nothing may still be in flight when TMEM is released and the CTA exits
    if (warp == 0 && lane == 0) {
        for (int it = max(0, it_issued - ns); it < it_issued; it++)
            mbar_wait(&full[it % ns], (uint32_t)(it / ns) & 1u, a.st, 0x900u);
    }
    __syncthreads();
    tc_fence_after();
    if (warp == 1) tmem_dealloc(tmem, a.tmem_cols);
}

// The work of a CTA pair: items i = pair, pair + pairs, ... of the (expert of the union,
// two 128-row tiles of A) items, one tile per CTA; each item's columns in tiles of BN.
// Both CTAs walk this same sequence with all their roles.
struct PairJobIter {
    const GemmArgs &a;
    int nu, i, nt, ntile, e, mt, row0, nrows, tile0;
    __device__ PairJobIter(const GemmArgs &args, int nu_) : a(args), nu(nu_), i((int)blockIdx.x / 2), nt(0), ntile(0) {
        load();
    }
    __device__ int items_per_expert() const { return (a.nmt + 1) / 2; }
    __device__ void load() {
        ntile = 0;
        const int nwi = items_per_expert();
        while (i < nu * nwi) {
            const int u = i / nwi;
            mt = (i % nwi) * 2;  // the even CTA's 128-row tile of the item
            e = a.uexp[u];
            row0 = a.offsets[e];
            nrows = a.offsets[e + 1] - a.offsets[e];
            ntile = (nrows + a.BN - 1) / a.BN;
            tile0 = a.tile_off[e];
            if (ntile > 0) break;
            i += (int)gridDim.x / 2;
        }
        nt = 0;
    }
    __device__ bool valid() const { return i < nu * items_per_expert() && ntile > 0; }
    __device__ int n0() const { return nt * a.BN; }
    __device__ int tile() const { return tile0 + nt; }
    __device__ int nn() const { return min(a.BN, nrows - nt * a.BN); }  // columns of the tile
    __device__ int nmma() const { return (nn() + 15) / 16 * 16; }       // MMA width
    __device__ void next() {
        if (++nt >= ntile) {
            i += (int)gridDim.x / 2;
            load();
        }
    }
};

// The grouped GEMM on CTA pairs (one-part rows, tiles of 128+ columns): clusters of two
// CTAs of 384 threads, one per SM, the same roles as grouped_gemm_kernel<384>.  The even
// CTA (rank 0) issues MMAs of M = 256 for both: A's rows 256 i.. (128 per CTA), B's
// columns split in halves (the even CTA the first nmma / 2).  Each CTA copies its own
// operands (its A tile, its half of B's rows, its A scale atoms and all of B's scale
// factors) with tensor copies whose completion counts on the even CTA's barrier, which
// expects the bytes of both; the even CTA's commits arrive in both CTAs; the odd CTA's
// epilogue reports a drained accumulator to the even CTA's barrier (one arrival per tile
// for all its epilogue warps).  Boxes past the end
// of a tensor (the odd CTA's A tile beyond the expert's last, the scales of the next K
// tile) arrive zero-filled and count whole.
template <bool FP4>
__global__ void __launch_bounds__(384, 1)
    grouped_gemm_pair_kernel(const __grid_constant__ CUtensorMap tmA, const __grid_constant__ CUtensorMap tmB,
                             const __grid_constant__ CUtensorMap tmSA, const __grid_constant__ CUtensorMap tmSB,
                             const GemmArgs a) {
    using Shape = GemmShape<384>;
    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the tensor copies with 128-byte swizzling need 1024-byte aligned tiles
    unsigned char *smem = (unsigned char *)(((uintptr_t)smem_raw + 1023) & ~(uintptr_t)1023);
    const int ns = a.ns;
    const GemmSmemLayout L(a.BN, ns, 1, FP4, a.bsr);
    uint8_t *sA = smem + L.a, *sB = smem + L.b, *sSFA = smem + L.sfa, *sSFB = smem + L.sfb;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + L.bars);
    uint64_t *empty = full + kMaxStages;
    uint64_t *acc_full = empty + kMaxStages;
    uint64_t *acc_empty = acc_full + 2;
    uint64_t *mma_done = acc_empty + 2;
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + L.misc);
    int *abort_flag = reinterpret_cast<int *>(smem + L.misc + 4);
    float *amax_x = reinterpret_cast<float *>(smem + L.misc + 16);  // [8 epilogue warps][16 columns]

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int rank = (int)cluster_ctarank();
    const int nu = *a.n_union;
    if ((int)blockIdx.x / 2 >= nu * ((a.nmt + 1) / 2)) return;  // both CTAs of the pair, before any barrier
    const int nsfb = a.nsfb;

    // the unpacked E2M1 copies (MXFP8 rows) write 8 of every 16 bytes of an A tile: keep
    // the other 8 zero
    for (int i = threadIdx.x; i < ns * kTileM * kTileK / 16; i += 384)
        reinterpret_cast<uint4 *>(sA)[i] = make_uint4(0u, 0u, 0u, 0u);
    fence_proxy_async_smem();
    if (threadIdx.x == 0) {
        for (int s = 0; s < ns; s++) {
            mbar_init(&full[s], 1);   // the even CTA's producer's expect-tx arrival
            mbar_init(&empty[s], 1);  // the even CTA's MMA commit
        }
        for (int b = 0; b < 2; b++) {
            mbar_init(&acc_full[b], 1);                        // MMA commit after a tile's last K step
            mbar_init(&acc_empty[b], 2 * Shape::kEpiWarps);  // the epilogue warps of both CTAs
        }
        mbar_init(mma_done, 1);  // the last commit
        *abort_flag = 0;
        fence_mbar_init();
    }
    if (warp == 1) tmem_alloc_pair(tmem_slot, a.tmem_cols);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // the other CTA's barriers exist before anything arrives on them
    tc_fence_after();
    const uint32_t tmem = *tmem_slot;
    const uint32_t sf_col0 = (uint32_t)(a.nacc * a.BN);  // scale factors after the accumulators
    // TMEM columns per stage: 4 per 512-byte scale atom (two atoms per operand with FP4)
    const uint32_t sf_stage = FP4 ? 8u + 8u * (uint32_t)nsfb : 4u + 4u * (uint32_t)nsfb;
    const uint32_t sfbk = sfb_stage_bytes(nsfb);  // B scale bytes per 128-K tile

    int it_issued = 0;  // producer: stages issued
    if (warp == 0) {
        // ------------------------------------------------------- tensor copies
        const uint32_t full_lead = mapa_shared(full, 0u);  // the even CTA's full[0]
        int it = 0, s = 0;  // stages issued; slot of stage it
        uint32_t ph = 0;    // phase parity of slot s's use by stage it
        bool run = true;
        for (PairJobIter J(a, nu); run && J.valid(); J.next()) {
            const int mta = J.mt + rank;                           // this CTA's A row tile
            const int brow = J.row0 + J.n0() + rank * (J.nmma() / 2);  // and its first B row
            for (int kt = 0; kt < a.nkt; kt++, it++) {
                int okl = 1;
                if (lane == 0) okl = mbar_wait_or_abort(&empty[s], ph ^ 1u, a.st, 0x500u + s, abort_flag);
                if (!__shfl_sync(0xffffffffu, okl, 0)) {
                    if (lane == 0) *abort_flag = 1;
                    run = false;
                    break;
                }
                // A: 128 rows (MXFP8 rows: unpacked by the copy, counted packed); B: this
                // CTA's half of the rows; A's scale atoms of the stage's 128-K tiles (nmt
                // atoms apart); one box of B's scale rows (both K tiles with FP4 rows)
                const int n2 = FP4 ? min(2, a.nkt_sf - 2 * kt) : 1;
                const int kt0 = FP4 ? 2 * kt : kt;  // first 128-K tile of the stage
                const uint32_t tx = (uint32_t)(FP4 ? kTileM * kTileK : kTileM * kTileK / 2) +
                                    (uint32_t)(a.bbox * kTileK) + (uint32_t)n2 * 512u + (FP4 ? 2u : 1u) * sfbk;
                const uint32_t fbar = full_lead + 8u * (uint32_t)s;
                if (elect_one()) {
                    if (rank == 0) mbar_arrive_expect_tx(&full[s], 2u * tx);  // both CTAs' bytes
                    tma_load_3d_pair(sA + (size_t)s * kTileM * kTileK, &tmA, kt * kTileK, mta * kTileM, J.e, fbar);
                    tma_load_2d_pair(sB + (size_t)s * a.bsr * kTileK, &tmB, kt * kTileK, brow, fbar);
                    for (int j = 0; j < n2; j++)
                        tma_load_3d_pair(sSFA + (size_t)s * L.sfa_stage + 512 * j, &tmSA, 0, (kt0 + j) * a.nmt + mta,
                                         J.e, fbar);
                    tma_load_2d_pair(sSFB + (size_t)s * L.sfb_stage, &tmSB, 0, J.tile() * a.nkt_sf + kt0, fbar);
                }
                __syncwarp();
                it_issued = it + 1;
                if (++s == ns) {
                    s = 0;
                    ph ^= 1u;
                }
            }
        }
    } else if (warp == 1 && rank == 0) {
        // ------------------------------------------------------- MMA issue (even CTA)
        // as in grouped_gemm_kernel: poll the next few stages at once and issue every
        // landed one; the scale copies, MMAs and commits act on both CTAs
        int jb = 0, s = 0;  // tiles; slot of the next stage
        uint32_t ph = 0;    // its phase parity
        bool run = true;
        const uint32_t a_stage16 = (uint32_t)(kTileM * kTileK) >> 4, b_stage16 = (uint32_t)(a.bsr * kTileK) >> 4;
        const uint32_t sfa_stage16 = L.sfa_stage >> 4, sfb_stage16 = L.sfb_stage >> 4;
        const uint64_t adesc0 = smem_desc(smem_u32(sA), 16, 1024, kSwizzle128B);
        const uint64_t bdesc0 = smem_desc(smem_u32(sB), 16, 1024, kSwizzle128B);
        const uint64_t sfadesc0 = smem_desc(smem_u32(sSFA), 128, 128, kSwizzleNone);
        const uint32_t sfb_rg = nsfb == 1 ? 128u : 256u;  // row groups of a B atom (256: two-atom block)
        const uint64_t sfbdesc0 = smem_desc(smem_u32(sSFB), sfb_rg, sfb_rg, kSwizzleNone);
        const int nlook = min(4, ns);
        for (PairJobIter J(a, nu); run && J.valid(); J.next(), jb++) {
            const int nmma = J.nmma();
            const uint32_t idesc0 = FP4 ? idesc_mxf4(nmma, 2 * kTileM) : idesc_mxf8f6f4(nmma, 0, 2 * kTileM);
            const int buf = a.nacc == 2 ? (jb & 1) : 0;
            const uint32_t use = a.nacc == 2 ? (uint32_t)(jb >> 1) : (uint32_t)jb;
            // both CTAs' epilogues have finished with this accumulator
            int okl = 1;
            if (lane == 0)
                okl = mbar_wait_cluster_or_abort(&acc_empty[buf], (use & 1u) ^ 1u, a.st, 0x680u + buf, abort_flag);
            if (!__shfl_sync(0xffffffffu, okl, 0)) {
                if (lane == 0) *abort_flag = 1;
                break;
            }
            tc_fence_after();
            const uint32_t acc = tmem + (uint32_t)(buf * a.BN);
            for (int kt = 0; kt < a.nkt;) {
                const int want = min(nlook, a.nkt - kt);
                bool rl = false;
                if (lane < want) {
                    const int q = s + lane;
                    rl = mbar_try_wait(&full[q % ns], ph ^ ((uint32_t)(q / ns) & 1u));
                }
                const uint32_t ready = __ballot_sync(0xffffffffu, rl);
                int r = min(__ffs(~ready) - 1, want);
                if (r == 0) {
                    okl = 1;
                    if (lane == 0) okl = mbar_wait_or_abort(&full[s], ph, a.st, 0x700u + s, abort_flag);
                    if (!__shfl_sync(0xffffffffu, okl, 0)) {
                        if (lane == 0) *abort_flag = 1;
                        run = false;
                        break;
                    }
                    r = 1;
                }
                tc_fence_after();
                if (elect_one()) {
                    int sq = s;
                    for (int q = 0; q < r; q++) {
                        const uint32_t sfa_t = tmem + sf_col0 + (uint32_t)sq * sf_stage;
                        const uint64_t sfad = sfadesc0 + (uint64_t)((uint32_t)sq * sfa_stage16);
                        const uint64_t sfbd = sfbdesc0 + (uint64_t)((uint32_t)sq * sfb_stage16);
                        const uint64_t ad0 = adesc0 + (uint64_t)((uint32_t)sq * a_stage16);
                        const uint64_t bd0 = bdesc0 + (uint64_t)((uint32_t)sq * b_stage16);
                        if constexpr (FP4) {
                            const int n2 = min(2, a.nkt_sf - 2 * (kt + q));
                            const uint32_t sfb_t4 = sfa_t + 8u, bw = 4u * (uint32_t)nsfb;
                            for (int j = 0; j < n2; j++) {
                                tc_cp_sf_pair(sfa_t + 4u * j, sfad + (uint64_t)(32 * j));
                                for (int b = 0; b < nsfb; b++)  // one atom, or the two of the 1 KB block
                                    tc_cp_sf_pair(sfb_t4 + bw * j + 4u * b,
                                                  sfbd + (uint64_t)(nsfb == 1 ? 32 * j : 64 * j + 8 * b));
                            }
                            for (int ks = 0; ks < 2 * n2; ks++)
                                tc_mma_f4_pair(acc, ad0 + (uint64_t)(2 * ks), bd0 + (uint64_t)(2 * ks),
                                               idesc0 + ((ks & 1) ? kIdescSf2 : 0u), sfa_t + 4u * (ks >> 1),
                                               sfb_t4 + bw * (ks >> 1), (kt + q > 0 || ks > 0) ? 1u : 0u);
                        } else {
                            const uint32_t sfb_t = sfa_t + 4u;
                            tc_cp_sf_pair(sfa_t, sfad);
                            for (int b = 0; b < nsfb; b++) tc_cp_sf_pair(sfb_t + 4u * b, sfbd + (uint64_t)(8 * b));
#pragma unroll
                            for (int ks = 0; ks < kTileK / 32; ks++)
                                tc_mma_pair(acc, ad0 + (uint64_t)(2 * ks), bd0 + (uint64_t)(2 * ks),
                                            idesc0 + (uint32_t)ks * kIdescSfStep, sfa_t, sfb_t,
                                            (kt + q > 0 || ks > 0) ? 1u : 0u);
                        }
                        tc_commit_pair(&empty[sq]);  // frees the stage in both CTAs
                        if (++sq == ns) sq = 0;
                    }
                }
                __syncwarp();
                kt += r;
                s += r;
                if (s >= ns) {
                    s -= ns;
                    ph ^= 1u;
                }
            }
            if (elect_one()) tc_commit_pair(&acc_full[buf]);  // the accumulator is complete (or as far as it got)
            __syncwarp();
        }
        // every MMA has finished before TMEM is released (in both CTAs)
        if (elect_one()) tc_commit_pair(mma_done);
        __syncwarp();
    } else if (warp >= Shape::kEpiFirst) {
        // ------------------------------------------------------- epilogue
        const int ew = warp & 3, wg = (warp - Shape::kEpiFirst) >> 2;
        float *amax_g = amax_x + 64 * wg;
        const uint32_t acc_empty_lead = mapa_shared(acc_empty, 0u);  // the even CTA's acc_empty[0]
        int jb = 0;
        for (PairJobIter J(a, nu); J.valid(); J.next(), jb++) {
            const int buf = a.nacc == 2 ? (jb & 1) : 0;
            const uint32_t use = a.nacc == 2 ? (uint32_t)(jb >> 1) : (uint32_t)jb;
            const int nn = J.nn(), nmma = J.nmma();
            bool okl = !*(volatile int *)abort_flag && mbar_wait(&acc_full[buf], use & 1u, a.st, 0x800u + buf);
            if (!okl) *abort_flag = 1;
            const bool ok = __all_sync(0xffffffffu, okl);  // warp-uniform for the .sync.aligned loads
            tc_fence_after();
            const int mt = J.mt + rank;  // this CTA's 128 rows of the tile
            if (mt < a.nmt) {            // (uniform) the odd CTA's tile may lie past the expert's rows
                const uint32_t lane_base = tmem + (uint32_t)(buf * a.BN) + ((uint32_t)(32 * ew) << 16);
                epilogue_mx1<FP4>(a, lane_base, ok, nn, nmma, mt, J.row0, J.n0(), J.tile(), ew, wg,
                                  Shape::kWarpGroups, lane, amax_g);
            }
            tc_fence_before();
            if (rank == 1) {
                // the odd CTA: its epilogue warps meet, and one arrival of all of them
                // (one cluster-scope release per tile, not one per warp)
                named_barrier(6, Shape::kEpiWarps * 32);
                if (warp == Shape::kEpiFirst && lane == 0)
                    mbar_arrive_cluster(acc_empty_lead + (uint32_t)(8 * buf), (uint32_t)Shape::kEpiWarps);
            } else {
                __syncwarp();
                if (lane == 0) mbar_arrive(&acc_empty[buf]);
            }
        }
    }
    // Nothing may still be in flight when TMEM is released and the CTA exits: the even
    // CTA waits for the last stages' copies (of both CTAs) and both wait for the last
    // commit (and with it every commit onto their stages) before the final cluster barrier.
    if (warp == 0 && lane == 0) {
        if (rank == 0)
            for (int it = max(0, it_issued - ns); it < it_issued; it++)
                mbar_wait(&full[it % ns], (uint32_t)(it / ns) & 1u, a.st, 0x900u);
        for (int it = max(0, it_issued - ns); it < it_issued; it++)
            mbar_wait(&empty[it % ns], (uint32_t)(it / ns) & 1u, a.st, 0x940u);
    }
    if (warp == 1 && lane == 0) mbar_wait(mma_done, 0u, a.st, 0x6c0u);
    tc_fence_before();
    __syncthreads();
    cluster_sync();  // both CTAs are done with TMEM and with each other's barriers
    tc_fence_after();
    if (warp == 1) tmem_dealloc_pair(tmem, a.tmem_cols);
}

// ------------------------------------------------------------- tensor maps

PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

cudaError_t get_encoder() {
    if (g_encode) return cudaSuccess;
    void *fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    cudaError_t e = cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q);
    if (e != cudaSuccess || q != cudaDriverEntryPointSuccess || fn == nullptr) return cudaErrorNotSupported;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
    return cudaSuccess;
}

// A: packed E2M1 weights of all experts, [E][rows][K] with the given strides,
// unpacked by the copy to 16 elements per 16 bytes (the f8f6f4 operand format).
cudaError_t make_map_a(CUtensorMap *m, const void *base, int K, int rows, int E, uint64_t row_stride,
                       uint64_t rec, int box_rows) {
    cuuint64_t dims[3] = {(cuuint64_t)K, (cuuint64_t)rows, (cuuint64_t)E};
    cuuint64_t strides[2] = {row_stride, rec};
    cuuint32_t box[3] = {kTileK, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B, 3, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// A with FP4 rows: the same weights as plain bytes (two E2M1 codes per byte, the
// packed operand format of kind::mxf4), K_bytes = K / 2 per row, boxes of 128 bytes.
cudaError_t make_map_a4(CUtensorMap *m, const void *base, int K_bytes, int rows, int E, uint64_t row_stride,
                        uint64_t rec, int box_rows) {
    cuuint64_t dims[3] = {(cuuint64_t)K_bytes, (cuuint64_t)rows, (cuuint64_t)E};
    cuuint64_t strides[2] = {row_stride, rec};
    cuuint32_t box[3] = {kTileK, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// B: activation rows [P][K] bytes (E4M3, one per element; or E2M1 pairs, K = row
// bytes), boxes of 128 bytes x box_rows rows.
cudaError_t make_map_b(CUtensorMap *m, const void *base, int K, int P, int box_rows) {
    cuuint64_t dims[2] = {(cuuint64_t)K, (cuuint64_t)P};
    cuuint64_t strides[1] = {(cuuint64_t)K};
    cuuint32_t box[2] = {kTileK, (cuuint32_t)box_rows};
    cuuint32_t es[2] = {1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

// Scale factors as 32-bit words for a pair's tensor copies.  A: the pool's tensor-core
// scale plane of each expert record, [E][rows][128 words] (rows = K tiles x row tiles,
// one 512-byte atom each); B: the tile-ordered activation scales, [rows][words] (rows
// = column tiles x K tiles, words = 128 per atom).  Boxes of box_rows whole rows.
cudaError_t make_map_sf(CUtensorMap *m, const void *base, int words, int rows, int E, uint64_t rec, int box_rows) {
    const int rank = E > 1 ? 3 : 2;
    cuuint64_t dims[3] = {(cuuint64_t)words, (cuuint64_t)rows, (cuuint64_t)(E > 1 ? E : 1)};
    cuuint64_t strides[2] = {(cuuint64_t)words * 4u, rec};
    cuuint32_t box[3] = {(cuuint32_t)words, (cuuint32_t)box_rows, 1};
    cuuint32_t es[3] = {1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_UINT32, rank, const_cast<void *>(base), dims, strides, box, es,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_NONE, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? cudaSuccess : cudaErrorInvalidValue;
}

uint32_t pow2_at_least(uint32_t v) {
    uint32_t p = 32;
    while (p < v) p <<= 1;
    return p;
}

PerDevice g_smem_max(0);
PerDevice g_sms(0);

PerDevice g_smem_set_384(0);
PerDevice g_smem_set_192(0);
PerDevice g_smem_set_384f4(0);
PerDevice g_smem_set_192f4(0);
PerDevice g_smem_set_pair(0);
PerDevice g_smem_set_pairf4(0);
std::atomic<int> g_cta_pairs{2};  // moe_grouped_set_cta_pairs: 0 never, 1 always, 2 MXFP8 rows only
PerDevice g_pair_clusters(0);    // co-resident CTA pairs of the paired kernel, MXFP8 rows (-1: none)
PerDevice g_pair_clusters_f4(0); // ... MXFP4 rows

// Launch configuration of the paired kernel: clusters of two CTAs of 384 threads.
inline cudaLaunchConfig_t pair_config(cudaLaunchAttribute *attr, int pairs, size_t smem, cudaStream_t stream) {
    cudaLaunchConfig_t cfg = {};
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 2;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.gridDim = dim3(2 * pairs);
    cfg.blockDim = dim3(384);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cfg;
}

// CTA pairs of the paired kernel that can be resident at once with `smem` bytes each
// (one CTA per SM at the sizes used), 0 if none; the persistent grid takes at most
// this many.  The kernel's dynamic shared-memory attribute must already allow `smem`.
template <bool FP4>
int pair_capacity(size_t smem) {
    int dev = 0;
    if (current_device(&dev) != cudaSuccess) return 0;
    PerDevice &cache = FP4 ? g_pair_clusters_f4 : g_pair_clusters;
    int pairs = cache.v[dev].load(std::memory_order_relaxed);
    if (pairs == 0) {
        int sms = 0;
        if (device_attr(cudaDevAttrMultiProcessorCount, g_sms, &sms) != cudaSuccess) return 0;
        cudaLaunchAttribute attr[1];
        const cudaLaunchConfig_t cfg = pair_config(attr, sms / 2, smem, nullptr);
        int n = 0;
        if (cudaOccupancyMaxActiveClusters(&n, grouped_gemm_pair_kernel<FP4>, &cfg) != cudaSuccess || n <= 0) {
            (void)cudaGetLastError();
            n = -1;
        }
        pairs = n;
        cache.v[dev].store(pairs, std::memory_order_relaxed);
    }
    return pairs > 0 ? pairs : 0;
}

template <bool FP4>
cudaError_t launch_pair(const CUtensorMap &mA, const CUtensorMap &mB, const CUtensorMap &mSA, const CUtensorMap &mSB,
                        const GemmArgs &ga, int pairs, size_t smem, cudaStream_t stream) {
    cudaLaunchAttribute attr[1];
    const cudaLaunchConfig_t cfg = pair_config(attr, pairs, smem, stream);
    return cudaLaunchKernelEx(&cfg, grouped_gemm_pair_kernel<FP4>, mA, mB, mSA, mSB, ga);
}

// One grouped GEMM launch (args complete but for the shape fields set here).  The
// kernel's shape: narrow tiles (BN <= 64, and the gate/up GEMM at BN <= 96) run two
// CTAs of 6 warps per SM with one 128-row tile per item and at most 256 TMEM columns
// each; wider tiles run one CTA of 12 warps per SM, with two 128-row tiles per item
// (one 256-row tensor copy) while their four accumulators fit in TMEM.  Measured on the
// full-size layer: two CTAs per SM took the 512-token GEMMs from 3.84 to 3.03 ms; the
// down GEMM at BN = 96 and all GEMMs at BN >= 128 are faster with one.  With FP4 rows
// every item is one 128-row tile and a stage covers two 128-K scale tiles: two A atoms
// (8 TMEM columns) and two B atoms or, for BN > 128, two interleaved two-atom blocks
// (16 columns).  (Two CTAs of one accumulator each per SM, tried for BN = 128, left
// only three stages per CTA and made the 32768-token GEMMs 1.34x slower.)  a_k and b_k
// are K in elements.
cudaError_t launch_one(GemmArgs ga, const uint8_t *a_base, int a_k, int a_rows, uint64_t a_ld, int E, const uint8_t *b_base,
                       int b_k, int b_rows, int nexp, int max_tiles, const char *trace_name, cudaStream_t stream,
                       bool fp4) {
    const int BN = ga.BN, nsfb = ga.nsfb;
    if (fp4 && nsfb > 2) return cudaErrorNotSupported;
    int smem_max = 0, sms = 0;
    cudaError_t e = device_attr(cudaDevAttrMaxSharedMemoryPerBlockOptin, g_smem_max, &smem_max);
    if (e != cudaSuccess) return e;
    if ((e = device_attr(cudaDevAttrMultiProcessorCount, g_sms, &sms)) != cudaSuccess) return e;
    // (FP4: the down GEMM too at BN <= 96, where its K loop is short: 7 stages at I = 1600)
    const bool two = BN <= 64 || (BN <= 96 && (ga.mode == 1 || fp4));
    const int tpi = fp4 || two ? 1 : (BN <= 96 ? 2 : 1);
    // wide one-part tiles run on CTA pairs (cta_group::2): each SM copies half of B
    if (ga.pair && (two || tpi != 1 || ga.nparts != 1 || BN < 128 || BN % 32 != 0)) ga.pair = 0;
    if (ga.pair) ga.bsr = BN / 2;
    const uint32_t smem_cap = two ? (uint32_t)(smem_max / 2 - 1024) : (uint32_t)smem_max;
    const uint32_t tmem_cap = two ? 256u : 512u;
    const uint32_t sf_cols = fp4 ? 8u * tpi + 8u * nsfb : 4u * tpi + 4u * nsfb;
    // two accumulators if they leave room for at least 4 stages of scale columns
    const int nacc = (uint32_t)(2 * tpi * BN) + 4u * sf_cols <= tmem_cap ? 2 : 1;
    // as many pipeline stages as fit the CTA's share of shared memory and TMEM
    int ns = kMaxStages;
    auto tmem_need = [&](int n) { return (uint32_t)(nacc * tpi * BN) + (uint32_t)n * sf_cols; };
    auto smem_need = [&](int n) { return GemmSmemLayout(BN, n, tpi, fp4, ga.bsr).total + 1024; };  // + alignment slack
    while (ns > 2 && (smem_need(ns) > smem_cap || tmem_need(ns) > tmem_cap)) ns--;
    const uint32_t tmem_cols = pow2_at_least(tmem_need(ns));
    if (tmem_cols > tmem_cap || smem_need(ns) > smem_cap) return cudaErrorNotSupported;
    const size_t smem = smem_need(ns);
    int pairs = 0;
    if (ga.pair) {
        e = fp4 ? ensure_dynamic_smem(grouped_gemm_pair_kernel<true>, smem, g_smem_set_pairf4)
                : ensure_dynamic_smem(grouped_gemm_pair_kernel<false>, smem, g_smem_set_pair);
        if (e != cudaSuccess) return e;
        pairs = fp4 ? pair_capacity<true>(smem) : pair_capacity<false>(smem);
        if (pairs == 0) {
            // no two SMs can hold a pair: the one-CTA tiles instead
            ga.pair = 0;
            ga.bsr = BN;
            return launch_one(ga, a_base, a_k, a_rows, a_ld, E, b_base, b_k, b_rows, nexp, max_tiles, trace_name, stream,
                              fp4);
        }
    } else if (fp4)
        e = two ? ensure_dynamic_smem(grouped_gemm_kernel<192, true>, smem, g_smem_set_192f4)
                : ensure_dynamic_smem(grouped_gemm_kernel<384, true>, smem, g_smem_set_384f4);
    else
        e = two ? ensure_dynamic_smem(grouped_gemm_kernel<192, false>, smem, g_smem_set_192)
                : ensure_dynamic_smem(grouped_gemm_kernel<384, false>, smem, g_smem_set_384);
    if (e != cudaSuccess) return e;
    ga.ns = ns;
    ga.tpi = tpi;
    ga.nacc = nacc;
    // narrow tiles copy B in 16-row boxes, only the rows the tile's MMAs read: verify
    // tiles (several parts per row) hold a few rows in a box sized for 32, and prefill
    // tiles up to 64 columns are sized for the expert rows' spread
    ga.bbox = ga.pair ? BN / 2 : ((ga.nparts > 1 || BN <= 64) ? 16 : BN);
    if (!ga.pair && ga.bsr != BN && ga.bbox != 16) return cudaErrorInvalidValue;
    ga.tmem_cols = tmem_cols;
    ga.nkt_sf = a_k / kTileK;
    ga.nkt = fp4 ? (ga.nkt_sf + 1) / 2 : ga.nkt_sf;
    CUtensorMap mA, mB, mSA = {}, mSB = {};
    if (ga.pair) {
        // the scales as tensors: A's plane in each record, B's tile-ordered blocks
        if ((e = make_map_sf(&mSA, ga.pool + ga.a_sf_off, 128, ga.nkt_sf * ga.nmt, E, ga.rec, 1)) != cudaSuccess)
            return e;
        if ((e = make_map_sf(&mSB, ga.bscale, 128 * nsfb, max_tiles * ga.nkt_sf, 1, 0, fp4 ? 2 : 1)) != cudaSuccess)
            return e;
    }
    if (fp4) {
        if ((e = make_map_a4(&mA, a_base, a_k / 2, a_rows, E, a_ld, ga.rec, kTileM)) != cudaSuccess) return e;
        if ((e = make_map_b(&mB, b_base, b_k / 2, b_rows, ga.bbox)) != cudaSuccess) return e;
    } else {
        if ((e = make_map_a(&mA, a_base, a_k, a_rows, E, a_ld, ga.rec, tpi * kTileM)) != cudaSuccess) return e;
        if ((e = make_map_b(&mB, b_base, b_k, b_rows, ga.bbox)) != cudaSuccess) return e;
    }
    const int items = nexp * ((ga.nmt + (ga.pair ? 2 : tpi) - 1) / (ga.pair ? 2 : tpi));
    TraceScope trace_scope(trace_name, stream);
    if (ga.pair) {
        pairs = std::min(pairs, items);
        e = fp4 ? launch_pair<true>(mA, mB, mSA, mSB, ga, pairs, smem, stream)
                : launch_pair<false>(mA, mB, mSA, mSB, ga, pairs, smem, stream);
        if (e != cudaSuccess) return e;
    } else if (fp4) {
        // (the multi-token decode's chain of kernels launches each one early)
        if (two && ga.nparts > 1)
            e = launch_pdl(grouped_gemm_kernel<192, true>, dim3(std::min(2 * sms, items)), dim3(192), smem, stream,
                           mA, mB, ga);
        else if (two)
            grouped_gemm_kernel<192, true><<<std::min(2 * sms, items), 192, smem, stream>>>(mA, mB, ga);
        else if (ga.nparts > 1)
            e = launch_pdl(grouped_gemm_kernel<384, true>, dim3(std::min(sms, items)), dim3(384), smem, stream, mA,
                           mB, ga);
        else
            grouped_gemm_kernel<384, true><<<std::min(sms, items), 384, smem, stream>>>(mA, mB, ga);
        if (e != cudaSuccess) return e;
    } else {
        if (two)
            grouped_gemm_kernel<192, false><<<std::min(2 * sms, items), 192, smem, stream>>>(mA, mB, ga);
        else
            grouped_gemm_kernel<384, false><<<std::min(sms, items), 384, smem, stream>>>(mA, mB, ga);
    }
    return cudaGetLastError();
}

}  // namespace

cudaError_t set_wait_limit_gemm(uint64_t ns) { return set_wait_limit_here(ns); }

void set_cta_pairs(int mode) { g_cta_pairs.store(mode, std::memory_order_relaxed); }

cudaError_t launch_grouped_gemms(const PoolView &v, int T, int k, const int32_t *offsets, const GroupedWs &g,
                                 void *partial, int partial_dtype, StatusWord *st, cudaStream_t stream, int nparts,
                                 bool fp4, int max_cols) {
    const int P = T * k;
    if (P == 0) return cudaSuccess;
    // one MXFP8 or MXFP4 row per pair, or five MXFP4 parts (mxf4)
    if (!(nparts == 1 || (nparts == 5 && fp4))) return cudaErrorInvalidValue;
    cudaError_t e = get_encoder();
    if (e != cudaSuccess) return e;
    // the sort laid out the activation scales for this BN
    const int BN = grouped_bn(P, v.E, T, nparts, fp4);
    if (BN == 0) return cudaErrorNotSupported;
    if (BN != g.BN) return cudaErrorInvalidValue;
    const int nsfb = g.nsfb;
    GemmArgs ga;
    ga.E = v.E;
    ga.pool = v.base;
    ga.rec = v.rec;
    ga.offsets = offsets;
    ga.tile_off = g.tile_off;
    ga.uexp = g.uexp;
    ga.n_union = g.n_union;
    ga.BN = BN;
    ga.nsfb = nsfb;
    ga.I = v.I;
    ga.H = v.H;
    ga.hq = g.hq;
    ga.hs = g.hs;
    ga.nkt_h = v.Ip / kTileK;
    ga.partial = partial;
    ga.partial_dtype = partial_dtype;
    ga.nparts = nparts;
    // CTA pairs where they measured faster (MXFP8 rows), or as set; launch_one decides per
    // GEMM whether the tile shape allows them
    const int pairs_mode = g_cta_pairs.load(std::memory_order_relaxed);
    ga.pair = pairs_mode == 1 || (pairs_mode == 2 && !fp4) ? 1 : 0;
    ga.st = st;
    // B rows a stage reserves: all BN, or (five-part rows, known bound) just the columns
    // any tile has, rounded to the 16-row boxes: more pipeline stages fit
    ga.bsr = (nparts > 1 && max_cols > 0 && max_cols < BN) ? (max_cols + 15) / 16 * 16 : BN;
    const int nexp = P < v.E ? P : v.E;  // at most this many experts have pairs

    // GEMM 1: gate/up
    ga.mode = 1;
    ga.a_sf_off = v.off_sgu_mma;
    ga.bscale = g.xs;
    ga.nmt = v.nmt_gu;
    e = launch_one(ga, v.base, v.H, 2 * v.I, (uint64_t)v.ld_gu, v.E, g.xq, v.H, nparts * P, nexp, g.max_tiles,
                   "gemm_gateup", stream, fp4);
    if (e != cudaSuccess) return e;

    // GEMM 2: down (K = Ip, the W_d rows padded with zero codes; h has I columns, the
    // rest of its last box is zero-filled)
    ga.mode = 2;
    ga.a_sf_off = v.off_sd_mma;
    ga.bscale = g.hs;
    ga.nmt = v.nmt_d;
    return launch_one(ga, v.base + v.off_d, v.Ip, v.H, (uint64_t)v.ld_d, v.E, g.hq, v.I, nparts * P, nexp, g.max_tiles,
                      "gemm_down", stream, fp4);
}

}  // namespace moe
