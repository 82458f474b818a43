/*
 * moe.h -- C ABI of the GB300 (sm_103a) routed-expert MXFP4 MoE layer.
 *
 * The layer follows the Deltafin pages' problem statement: a token's hidden state
 * goes in, the router picks 16 routed experts per layer ("Deltafin：在Apple Silicon
 * Mac上运行Kimi K3", section 工作原理), the experts come from a resident pool of
 * per-(layer, expert) MXFP4 records ("Deltafin 在配备四个 SSD 的 MacBook Pro 上…",
 * section Deltafin 的功能), several rows can be verified in one pass (same page,
 * section 可选的 Qwen 扩展) and prefill reads each expert once for all its rows
 * (same page, section 作者仍需帮助的事项).  The layer math, which the pages do not
 * spell out, is: router logits l = W_r x (+ skew), top-k by l with ties to the
 * lower expert index, softmax over the k selected logits, per expert
 * h = silu(W_g x) * (W_u x), o = W_d h, and y = sum_j w_j o_j (+ residual).
 *
 * Conventions (all entry points):
 *  - Every pointer argument named *_dev, and every tensor argument unless stated
 *    otherwise, is a DEVICE pointer owned by the caller.  The library never
 *    allocates device memory, and keeps no reference after the call returns
 *    (except the pool view, which refers to caller memory until destroyed).
 *  - bf16 tensors are passed as uint16_t bit patterns.  Matrices are row-major
 *    with the hidden dimension contiguous.
 *  - `stream` is a cudaStream_t.  Calls are asynchronous on that stream; the
 *    return value reports host-side validation and launch errors only.
 *  - Errors the GPU detects (an expert index out of range, a non-finite router
 *    logit, a bounded device wait that expired) are recorded in a status word at
 *    the start of the workspace `ws` and returned by moe_check_status().  Kernels
 *    never trap; a bad expert index makes its (token, slot) pair contribute zero.
 *  - Supported shapes: 1 <= k <= 32, k <= E <= 65536, H a multiple of 128,
 *    I a multiple of 32 (decode) or of 64 (prefill), H, I <= 32768.
 */
#ifndef MOE_H
#define MOE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    MOE_OK = 0,
    MOE_ERR_INVALID_ARG = 1,       /* null pointer, negative size, k > E, ... */
    MOE_ERR_UNSUPPORTED_SHAPE = 2, /* shape outside the supported set above */
    MOE_ERR_WORKSPACE = 3,         /* ws smaller than moe_workspace_size() */
    MOE_ERR_CUDA = 4,              /* a CUDA runtime call or launch failed */
    MOE_ERR_BAD_INDEX = 5,         /* device: an expert index outside [0, E), or named too
                                      often in one multi-row decode call */
    MOE_ERR_TIMEOUT = 6,           /* device: a bounded wait gave up */
    MOE_ERR_NONFINITE = 7          /* device: non-finite router input or logit */
} moe_status;

typedef void *moe_stream_t;        /* a cudaStream_t */
typedef struct moe_pool moe_pool;  /* host-side view of a resident expert pool */

/* Operation codes for moe_workspace_size(). */
enum { MOE_OP_ROUTE = 0, MOE_OP_DECODE = 1, MOE_OP_GROUPED = 2 };

/* Activation formats of the expert-major (grouped) path. */
enum { MOE_ACT_MXFP8 = 1, MOE_ACT_MXFP4 = 2 };

/* Element types of the grouped path's partial outputs. */
enum { MOE_PARTIAL_F32 = 0, MOE_PARTIAL_BF16 = 1 };

/* ------------------------------------------------------------ expert pool
 * One record per expert (the pages' per-(layer, expert) MXFP4 file, 17.5 MiB at
 * the full shape), resident in device memory the caller allocates.  A record
 * holds W_gu = the gate and up rows interleaved in groups of 16 (rows 32q..32q+15
 * are gate rows 16q..16q+15, rows 32q+16..32q+31 the matching up rows), shape
 * [2I][H], and W_d [H][I], as packed E2M1 codes (two per byte, element 2j in
 * the low nibble, K contiguous) followed by their E8M0 scale bytes (one per 32
 * consecutive K elements, row-major).  Rows of W_d are padded with zero codes and
 * zero scale bytes to a multiple of 128 elements.  The record ends with the same
 * scale bytes once more, reordered for the tensor-core path (for each K tile of 128
 * elements and 128-row tile, one 512-byte block: row 128mt + 32q + l keeps the
 * tile's 4 scale bytes at 16l + 4q); the pool functions write both copies. */

/* Bytes one pool of E experts needs (a multiple of 1024 per record); 0 when the
 * shape is unsupported. */
size_t moe_pool_bytes(int E, int H, int I);

/* Bytes of one expert record. */
size_t moe_pool_record_bytes(int H, int I);

/* Create a view of a pool over caller memory `dev_mem` of `bytes` bytes (at
 * least moe_pool_bytes(E,H,I), 1024-byte aligned).  Contents are undefined until
 * filled.  *out receives a host object freed by moe_pool_destroy(). */
moe_status moe_pool_create(moe_pool **out, void *dev_mem, size_t bytes, int E, int H, int I);
void moe_pool_destroy(moe_pool *pool);

/* Fill experts [e_lo, e_hi) with synthetic data drawn on the device from the
 * counter-based SplitMix64 definition (codes of expert e: byte b is byte b%8 of
 * u64(seed, 2e, b/8) in the logical row-major order gate, up, down; scale byte j
 * is 118 + (u64(seed, 2e+1, j) >> 32) % 5, i.e. exponents -9..-5), where
 * u64(seed, s, i) = mix(key + (i+1) G), key = mix(mix(seed + G) ^ mix(s + 2G)),
 * G = 0x9E3779B97F4A7C15, mix = the SplitMix64 finaliser. */
moe_status moe_pool_fill_synthetic(moe_pool *pool, uint64_t seed, int e_lo, int e_hi,
                                   moe_stream_t stream);

/* Pack expert e from its logical row-major form (device buffers):
 * codes_dev [3*H*I/2] = gate [I][H/2] | up [I][H/2] | down [H][I/2],
 * scales_dev [3*H*I/32] = gate [I][H/32] | up [I][H/32] | down [H][I/32]. */
moe_status moe_pool_upload_expert(moe_pool *pool, int e, const uint8_t *codes_dev,
                                  const uint8_t *scales_dev, moe_stream_t stream);

/* Inverse of moe_pool_upload_expert (for inspection and tests). */
moe_status moe_pool_download_expert(const moe_pool *pool, int e, uint8_t *codes_dev,
                                    uint8_t *scales_dev, moe_stream_t stream);

/* ------------------------------------------------------ streamed expert pool
 * The pages' streamed experts ("技术亮点" on the hn page: experts read on demand,
 * with a cache; "存储子系统" on the four-SSD page: demand reads of one unit per
 * (layer, expert)) in GB300 form.  The E records of a layer (the pool record layout
 * above) live in caller-owned host memory, pinned so that the copy engines read
 * them over NVLink-C2C; a cache of C = cache_bytes / moe_pool_record_bytes(H, I)
 * record slots lives in caller-owned device memory.  The cache is an ordinary pool
 * view of C records (moe_stream_pool_cache), so moe_expert_forward_decode and
 * moe_expert_forward_grouped run on it with slot indices in place of expert indices.
 *
 * moe_stream_pool_create: host_records >= E records (host_bytes), dev_cache
 * 1024-byte aligned with room for C >= 1 records (C <= E).  dev_cache may be NULL:
 * the object then only plans (assigns slots, counts hits and misses) and copies
 * nothing, which tests the replacement policy without a GPU. */
typedef struct moe_stream_pool moe_stream_pool;
moe_status moe_stream_pool_create(moe_stream_pool **out, const void *host_records, size_t host_bytes, int E, int H,
                                  int I, void *dev_cache, size_t cache_bytes);
void moe_stream_pool_destroy(moe_stream_pool *sp);

/* The cache as a pool of C records (slot s is "expert" s); NULL when planning only. */
const moe_pool *moe_stream_pool_cache(const moe_stream_pool *sp);
int moe_stream_pool_slots(const moe_stream_pool *sp);

/* Make the experts idx_host[0..n) (host memory; n = M*k of a decode or grouped call)
 * resident and write their slots to slot_host[0..n) (host memory; copy them to the
 * device for the kernels).  A missing expert takes the least recently used slot that
 * this call does not use, and its record is copied with one cudaMemcpyAsync
 * (host -> device) on `stream`: after every earlier use of the slot on that stream
 * and before every later one, so all work that uses the cache must be issued on
 * `stream` (or ordered with it).  An index outside [0, E) gets slot -1 (the kernels
 * report MOE_ERR_BAD_INDEX and add nothing for it).  MOE_ERR_UNSUPPORTED_SHAPE if the
 * call names more distinct experts than C.  Not thread-safe per object. */
moe_status moe_stream_pool_map(moe_stream_pool *sp, const int32_t *idx_host, int n, int32_t *slot_host,
                               moe_stream_t stream);

/* Counters since creation: distinct experts per call found resident (hits) and
 * copied (misses), and the bytes copied. */
moe_status moe_stream_pool_stats(const moe_stream_pool *sp, uint64_t *hits, uint64_t *misses, uint64_t *bytes);

/* Pinned host memory for the records, placed on the host NUMA node closest to GPU
 * `device` (cudaDevAttrHostNumaId).  On a Grace host each CPU die is a NUMA node and
 * the GPU's copy engines read their own die's memory over NVLink-C2C, the other
 * die's only through the CPU-to-CPU link, several times slower; ordinary pinned
 * memory lands on the node of whichever CPU the allocating thread runs on.
 * *out: page-aligned, `bytes` rounded up to whole pages, readable and writable by
 * the host and registered with CUDA (cudaHostRegister).  *numa_node (may be NULL):
 * the node the first page actually lies on, -1 if unknown (placement is a
 * preference: a full node falls back to another).  MOE_ERR_CUDA if the registration
 * fails; free with moe_host_free(p, bytes) using the same `bytes`. */
moe_status moe_host_alloc(int device, size_t bytes, void **out, int *numa_node);
moe_status moe_host_free(void *p, size_t bytes);

/* The host NUMA node closest to GPU `device`, or -1 (no NUMA, or unknown). */
int moe_host_numa_node(int device);

/* ------------------------------------------------------------- workspace */

/* Workspace bytes of operation `op` (MOE_OP_*) for M (decode) or T (prefill)
 * rows.  The workspace is caller-owned device memory, 256-byte aligned; its
 * first 256 bytes hold the device status word and the kernels' own counters.
 * They must be zero before the first call on a workspace (moe_clear_status, or a
 * zero-filled allocation); the kernels leave them zero again after each call
 * that succeeds.  After a call that recorded a device error (a bounded wait that
 * expired, for instance) moe_check_status or moe_clear_status resets them. */
moe_status moe_workspace_size(int op, int E, int H, int I, int rows, int k, size_t *bytes);

/* Clear the status word of `ws` (asynchronously, on `stream`). */
moe_status moe_clear_status(void *ws, moe_stream_t stream);

/* Synchronise `stream`, return the first device-detected error recorded in
 * `ws` since it was last cleared (MOE_OK if none), and clear it. */
moe_status moe_check_status(void *ws, moe_stream_t stream);

const char *moe_status_string(moe_status s);

/* ---------------------------------------------------------------- routing
 * Router top-k with softmax ("工作原理": 16 experts per layer per token).
 * x [M][H] bf16, Wr [E][H] bf16, skew [E] fp32 or NULL (added to the logits).
 * Out: idx [M][k] int32, the k experts of largest exact logit
 * sum_h x_h Wr[e,h] (+ skew_e) in descending order, ties to the lower index;
 * w [M][k] fp32 = softmax over those k logits.  The selection is exact: fp32
 * logits carry a rigorous error bound and any order the bound cannot decide is
 * settled with exact integer arithmetic.  ws: MOE_OP_ROUTE bytes; after the call
 * it holds, for diagnostics, the status word (256 B), then the fp32 logits
 * [M][E] and then their error bounds [M][E], each region starting on a 256-byte
 * boundary (|logit - exact logit| <= bound). */
moe_status moe_route_topk(const uint16_t *x, int M, int H, const uint16_t *Wr, int E,
                          const float *skew, int k, int32_t *idx, float *w,
                          void *ws, size_t ws_bytes, moe_stream_t stream);

/* Router variant that allocates nothing and takes no workspace.  The pages have
 * no counterpart to this entry point; it exists for callers that cannot call
 * cudaMalloc or hand over a workspace -- code running while a caching allocator
 * or a host framework owns all device memory, plugins whose host provides no
 * scratch buffers, and latency-critical threads that must not risk the
 * device-wide synchronisation cudaMalloc/cudaFree can cause.
 * Same arguments, kernels and results as moe_route_topk, but the scratch (status
 * word, fp32 logits and their bounds, the row norms of the many-token logit
 * kernel) lives in one static device array of the library, about 1.5 MiB, that
 * every GPU which loads the library keeps until the process exits.  Limit: M * E <= 131072 (else MOE_ERR_UNSUPPORTED_SHAPE).
 * The first call on a device looks up the array's device address (with that
 * device current), so make that first call before any stream capture; host threads
 * that make their first calls at the same time look it up alike (the per-device
 * entries are atomic).  All calls share the array: calls that overlap on the GPU
 * (other streams, other threads) race and must be serialised by the caller.  The status word is cleared at the
 * start of every call; device-detected errors are recorded there but not
 * returned -- use moe_route_topk with a workspace to read them. */
moe_status moe_route_topk_static(const uint16_t *x, int M, int H, const uint16_t *Wr, int E,
                                 const float *skew, int k, int32_t *idx, float *w,
                                 moe_stream_t stream);

/* Pre-scaled routing for stacked layers: x_hat = moe_prescale(x) is written to
 * xhat [M][H] bf16 (16-byte aligned) and the rows are routed as moe_route_topk
 * routes x_hat (same idx, w and status).  For M = 1 the pre-scale is folded into
 * the router's own staging of the token (one launch); for M > 1 it runs first.
 * ws: MOE_OP_ROUTE bytes. */
moe_status moe_route_topk_prescaled(const uint16_t *x, int M, int H, const uint16_t *Wr, int E,
                                    const float *skew, int k, int32_t *idx, float *w, uint16_t *xhat,
                                    void *ws, size_t ws_bytes, moe_stream_t stream);

/* ------------------------------------------------------- decode / verify
 * Expert forward for M (1..32) rows that were routed by moe_route_topk: each
 * distinct selected expert is read from the pool once and applied to every row
 * routed to it (the pages' speculative-verify batch, "可选的 Qwen 扩展").
 * x [M][H] bf16, idx/w [M][k] as from moe_route_topk, residual [M][H] bf16 or
 * NULL.  Out: y [M][H] bf16 = sum_j w[m,j] * expert_{idx[m,j]}(x[m]) (+ residual),
 * fp32 accumulation, rounded to nearest-even.  ws: MOE_OP_DECODE bytes.
 * M = 1 runs on the CUDA cores (E2M1 -> f16 dequantisation, f16 products summed
 * per 32-element block, then fp32).  M > 1 runs on the tensor cores when I is a
 * multiple of 64: each 32-element block of a row is written as the sum of five
 * MXFP4 parts (each the OCP rule applied to what the earlier parts left; the
 * block's largest remainder shrinks at least threefold per part), multiplied with
 * the E2M1 weights in kind::mxf4 block-scaled MMAs with fp32 accumulation; h is
 * split the same way for W_d.  What the five parts leave out is below 3^-5 of each
 * block's max |value| (about 3e-4 of RMS on the outputs of full-size layers).
 * On that path the k indices of each row should be distinct (moe_route_topk gives
 * them so): for M <= 15 the GEMM stages reserve room for ceil16(5 M) activation
 * rows per expert, and an expert named more than ceil16(5 M) / 5 times in all is
 * reported as MOE_ERR_BAD_INDEX (y is then not valid).  A row may repeat an index
 * as long as no expert exceeds that count. */
moe_status moe_expert_forward_decode(const moe_pool *pool, const uint16_t *x, int M,
                                     const int32_t *idx, const float *w, int k,
                                     const uint16_t *residual, uint16_t *y,
                                     void *ws, size_t ws_bytes, moe_stream_t stream);

/* Exact power-of-two pre-scale of layer inputs (stacked layers): for each row,
 * out = x * 2^-p with p = floor(log2(max|x|)) - 2, so max|out| lies in [4, 8);
 * an all-zero row is copied.  x, out [M][H] bf16. */
moe_status moe_prescale(const uint16_t *x, int M, int H, uint16_t *out, moe_stream_t stream);

/* ---------------------------------------------------- expert-major prefill
 * Expert-major forward of T rows ("作者仍需帮助的事项": each expert read once per
 * layer for all rows routed to it).  The T*k (token, slot) pairs p = t*k + j are
 * stably sorted by expert: perm [T*k] (sorted position -> pair), inv_perm [T*k]
 * (pair -> sorted position), offsets [E+1] (first sorted position of each
 * expert).  With act_mode MOE_ACT_MXFP8 the rows are quantised to MXFP8 (E4M3
 * elements, one E8M0 scale per 32, shared exponent floor(log2 amax) - 8,
 * round-to-nearest-even with saturation) before W_g/W_u, and h likewise before
 * W_d; the contractions run on the tensor cores as block-scaled MMAs of
 * kind::mxf8f6f4 (the FP8 rate).  With MOE_ACT_MXFP4 the rows and h are quantised
 * to MXFP4 instead (E2M1 elements, shared exponent floor(log2 amax) - 2, RNE with
 * saturation at 6) and the MMAs are kind::mxf4 (both operands FP4: the FP4 rate).
 * The tile shape (one CTA per 128 weight rows, or pairs of SMs for wide tiles) is set
 * by moe_grouped_set_cta_pairs.
 * Out: partial [T*k][H] (partial_dtype MOE_PARTIAL_*), row r = o of pair perm[r]
 * (unweighted).  ws: MOE_OP_GROUPED bytes. */
moe_status moe_expert_forward_grouped(const moe_pool *pool, const uint16_t *x, int T,
                                      const int32_t *idx, int k, int act_mode,
                                      int32_t *perm, int32_t *inv_perm, int32_t *offsets,
                                      void *partial, int partial_dtype,
                                      void *ws, size_t ws_bytes, moe_stream_t stream);

/* Diagnostics of the expert-major path: after moe_expert_forward_grouped(T, k,
 * act_mode) with workspace `ws` and its `offsets` output, copy the MX-quantised h
 * that the gate/up GEMM wrote for W_d, in sorted row order: hq [T*k][I] element
 * codes, one per byte (E4M3 for MOE_ACT_MXFP8, E2M1 in the low nibble for
 * MOE_ACT_MXFP4; 16-byte aligned) and hs [T*k][I/32] E8M0 scale bytes;
 * h[r][i] = code value * 2^(hs[r][i/32] - 127).  Rows past offsets[E] (pairs with
 * an invalid expert index) are left untouched.  It lets a caller check each
 * quantisation decision on h against a reference; the workspace must not have been
 * reused since the grouped call. */
moe_status moe_grouped_read_h(const moe_pool *pool, int T, int k, int act_mode, const int32_t *offsets,
                              const void *ws, size_t ws_bytes, uint8_t *hq, uint8_t *hs, moe_stream_t stream);

/* Weighted combine of the grouped path: y[t] = sum_{j<k} w[t,j] *
 * partial[inv_perm[t*k+j]] (+ residual[t]), summed in slot order j in fp32 and
 * rounded to bf16.  No atomics: the result is deterministic. */
moe_status moe_combine(const void *partial, int partial_dtype, const int32_t *inv_perm,
                       const float *w, int T, int k, int H, const uint16_t *residual,
                       uint16_t *y, moe_stream_t stream);

/* Tile shape of moe_expert_forward_grouped's tensor-core GEMMs (process-wide, for
 * calls that start after it returns).  One-part tiles of 128 or more columns can run
 * on pairs of SMs: a cluster of two CTAs issuing tcgen05 MMAs of cta_group::2, M = 256,
 * each CTA holding 128 weight rows and half of the tile's activation rows (so each SM
 * copies half of B), the odd CTA's tensor copies counted on the even CTA's barrier.
 * mode 0: never (one CTA per 128-row tile); 1: always where the tile allows it;
 * 2 (the default): with MXFP8 rows only.  Measured on a GB300 at 8192 tokens the
 * pairs took the MXFP8 GEMMs 5.35 -> 4.69 ms and the MXFP4 GEMMs 4.52 -> 4.62 ms
 * (32768 tokens: 16.4 -> 17.0 ms), hence the default.  Results agree up to the fp32
 * accumulation order of the tensor pipe, which neither shape fixes.
 * MOE_ERR_INVALID_ARG for other modes. */
moe_status moe_grouped_set_cta_pairs(int mode);

/* ------------------------------------------------------------- test support
 * Failure detection without a GPU fault.  Every device wait of the library (the
 * mbarrier waits of the copy/MMA pipelines, the grid barrier of the single-token
 * decode kernel) is bounded; on expiry the kernel records MOE_ERR_TIMEOUT in the
 * status word, stops issuing work, waits (bounded) for its own copies in flight,
 * frees any TMEM it holds and returns.  These two calls let a test make one such
 * wait run out.  Both are process-wide; call them with no work of the library in
 * flight (the wait limit is written to the current device with a synchronous copy).
 *
 * moe_debug_set_wait_limit: bound every wait by `ns` nanoseconds (0 restores the
 * default of 1 s).  MOE_ERR_CUDA if the copy fails. */
moe_status moe_debug_set_wait_limit(uint64_t ns);

/* moe_debug_set_barrier_extra: make the grid barrier of the single-token decode
 * kernel wait for `extra` (0..1024) arrivals beyond its grid, which never come, so
 * that the barrier's bounded wait runs out (0 turns the hook off).  The call then
 * writes no y, records MOE_ERR_TIMEOUT, and leaves the workspace's counters zero, so
 * the next call on the same workspace (after moe_check_status) runs normally. */
moe_status moe_debug_set_barrier_extra(int extra);

/* ----------------------------------------------------------------- tracing
 * Between moe_trace_begin(name) and moe_trace_end(), every launch of the named
 * kernel ("route_single", "route_logits", "route_select", "decode_fused",
 * "decode_prep", "decode_gateup", "decode_down", "sort_rank", "sort_scan",
 * "sort_scatter", "sort_small", "gather_quant", "gather_split", "gemm_gateup", "gemm_down",
 * "combine", "prescale") is bracketed by CUDA events
 * on its stream (at most 65536 launches are recorded).  moe_trace_end()
 * synchronises the device and returns the number of recorded launches and their
 * summed device time in milliseconds.  Tracing is process-wide and not
 * thread-safe; it creates CUDA events on first use but allocates no device
 * memory. */
moe_status moe_trace_begin(const char *kernel_name);
moe_status moe_trace_end(int *launches, double *total_ms);

#ifdef __cplusplus
}
#endif

#endif /* MOE_H */
