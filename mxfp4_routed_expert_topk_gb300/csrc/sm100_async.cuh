// Thin wrappers over the sm_100-family asynchronous data-movement PTX used by the
// kernels: mbarriers (with bounded waits), bulk copies, fences, a grid barrier.
#pragma once

#include <stdint.h>

#include "moe_internal.cuh"

namespace moe {

// Every wait in the library gives up after g_wait_limit_ns nanoseconds and reports
// MOE_ERR_TIMEOUT: 1 s unless moe_debug_set_wait_limit changed it.  Without relocatable
// device code each translation unit that waits holds its own copy of the variable,
// set through set_wait_limit_here() from a wrapper in that unit.
constexpr uint64_t kDefaultWaitLimitNs = 1000ull * 1000ull * 1000ull;  // 1 s
static __device__ uint64_t g_wait_limit_ns = kDefaultWaitLimitNs;

static inline cudaError_t set_wait_limit_here(uint64_t ns) {
    return cudaMemcpyToSymbol(g_wait_limit_ns, &ns, sizeof(ns));
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t global_timer_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
    return t;
}

__device__ __forceinline__ void mbar_init(uint64_t *bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive(uint64_t *bar) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.shared::cta.b64 st, [%0];\n\t}" ::"r"(smem_u32(bar))
                 : "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t *bar, uint32_t bytes) {
    asm volatile("{\n\t.reg .b64 st;\n\tmbarrier.arrive.expect_tx.shared::cta.b64 st, [%0], %1;\n\t}" ::"r"(
                     smem_u32(bar)),
                 "r"(bytes)
                 : "memory");
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t *bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}"
        : "=r"(ok)
        : "r"(smem_u32(bar)), "r"(parity)
        : "memory");
    return ok != 0;
}

// Wait for the phase of parity `parity` to complete; false (and the status word
// set to MOE_ERR_TIMEOUT with `where`) if it does not within the wait limit.
__device__ __forceinline__ bool mbar_wait(uint64_t *bar, uint32_t parity, StatusWord *st, unsigned where) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns(), lim = g_wait_limit_ns;
    for (uint32_t it = 0;; it++) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 63u && global_timer_ns() - t0 > lim) {
            set_status(st, MOE_ERR_TIMEOUT, where);
            return false;
        }
    }
}

// mbar_wait that also gives up (false, no status) once *abort_flag is set.  The flag
// is read only while the phase is still open, so a phase that is already complete
// costs one try_wait.
__device__ __forceinline__ bool mbar_wait_or_abort(uint64_t *bar, uint32_t parity, StatusWord *st, unsigned where,
                                                   const int *abort_flag) {
    if (mbar_try_wait(bar, parity)) return true;
    const uint64_t t0 = global_timer_ns(), lim = g_wait_limit_ns;
    for (uint32_t it = 0;; it++) {
        if (mbar_try_wait(bar, parity)) return true;
        if (*(const volatile int *)abort_flag) return false;
        if ((it & 63u) == 63u && global_timer_ns() - t0 > lim) {
            set_status(st, MOE_ERR_TIMEOUT, where);
            return false;
        }
    }
}

__device__ __forceinline__ uint64_t policy_evict_first() {
    uint64_t pol;
    asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
    return pol;
}

// Bulk copy global -> shared (16-byte aligned addresses, size a multiple of 16),
// completion counted on `bar` in bytes.
__device__ __forceinline__ void bulk_g2s(void *dst, const void *src, uint32_t bytes, uint64_t *bar, uint64_t pol) {
    asm volatile(
        "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint [%0], [%1], %2, [%3], %4;" ::"r"(
            smem_u32(dst)),
        "l"(src), "r"(bytes), "r"(smem_u32(bar)), "l"(pol)
        : "memory");
}

// Named barrier over `count` threads (a multiple of 32) with id `id` (1..15).
__device__ __forceinline__ void named_barrier(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__device__ __forceinline__ unsigned int ld_acquire_gpu(const unsigned int *p) {
    unsigned int v;
    asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
    return v;
}

__device__ __forceinline__ void red_release_gpu_add(unsigned int *p, unsigned int v) {
    asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}

// Grid-wide barrier among the CTAs of a cooperative launch, for the `nthreads`
// threads of the calling CTA that take part (named barrier `bar_id`; thread 0 of
// the CTA must be one of them).  The counter is zero before the launch; each of
// the G CTAs adds 1.  A CTA that has aborted does not arrive; the others then give
// up after the wait limit.  Returns false if this CTA aborted or timed out.
//
// Ordering: the CTA's writes before the barrier precede thread 0's release add
// (CTA barrier, then release at GPU scope); thread 0's acquire load that sees the
// full count precedes the CTA's reads after the barrier (acquire, then CTA
// barrier).  Data written by other CTAs before the barrier must be read through
// L2 afterwards (ld.global.cg or stronger), not through a possibly stale L1 line.
__device__ __forceinline__ bool grid_barrier(unsigned int *counter, unsigned int G, int bar_id, int nthreads,
                                             StatusWord *st, unsigned where, int *abort_flag) {
    named_barrier(bar_id, nthreads);
    if (threadIdx.x == 0 && *(volatile int *)abort_flag == 0) {
        red_release_gpu_add(counter, 1u);
        const uint64_t t0 = global_timer_ns(), lim = g_wait_limit_ns;
        while (ld_acquire_gpu(counter) < G) {
            if (global_timer_ns() - t0 > lim) {
                set_status(st, MOE_ERR_TIMEOUT, where);
                *abort_flag = 1;
                break;
            }
        }
    }
    named_barrier(bar_id, nthreads);
    return (*(volatile int *)abort_flag) == 0;
}

}  // namespace moe
