// Streamed expert pool: the expert records of a layer live in caller-owned host
// memory, and an HBM cache of C record slots holds the experts in use.  This is the
// pages' streamed-expert design ("技术亮点": experts read on demand with a cache;
// "存储子系统" on the four-SSD page: demand reads, one unit per (layer, expert)) in
// GB300 form: the records sit in pinned host memory and are copied over NVLink-C2C
// with one cudaMemcpyAsync per record.  The cache is an ordinary pool view of C
// records, so the decode and grouped kernels run on it unchanged with slot indices
// in place of expert indices.
//
// Host code only: a least-recently-used slot map with the slots of the current call
// pinned, and the allocation of the host records on the GPU's own NUMA node.
#include <linux/mempolicy.h>
#include <stdlib.h>
#include <string.h>
#include <sys/mman.h>
#include <sys/syscall.h>
#include <unistd.h>

#include <new>
#include <vector>

#include "moe_internal.cuh"

struct moe_stream_pool {
    const uint8_t *host;        // E records of rec bytes
    int E;
    uint64_t rec;
    moe_pool *cache;            // view over the device cache (C records); null when planning only
    uint8_t *dev;               // device cache base (null: plan only, no copies)
    int C;
    std::vector<int> slot_of;   // [E] slot holding expert e, or -1
    std::vector<int> expert_in; // [C] expert in slot s, or -1
    std::vector<uint64_t> last; // [C] clock of the last call that used slot s
    uint64_t clock = 0;
    uint64_t hits = 0, misses = 0, bytes = 0;
};

extern "C" {

moe_status moe_stream_pool_create(moe_stream_pool **out, const void *host_records, size_t host_bytes, int E, int H,
                                  int I, void *dev_cache, size_t cache_bytes) {
    if (out == nullptr || host_records == nullptr) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    const size_t rec = moe_pool_record_bytes(H, I);
    if (rec == 0 || E < 1) return MOE_ERR_UNSUPPORTED_SHAPE;
    if (host_bytes < (size_t)E * rec) return MOE_ERR_INVALID_ARG;
    const size_t C = cache_bytes / rec;
    if (C < 1 || C > (size_t)E) return MOE_ERR_INVALID_ARG;
    moe_stream_pool *sp = new (std::nothrow) moe_stream_pool();
    if (sp == nullptr) return MOE_ERR_INVALID_ARG;
    sp->host = (const uint8_t *)host_records;
    sp->E = E;
    sp->rec = rec;
    sp->C = (int)C;
    sp->dev = (uint8_t *)dev_cache;
    sp->cache = nullptr;
    if (dev_cache != nullptr) {
        const moe_status s = moe_pool_create(&sp->cache, dev_cache, C * rec, (int)C, H, I);
        if (s != MOE_OK) {
            delete sp;
            return s;
        }
    }
    sp->slot_of.assign((size_t)E, -1);
    sp->expert_in.assign(C, -1);
    sp->last.assign(C, 0);
    *out = sp;
    return MOE_OK;
}

void moe_stream_pool_destroy(moe_stream_pool *sp) {
    if (sp == nullptr) return;
    moe_pool_destroy(sp->cache);
    delete sp;
}

const moe_pool *moe_stream_pool_cache(const moe_stream_pool *sp) { return sp == nullptr ? nullptr : sp->cache; }

int moe_stream_pool_slots(const moe_stream_pool *sp) { return sp == nullptr ? 0 : sp->C; }

moe_status moe_stream_pool_map(moe_stream_pool *sp, const int32_t *idx_host, int n, int32_t *slot_host,
                               moe_stream_t stream) {
    if (sp == nullptr || (n > 0 && (idx_host == nullptr || slot_host == nullptr)) || n < 0) return MOE_ERR_INVALID_ARG;
    const uint64_t now = ++sp->clock;
    // distinct valid experts of this call must fit the cache
    int distinct = 0;
    for (int i = 0; i < n; i++) {
        const int e = idx_host[i];
        if (e < 0 || e >= sp->E) continue;
        bool seen = false;
        for (int j = 0; j < i && !seen; j++) seen = idx_host[j] == e;
        distinct += !seen;
    }
    if (distinct > sp->C) return MOE_ERR_UNSUPPORTED_SHAPE;
    // hits first, so that their slots are marked in use before any eviction
    for (int i = 0; i < n; i++) {
        const int e = idx_host[i];
        if (e < 0 || e >= sp->E) continue;
        const int s = sp->slot_of[(size_t)e];
        if (s >= 0 && sp->last[(size_t)s] != now) {
            sp->last[(size_t)s] = now;
            sp->hits++;
        }
    }
    cudaStream_t st = (cudaStream_t)stream;
    for (int i = 0; i < n; i++) {
        const int e = idx_host[i];
        if (e < 0 || e >= sp->E) {
            slot_host[i] = -1;  // the kernels report it (MOE_ERR_BAD_INDEX) and add nothing
            continue;
        }
        int s = sp->slot_of[(size_t)e];
        if (s < 0) {
            // least recently used slot among those this call does not use (one exists:
            // distinct <= C)
            int v = -1;
            for (int c = 0; c < sp->C; c++) {
                if (sp->last[(size_t)c] == now) continue;
                if (v < 0 || sp->last[(size_t)c] < sp->last[(size_t)v]) v = c;
            }
            if (v < 0) return MOE_ERR_UNSUPPORTED_SHAPE;
            if (sp->expert_in[(size_t)v] >= 0) sp->slot_of[(size_t)sp->expert_in[(size_t)v]] = -1;
            sp->expert_in[(size_t)v] = e;
            sp->slot_of[(size_t)e] = v;
            sp->last[(size_t)v] = now;
            s = v;
            sp->misses++;
            sp->bytes += sp->rec;
            if (sp->dev != nullptr) {
                // after every earlier use of the slot on this stream; before every later one
                if (cudaMemcpyAsync(sp->dev + (size_t)v * sp->rec, sp->host + (size_t)e * sp->rec, sp->rec,
                                    cudaMemcpyHostToDevice, st) != cudaSuccess)
                    return MOE_ERR_CUDA;
            }
        }
        slot_host[i] = s;
    }
    return MOE_OK;
}

// A Grace host has one NUMA node per CPU die, and a GPU's copy engines reach the
// memory of their own die over NVLink-C2C but the other die's only through the
// CPU-to-CPU link, several times slower.  The pages are given a preferred node
// before they exist (mbind on the fresh mapping), then faulted in and pinned by
// cudaHostRegister; MPOL_PREFERRED rather than MPOL_BIND, so that a full node falls
// back to another instead of failing the allocation.
static size_t host_map_len(size_t bytes) {
    const long pg = sysconf(_SC_PAGESIZE);
    const size_t page = pg > 0 ? (size_t)pg : 4096;
    return (bytes + page - 1) / page * page;
}

moe_status moe_host_alloc(int device, size_t bytes, void **out, int *numa_node) {
    if (out == nullptr || bytes == 0) return MOE_ERR_INVALID_ARG;
    *out = nullptr;
    if (numa_node != nullptr) *numa_node = -1;
    int want = -1;
    if (cudaDeviceGetAttribute(&want, cudaDevAttrHostNumaId, device) != cudaSuccess) {
        (void)cudaGetLastError();
        want = -1;
    }
    const size_t len = host_map_len(bytes);
    void *p = mmap(nullptr, len, PROT_READ | PROT_WRITE, MAP_PRIVATE | MAP_ANONYMOUS, -1, 0);
    if (p == MAP_FAILED) return MOE_ERR_INVALID_ARG;
    constexpr int kMaskBits = 1024;
    if (want >= 0 && want < kMaskBits) {
        unsigned long mask[kMaskBits / (8 * sizeof(unsigned long))] = {};
        mask[(size_t)want / (8 * sizeof(unsigned long))] |= 1ul << ((size_t)want % (8 * sizeof(unsigned long)));
        // failure (a node outside this process's cpuset) leaves the kernel's default
        (void)syscall(SYS_mbind, p, len, (unsigned long)MPOL_PREFERRED, mask, (unsigned long)kMaskBits + 1, 0ul);
    }
    if (cudaHostRegister(p, len, cudaHostRegisterDefault) != cudaSuccess) {
        (void)cudaGetLastError();
        munmap(p, len);
        return MOE_ERR_CUDA;
    }
    if (numa_node != nullptr) {
        int node = -1;
        if (syscall(SYS_get_mempolicy, &node, nullptr, 0ul, p, (unsigned long)(MPOL_F_NODE | MPOL_F_ADDR)) == 0)
            *numa_node = node;
    }
    *out = p;
    return MOE_OK;
}

moe_status moe_host_free(void *p, size_t bytes) {
    if (p == nullptr) return MOE_OK;
    if (bytes == 0) return MOE_ERR_INVALID_ARG;
    const cudaError_t e = cudaHostUnregister(p);
    if (e != cudaSuccess) (void)cudaGetLastError();
    munmap(p, host_map_len(bytes));
    return e == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}

int moe_host_numa_node(int device) {
    int n = -1;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrHostNumaId, device) != cudaSuccess) {
        (void)cudaGetLastError();
        return -1;
    }
    return n;
}

moe_status moe_stream_pool_stats(const moe_stream_pool *sp, uint64_t *hits, uint64_t *misses, uint64_t *bytes) {
    if (sp == nullptr || hits == nullptr || misses == nullptr || bytes == nullptr) return MOE_ERR_INVALID_ARG;
    *hits = sp->hits;
    *misses = sp->misses;
    *bytes = sp->bytes;
    return MOE_OK;
}

}  // extern "C"
