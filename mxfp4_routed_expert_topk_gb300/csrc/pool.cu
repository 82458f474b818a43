// Resident MXFP4 expert pool: synthetic generation, packing and unpacking.
//
// One record per expert (the pages' per-(layer, expert) 17.5 MiB file, "Deltafin
// 的功能" on the four-SSD page), laid out for both consumers:
//   W_gu codes  [2I][H/2]     gate/up rows interleaved in groups of 16
//   W_d  codes  [H][Ip/2]     Ip = I rounded up to 128 (zero padded)
//   W_gu scales [2I][H/32]    E8M0, one per 32 elements along K
//   W_d  scales [H][Ip/32]
//   W_gu scales again, [H/128][ceil(2I/128)][512], in tensor-core order
//   W_d  scales again, [Ip/128][H/128][512],      in tensor-core order
// K is contiguous in the codes and the first two scale planes, so the decode
// kernels stream whole rows and the prefill kernels cut 128-element K tiles with
// the tensor-memory-accelerator.  The last two planes (derived from the first two
// whenever a record is written) give the grouped GEMMs each stage's weight scale
// factors as one contiguous 512-byte block per 128-row tile, the layout tcgen05.cp
// copies into tensor memory, instead of 4 bytes from each of 128 rows.
#include "moe_internal.cuh"

namespace moe {
namespace {

constexpr uint64_t kGamma = 0x9E3779B97F4A7C15ull;

__device__ __forceinline__ uint64_t splitmix_finalise(uint64_t z) {
    z = (z ^ (z >> 30)) * 0xBF58476D1CE4E5B9ull;
    z = (z ^ (z >> 27)) * 0x94D049BB133111EBull;
    return z ^ (z >> 31);
}

// Counter-mode SplitMix64: output i of the stream started at key(seed, stream).
__device__ __forceinline__ uint64_t stream_key(uint64_t seed, uint64_t stream) {
    return splitmix_finalise(splitmix_finalise(seed + kGamma) ^ splitmix_finalise(stream + 2 * kGamma));
}

enum { kGen = 0, kPack = 1, kUnpack = 2 };

// Destination byte offset (within a record) of logical code byte b (b multiple of 8).
__device__ __forceinline__ uint64_t code_dst(const PoolView &v, uint64_t b) {
    const uint64_t gate = (uint64_t)v.I * v.H / 2;
    const int half_h = v.H / 2, half_i = v.I / 2;
    if (b < 2 * gate) {
        const bool up = b >= gate;
        const uint64_t bb = up ? b - gate : b;
        const uint64_t i = bb / half_h, c = bb % half_h;
        const uint64_t r = 32 * (i / kGroupRows) + (up ? kGroupRows : 0) + (i % kGroupRows);
        return r * v.ld_gu + c;
    }
    const uint64_t bb = b - 2 * gate;
    const uint64_t o = bb / half_i, c = bb % half_i;
    return v.off_d + o * v.ld_d + c;
}

__device__ __forceinline__ uint64_t scale_dst(const PoolView &v, uint64_t j) {
    const uint64_t gate = (uint64_t)v.I * v.H / 32;
    const int nh = v.H / 32, ni = v.I / 32;
    if (j < 2 * gate) {
        const bool up = j >= gate;
        const uint64_t jj = up ? j - gate : j;
        const uint64_t i = jj / nh, c = jj % nh;
        const uint64_t r = 32 * (i / kGroupRows) + (up ? kGroupRows : 0) + (i % kGroupRows);
        return v.off_sgu + r * v.lds_gu + c;
    }
    const uint64_t jj = j - 2 * gate;
    const uint64_t o = jj / ni, c = jj % ni;
    return v.off_sd + o * v.lds_d + c;
}

__global__ void pool_codes_kernel(PoolView v, int mode, uint64_t seed, int e_lo, const uint8_t *src,
                                  uint8_t *dst_logical) {
    const int e = e_lo + blockIdx.y;
    const uint64_t nwords = (uint64_t)3 * v.H * v.I / 16;
    uint8_t *rec = v.base + (uint64_t)e * v.rec;
    const uint64_t key = stream_key(seed, 2ull * (uint64_t)e);
    for (uint64_t wd = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; wd < nwords;
         wd += (uint64_t)gridDim.x * blockDim.x) {
        uint64_t *p = reinterpret_cast<uint64_t *>(rec + code_dst(v, 8 * wd));
        if (mode == kGen) {
            *p = splitmix_finalise(key + (wd + 1) * kGamma);
        } else if (mode == kPack) {
            *p = reinterpret_cast<const uint64_t *>(src)[wd];
        } else {
            reinterpret_cast<uint64_t *>(dst_logical)[wd] = *p;
        }
    }
}

__global__ void pool_scales_kernel(PoolView v, int mode, uint64_t seed, int e_lo, const uint8_t *src,
                                   uint8_t *dst_logical) {
    const int e = e_lo + blockIdx.y;
    const uint64_t n = (uint64_t)3 * v.H * v.I / 32;
    uint8_t *rec = v.base + (uint64_t)e * v.rec;
    const uint64_t key = stream_key(seed, 2ull * (uint64_t)e + 1);
    for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n; j += (uint64_t)gridDim.x * blockDim.x) {
        uint8_t *p = rec + scale_dst(v, j);
        if (mode == kGen) {
            const uint64_t r = splitmix_finalise(key + (j + 1) * kGamma);
            *p = (uint8_t)(118 + (r >> 32) % 5);
        } else if (mode == kPack) {
            *p = src[j];
        } else {
            dst_logical[j] = *p;
        }
    }
}

// Zero the padding of W_d rows (elements I..Ip-1 and their scale bytes).
__global__ void pool_pad_kernel(PoolView v, int e_lo) {
    const int e = e_lo + blockIdx.y;
    uint8_t *rec = v.base + (uint64_t)e * v.rec;
    const int pad_c = (v.Ip - v.I) / 2, pad_s = (v.Ip - v.I) / 32;
    for (int o = blockIdx.x * blockDim.x + threadIdx.x; o < v.H; o += gridDim.x * blockDim.x) {
        uint8_t *c = rec + v.off_d + (uint64_t)o * v.ld_d + v.I / 2;
        for (int q = 0; q < pad_c; q++) c[q] = 0;
        uint8_t *s = rec + v.off_sd + (uint64_t)o * v.lds_d + v.I / 32;
        for (int q = 0; q < pad_s; q++) s[q] = 0;
    }
}

// The tensor-core copies of the scale planes: byte w of the 512-byte block of (K tile
// kt, row tile mt) is scale block 4kt + w % 4 of row mt*128 + 32 ((w / 4) % 4) + w / 16
// (0 past the matrix's rows).
__global__ void pool_mma_scales_kernel(PoolView v, int e_lo) {
    const int e = e_lo + blockIdx.y;
    uint8_t *rec = v.base + (uint64_t)e * v.rec;
    const uint64_t n_gu = (uint64_t)(v.H / 128) * v.nmt_gu * 512;
    const uint64_t n_d = (uint64_t)(v.Ip / 128) * v.nmt_d * 512;
    for (uint64_t j = (uint64_t)blockIdx.x * blockDim.x + threadIdx.x; j < n_gu + n_d;
         j += (uint64_t)gridDim.x * blockDim.x) {
        const bool gu = j < n_gu;
        const uint64_t jj = gu ? j : j - n_gu;
        const int nmt = gu ? v.nmt_gu : v.nmt_d;
        const uint64_t kt = jj / ((uint64_t)nmt * 512);
        const int mt = (int)((jj / 512) % (uint64_t)nmt);
        const int w = (int)(jj % 512);
        const int row = mt * 128 + ((w >> 2) & 3) * 32 + (w >> 4);
        const uint64_t blk = 4 * kt + (uint64_t)(w & 3);
        uint8_t val = 0;
        if (gu && row < 2 * v.I) val = rec[v.off_sgu + (uint64_t)row * v.lds_gu + blk];
        if (!gu && row < v.H) val = rec[v.off_sd + (uint64_t)row * v.lds_d + blk];
        rec[(gu ? v.off_sgu_mma : v.off_sd_mma) + jj] = val;
    }
}

}  // namespace

cudaError_t launch_pool_kernel(const PoolView &v, int mode, uint64_t seed, int e_lo, int e_hi,
                               const uint8_t *codes, const uint8_t *scales, uint8_t *out_codes,
                               uint8_t *out_scales, cudaStream_t st) {
    const int ne = e_hi - e_lo;
    if (ne <= 0) return cudaSuccess;
    int chunk = 65535;
    for (int e0 = e_lo; e0 < e_hi; e0 += chunk) {
        const int n = (e_hi - e0) < chunk ? (e_hi - e0) : chunk;
        const uint64_t nwords = (uint64_t)3 * v.H * v.I / 16;
        const unsigned gx = (unsigned)((nwords + 255) / 256 < 4096 ? (nwords + 255) / 256 : 4096);
        pool_codes_kernel<<<dim3(gx, n), 256, 0, st>>>(v, mode, seed, e0, codes, out_codes);
        const uint64_t ns = (uint64_t)3 * v.H * v.I / 32;
        const unsigned gs = (unsigned)((ns + 255) / 256 < 2048 ? (ns + 255) / 256 : 2048);
        pool_scales_kernel<<<dim3(gs, n), 256, 0, st>>>(v, mode, seed, e0, scales, out_scales);
        if (mode != kUnpack && v.Ip != v.I)
            pool_pad_kernel<<<dim3((v.H + 255) / 256, n), 256, 0, st>>>(v, e0);
        if (mode != kUnpack) {
            const uint64_t nm = ((uint64_t)(v.H / 128) * v.nmt_gu + (uint64_t)(v.Ip / 128) * v.nmt_d) * 512;
            const unsigned gm = (unsigned)((nm + 255) / 256 < 2048 ? (nm + 255) / 256 : 2048);
            pool_mma_scales_kernel<<<dim3(gm, n), 256, 0, st>>>(v, e0);
        }
    }
    return cudaGetLastError();
}

}  // namespace moe
