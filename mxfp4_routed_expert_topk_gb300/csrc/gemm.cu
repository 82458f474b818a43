// Grouped block-scaled GEMMs of the prefill path (tcgen05).  Not built yet.
#include "prefill_internal.cuh"

namespace moe {

cudaError_t launch_grouped_gemms(const PoolView &v, int T, int k, const int32_t *offsets, const GroupedWs &g,
                                 void *partial, int partial_dtype, StatusWord *st, cudaStream_t stream) {
    (void)v; (void)T; (void)k; (void)offsets; (void)g; (void)partial; (void)partial_dtype; (void)st; (void)stream;
    return cudaErrorNotSupported;
}

}  // namespace moe
