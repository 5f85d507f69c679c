// pa_multi_f16.cu -- persistent kernel for multi-token queries (a few new tokens
// per sequence attending causally over the paged cache), f16 storage.
#include "pa_internal.h"
#include "pa_persistent.cuh"

namespace pa {

cudaError_t decode_multi_f16(const DecodeParams &p, int D, int G, long long unit_bound,
                          int cluster, cudaStream_t st) {
    return dispatch_persistent<__half, MODE_MULTI>(p, D, G, unit_bound, cluster, st);
}

}  // namespace pa
