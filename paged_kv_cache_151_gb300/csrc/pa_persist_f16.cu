// pa_persist_f16.cu -- persistent decode kernels (whole sequences and split-KV
// partitions), f16 storage.
#include "pa_internal.h"
#include "pa_persistent.cuh"

namespace pa {

cudaError_t decode_persistent_f16(const DecodeParams &p, int D, int G, bool partial,
                                long long unit_bound, int cluster, cudaStream_t st) {
    return partial ? dispatch_persistent<__half, MODE_PARTITIONED>(p, D, G, unit_bound, cluster, st)
                   : dispatch_persistent<__half, MODE_DECODE>(p, D, G, unit_bound, cluster, st);
}

}  // namespace pa
