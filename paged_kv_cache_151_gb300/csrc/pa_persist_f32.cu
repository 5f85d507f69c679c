// pa_persist_f32.cu -- persistent decode kernels (whole sequences and split-KV
// partitions), f32 storage.
#include "pa_internal.h"
#include "pa_persistent.cuh"

namespace pa {

cudaError_t decode_persistent_f32(const DecodeParams &p, int D, int G, bool partial,
                                long long unit_bound, int cluster, cudaStream_t st) {
    return partial ? dispatch_persistent<float, MODE_PARTITIONED>(p, D, G, unit_bound, cluster, st)
                   : dispatch_persistent<float, MODE_DECODE>(p, D, G, unit_bound, cluster, st);
}

}  // namespace pa
