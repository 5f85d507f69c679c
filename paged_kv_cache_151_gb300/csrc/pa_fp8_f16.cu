// pa_fp8_f16.cu -- persistent decode kernels over E4M3 caches (whole sequences
// and split-KV partitions), f16 queries and outputs.
#include "pa_internal.h"
#include "pa_persistent.cuh"

namespace pa {

cudaError_t decode_fp8_f16(const DecodeParams &p, int D, int G, bool partial,
                          long long unit_bound, int cluster, cudaStream_t st) {
    return partial
               ? dispatch_persistent<__half, MODE_PARTITIONED, e4m3>(p, D, G, unit_bound, cluster, st)
               : dispatch_persistent<__half, MODE_DECODE, e4m3>(p, D, G, unit_bound, cluster, st);
}

}  // namespace pa
