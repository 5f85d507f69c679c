// pa_decode_f16.cu -- decode / partitioned decode / merge kernels for f16 storage.
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

cudaError_t decode_f16(const DecodeParams &p, int D, int G, bool partial, dim3 grid,
                     int splits, cudaStream_t st) {
    return dispatch_decode<__half>(p, D, G, partial, grid, splits, st);
}

cudaError_t merge_f16(const MergeParams &p, int num_seqs, cudaStream_t st) {
    return launch_merge<__half>(p, num_seqs, st);
}

}  // namespace pa
