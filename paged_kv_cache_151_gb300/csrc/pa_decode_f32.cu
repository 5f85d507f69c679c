// pa_decode_f32.cu -- decode / partitioned decode / merge kernels for f32 storage.
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

cudaError_t decode_f32(const DecodeParams &p, int D, int G, bool partial, dim3 grid,
                     int splits, cudaStream_t st) {
    return dispatch_decode<float>(p, D, G, partial, grid, splits, st);
}

cudaError_t merge_f32(const MergeParams &p, int num_seqs, cudaStream_t st) {
    return launch_merge<float>(p, num_seqs, st);
}

}  // namespace pa
