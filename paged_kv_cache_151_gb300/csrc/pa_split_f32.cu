// pa_split_f32.cu -- cluster-split decode and partition merge kernels, f32 storage.
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

cudaError_t decode_split_f32(const DecodeParams &p, int D, int G, dim3 grid, int splits,
                           cudaStream_t st) {
    return dispatch_split<float>(p, D, G, grid, splits, st);
}

cudaError_t merge_f32(const MergeParams &p, int num_seqs, cudaStream_t st) {
    return launch_merge<float>(p, num_seqs, st);
}

}  // namespace pa
