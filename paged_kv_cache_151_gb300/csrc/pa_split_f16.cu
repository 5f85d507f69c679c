// pa_split_f16.cu -- cluster-split decode and partition merge kernels, f16 storage.
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

cudaError_t decode_split_f16(const DecodeParams &p, int D, int G, dim3 grid, int splits,
                           cudaStream_t st) {
    return dispatch_split<__half>(p, D, G, grid, splits, st);
}

cudaError_t merge_f16(const MergeParams &p, int num_seqs, cudaStream_t st) {
    return launch_merge<__half>(p, num_seqs, st);
}

}  // namespace pa
