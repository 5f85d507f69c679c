// pa_split_bf16.cu -- cluster-split decode and partition merge kernels, bf16 storage.
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

cudaError_t decode_split_bf16(const DecodeParams &p, int D, int G, dim3 grid, int splits,
                           cudaStream_t st) {
    return dispatch_split<__nv_bfloat16>(p, D, G, grid, splits, st);
}

cudaError_t merge_bf16(const MergeParams &p, int num_seqs, cudaStream_t st) {
    return launch_merge<__nv_bfloat16>(p, num_seqs, st);
}

}  // namespace pa
