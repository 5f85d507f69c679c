// pa_decode_bf16.cu -- decode / partitioned decode / merge kernels for bf16 storage.
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

cudaError_t decode_bf16(const DecodeParams &p, int D, int G, bool partial, dim3 grid,
                     int splits, cudaStream_t st) {
    return dispatch_decode<__nv_bfloat16>(p, D, G, partial, grid, splits, st);
}

cudaError_t merge_bf16(const MergeParams &p, int num_seqs, cudaStream_t st) {
    return launch_merge<__nv_bfloat16>(p, num_seqs, st);
}

}  // namespace pa
