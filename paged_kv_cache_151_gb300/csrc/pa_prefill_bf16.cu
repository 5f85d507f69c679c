// pa_prefill_bf16.cu -- prefill kernel for multi-token queries with many rows per
// sequence (a chunk of a long prompt), bf16 storage.
#include "pa_internal.h"
#include "pa_prefill.cuh"
#include "pa_prefill_tc.cuh"

namespace pa {

cudaError_t prefill_bf16(const DecodeParams &p, int D, int G, int groups, cudaStream_t st) {
    return dispatch_prefill<__nv_bfloat16>(p, D, G, groups, st);
}

cudaError_t prefill_tc_bf16(const DecodeParams &p, const CUtensorMap &tmap_q, int D, int G,
                            int groups, cudaStream_t st) {
    return dispatch_prefill_tc<__nv_bfloat16>(p, tmap_q, D, G, groups, st);
}

}  // namespace pa
