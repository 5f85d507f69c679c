// pa_prefill_f16.cu -- prefill kernel for multi-token queries with many rows per
// sequence (a chunk of a long prompt), f16 storage.
#include "pa_internal.h"
#include "pa_prefill.cuh"
#include "pa_prefill_tc.cuh"

namespace pa {

cudaError_t prefill_f16(const DecodeParams &p, int D, int G, int groups, cudaStream_t st) {
    return dispatch_prefill<__half>(p, D, G, groups, st);
}

cudaError_t prefill_tc_f16(const DecodeParams &p, const CUtensorMap &tmap_q, int D, int G,
                           int groups, cudaStream_t st) {
    return dispatch_prefill_tc<__half>(p, tmap_q, D, G, groups, st);
}

}  // namespace pa
