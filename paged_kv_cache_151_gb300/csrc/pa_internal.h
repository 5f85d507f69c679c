// pa_internal.h -- declarations shared by the translation units of the
// library (not part of the public ABI).
#pragma once

#include <cuda.h>   // CUtensorMap (a plain 128-byte descriptor)
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

// Kernels that let a following decode start early (they call
// launch_dependents()) keep the shared-memory carveout the decode needs:
// an SM cannot change its L1 / shared split while one of their blocks is
// resident, and a decode block that cannot be placed would wait for that.
// Set once per kernel (and per process: the attribute is the function's).
template <auto Kernel>
inline void prefer_shared_carveout() {
    static const bool done = [] {
        cudaFuncSetAttribute(Kernel, cudaFuncAttributePreferredSharedMemoryCarveout,
                             (int)cudaSharedmemCarveoutMaxShared);
        return true;
    }();
    (void)done;
}

struct DecodeParams;
struct MergeParams;

// per storage type: cluster-split decode, persistent decode (whole sequences
// or partitions) and the partition merge; D in {64,128}, G in {1,2,4,8}.
// cudaErrorNotSupported: shape not built (or too many sequences for the
// persistent kernel's in-block sort).
cudaError_t decode_split_f32(const DecodeParams &p, int D, int G, dim3 grid, int splits,
                             cudaStream_t st);
cudaError_t decode_split_bf16(const DecodeParams &p, int D, int G, dim3 grid, int splits,
                              cudaStream_t st);
cudaError_t decode_split_f16(const DecodeParams &p, int D, int G, dim3 grid, int splits,
                             cudaStream_t st);
cudaError_t decode_persistent_f32(const DecodeParams &p, int D, int G, bool partial,
                                  long long unit_bound, int cluster, cudaStream_t st);
cudaError_t decode_persistent_bf16(const DecodeParams &p, int D, int G, bool partial,
                                   long long unit_bound, int cluster, cudaStream_t st);
cudaError_t decode_persistent_f16(const DecodeParams &p, int D, int G, bool partial,
                                  long long unit_bound, int cluster, cudaStream_t st);
// multi-token queries (16-bit storage only)
cudaError_t decode_multi_bf16(const DecodeParams &p, int D, int G, long long unit_bound,
                              int cluster, cudaStream_t st);
cudaError_t decode_multi_f16(const DecodeParams &p, int D, int G, long long unit_bound,
                             int cluster, cudaStream_t st);
// the rows of sequences with many (token, head) rows: groups of 64 rows per block
cudaError_t prefill_bf16(const DecodeParams &p, int D, int G, int groups, cudaStream_t st);
cudaError_t prefill_f16(const DecodeParams &p, int D, int G, int groups, cudaStream_t st);
constexpr int PREFILL_GROUP_ROWS = 64;     // rows of one prefill block (= its minimum)
constexpr int PREFILL_TC_ROWS = 128;      // rows of one item of the tcgen05 prefill kernel
// tmap_q: q [num_q_rows][H][D] as the 3-D tensor (D, H, rows) in boxes of
// 64 elements x G heads x 128 / G tokens with the 128-byte swizzle
cudaError_t prefill_tc_bf16(const DecodeParams &p, const CUtensorMap &tmap_q, int D, int G,
                            int groups, cudaStream_t st);
cudaError_t prefill_tc_f16(const DecodeParams &p, const CUtensorMap &tmap_q, int D, int G,
                           int groups, cudaStream_t st);
cudaError_t merge_f32(const MergeParams &p, int num_seqs, cudaStream_t st);
cudaError_t merge_bf16(const MergeParams &p, int num_seqs, cudaStream_t st);
cudaError_t merge_f16(const MergeParams &p, int num_seqs, cudaStream_t st);

// cache write
cudaError_t reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                              const int64_t *slot_mapping, int64_t num_tokens,
                              int num_kv_heads, int row_bytes, int64_t k_tok_stride_bytes,
                              int64_t v_tok_stride_bytes, int64_t num_slots,
                              cudaStream_t st);

// FP8 (E4M3) cache write; src_dtype 0 f32, 1 bf16, 2 f16; strides in elements
cudaError_t reshape_and_cache_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                                  const int64_t *slot_mapping, int64_t num_tokens,
                                  int num_kv_heads, int head_dim, int64_t k_tok_stride,
                                  int64_t v_tok_stride, int64_t num_slots, int src_dtype,
                                  const float *k_scale, const float *v_scale,
                                  cudaStream_t st);

// persistent decode over E4M3 caches (q and out bf16 / f16); partial as above
cudaError_t decode_fp8_bf16(const DecodeParams &p, int D, int G, bool partial,
                            long long unit_bound, int cluster, cudaStream_t st);
cudaError_t decode_fp8_f16(const DecodeParams &p, int D, int G, bool partial,
                           long long unit_bound, int cluster, cudaStream_t st);

// block copies for copy-on-write: every (src, dst) pair of `mapping`, in every cache
constexpr int COPY_MAX_CACHES = 256;
struct CopyParams {
    unsigned char *caches[COPY_MAX_CACHES];   // device bases, 16-byte aligned
    const int64_t *mapping;                   // device [num_pairs][2]
    int64_t num_pairs, num_blocks, block_bytes;
    int num_caches;
    unsigned int *err;
};
cudaError_t copy_blocks(const CopyParams &p, cudaStream_t st);

// device error word
cudaError_t device_error_ptr(unsigned int **out);
cudaError_t read_device_error(unsigned int *flags, bool clear);
int sm_count_of_current_device();

}  // namespace pa
