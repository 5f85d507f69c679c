// pa_api.cu -- the C ABI (include/pa.h): host-side argument checks, launch
// configuration and dispatch.  No entry point allocates, frees or
// synchronises (except pa_device_error).
#include <atomic>
#include <cstring>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>

#include "../../include/pa.h"
#include "pa_decode.cuh"
#include "pa_internal.h"

namespace pa {

int sm_count_of_current_device() {
    static std::atomic<int> cache[64];
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) {
        int v = cache[dev].load(std::memory_order_relaxed);
        if (v > 0) return v;
    }
    int n = 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    if (dev >= 0 && dev < 64) cache[dev].store(n, std::memory_order_relaxed);
    return n;
}

}  // namespace pa

namespace {

constexpr size_t kAlign = 256;

size_t align_up(size_t x) { return (x + kAlign - 1) / kAlign * kAlign; }

int elem_size(int32_t dtype) {
    switch (dtype) {
        case PA_F32: return 4;
        case PA_BF16: return 2;
        case PA_F16: return 2;
        default: return 0;
    }
}

bool aligned16(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

// Checks shared by the decode entry points.
int check_decode_args(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *seq_lens, int32_t num_seqs,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int64_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                      int64_t q_seq_stride, float scale, int32_t dtype) {
    if (num_seqs < 0 || num_heads <= 0 || num_kv_heads <= 0 || head_dim <= 0 ||
        num_blocks < 0 || max_blocks_per_seq < 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens)
        return PA_ERR_INVALID_ARG;
    if (elem_size(dtype) == 0) return PA_ERR_UNSUPPORTED;
    if (num_heads % num_kv_heads) return PA_ERR_INVALID_ARG;
    const int G = num_heads / num_kv_heads;
    if (block_size != 16) return PA_ERR_UNSUPPORTED;
    if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
    if (G != 1 && G != 2 && G != 4 && G != 8) return PA_ERR_UNSUPPORTED;
    if (num_seqs > 65535 || num_kv_heads > 65535) return PA_ERR_UNSUPPORTED;
    if (q_seq_stride < (int64_t)num_heads * head_dim) return PA_ERR_INVALID_ARG;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return PA_ERR_INVALID_ARG;
    if (!(scale == scale)) return PA_ERR_INVALID_ARG;        // NaN scale
    if (num_blocks > (int64_t)INT32_MAX) return PA_ERR_UNSUPPORTED;
    return PA_OK;
}

cudaError_t run_split(const pa::DecodeParams &p, int dtype, int D, int G, dim3 grid,
                      int splits, cudaStream_t st) {
    switch (dtype) {
        case PA_F32: return pa::decode_split_f32(p, D, G, grid, splits, st);
        case PA_BF16: return pa::decode_split_bf16(p, D, G, grid, splits, st);
        default: return pa::decode_split_f16(p, D, G, grid, splits, st);
    }
}

// Blocks per cluster of the persistent kernel.  Whole-sequence decode shares
// each cluster's block stream over several SMs (over 16-bit caches: four
// blocks of eight warps, one block per SM) so that long sequences spread out;
// partitions are already uniform work units.
#ifndef PA_DECODE_CLUSTER
#define PA_DECODE_CLUSTER 4
#endif
// Multi-token queries over 16-bit caches: blocks of eight warps, clusters of
// four, like whole-sequence decode.
#ifndef PA_MULTI_CLUSTER
#define PA_MULTI_CLUSTER 4
#endif
// The prefill path (long multi-token runs) on the tcgen05 tensor cores (1) or
// on warp-level MMAs (0).
#ifndef PA_PREFILL_TC
#define PA_PREFILL_TC 1
#endif
// E4M3 caches run three blocks per SM; clusters of four deal their units
// more evenly there.
#ifndef PA_F8_CLUSTER
#define PA_F8_CLUSTER 4
#endif

cudaError_t run_persistent(const pa::DecodeParams &p, int dtype, int D, int G, bool partial,
                           long long unit_bound, cudaStream_t st) {
    const int cluster = partial ? 1 : PA_DECODE_CLUSTER;
    switch (dtype) {
        case PA_F32: return pa::decode_persistent_f32(p, D, G, partial, unit_bound, cluster, st);
        case PA_BF16: return pa::decode_persistent_bf16(p, D, G, partial, unit_bound, cluster, st);
        default: return pa::decode_persistent_f16(p, D, G, partial, unit_bound, cluster, st);
    }
}

// cuTensorMapEncodeTiled from the driver, looked up once through the runtime
// (no link-time dependency on the driver library).
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
    static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
    static std::once_flag once;
    std::call_once(once, [] {
        void *ptr = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                             cudaEnableDefault, &q) == cudaSuccess &&
            q == cudaDriverEntryPointSuccess)
            fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(ptr);
    });
    return fn;
}

// A cache [num_blocks][H_kv][16][D] as the 3-D tensor (D, 16 rows,
// num_blocks*H_kv).  16-bit caches are read in boxes of 64 elements (128
// bytes) x 16 rows with the 128-byte swizzle; E4M3 caches in boxes of the
// whole row (D bytes) x 16 rows with the D-byte swizzle.
bool encode_cache_map(CUtensorMap *m, const void *base, int64_t num_blocks, int32_t hkv,
                      int32_t head_dim, int32_t kv_dtype, uint32_t box_rows = 16) {
    auto enc = tensor_map_encoder();
    if (!enc) return false;
    const bool f8 = kv_dtype == PA_E4M3;
    const cuuint64_t es = f8 ? 1 : 2;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, 16, (cuuint64_t)(num_blocks * hkv)};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * es, (cuuint64_t)head_dim * es * 16};
    const cuuint32_t box[3] = {f8 ? (cuuint32_t)head_dim : 64u, box_rows, 1};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = f8 ? CU_TENSOR_MAP_DATA_TYPE_UINT8
                                   : kv_dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                         : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    const CUtensorMapSwizzle sw = (f8 && head_dim == 64) ? CU_TENSOR_MAP_SWIZZLE_64B
                                                         : CU_TENSOR_MAP_SWIZZLE_128B;
    return enc(m, dt, 3, const_cast<void *>(base), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, sw, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
               CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// q [rows][H][D] (rows q_row_stride elements apart, 16-bit) as the 3-D tensor
// (D, H, rows), read in boxes of 64 elements x G heads x 128 / G tokens with
// the 128-byte swizzle: one box is 128 rows of 128 bytes, row = token * G +
// head, the layout of one prefill item's Q operand.
bool encode_q_map(CUtensorMap *m, const void *q, int64_t rows, int32_t num_heads,
                  int32_t head_dim, int64_t q_row_stride, int32_t G, int32_t dtype) {
    auto enc = tensor_map_encoder();
    if (!enc || G <= 0 || pa::PREFILL_TC_ROWS % G != 0 || rows <= 0) return false;
    const cuuint64_t dims[3] = {(cuuint64_t)head_dim, (cuuint64_t)num_heads, (cuuint64_t)rows};
    const cuuint64_t strides[2] = {(cuuint64_t)head_dim * 2, (cuuint64_t)q_row_stride * 2};
    const cuuint32_t box[3] = {64u, (cuuint32_t)G, (cuuint32_t)(pa::PREFILL_TC_ROWS / G)};
    const cuuint32_t estr[3] = {1, 1, 1};
    const CUtensorMapDataType dt = dtype == PA_BF16 ? CU_TENSOR_MAP_DATA_TYPE_BFLOAT16
                                                    : CU_TENSOR_MAP_DATA_TYPE_FLOAT16;
    return enc(m, dt, 3, const_cast<void *>(q), dims, strides, box, estr,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// One-shot test hook armed by pa_test_stall_next_decode, taken by the next
// decode call that prepares its parameters here.
std::atomic<int> g_test_stall{0};

// Fill the tensor maps the persistent kernel needs for 16-bit and E4M3
// caches (kv_dtype: the caches' storage type).
bool prepare_maps(pa::DecodeParams &p, int32_t kv_dtype, int32_t head_dim) {
    p.test_stall = g_test_stall.exchange(0, std::memory_order_acq_rel);
    if (kv_dtype == PA_F32) return true;
    if (p.num_blocks <= 0) return true;            // nothing can be read
    if (!encode_cache_map(&p.tmap_k, p.k_cache, p.num_blocks, p.num_kv_heads, head_dim,
                          kv_dtype) ||
        !encode_cache_map(&p.tmap_v, p.v_cache, p.num_blocks, p.num_kv_heads, head_dim,
                          kv_dtype))
        return false;
    if (kv_dtype == PA_E4M3) return true;
    // 8-row boxes: with the 128-byte swizzle they land exactly where rows 0..7
    // of a 16-row box would
    return encode_cache_map(&p.tmap_k8, p.k_cache, p.num_blocks, p.num_kv_heads, head_dim,
                            kv_dtype, 8) &&
           encode_cache_map(&p.tmap_v8, p.v_cache, p.num_blocks, p.num_kv_heads, head_dim,
                            kv_dtype, 8);
}

// The persistent kernel reads each query row with 16-byte loads.
bool q_rows_aligned(const void *q, int64_t q_seq_stride, int32_t dtype) {
    return aligned16(q) && ((q_seq_stride * elem_size(dtype)) % 16) == 0;
}

cudaError_t run_merge(const pa::MergeParams &p, int dtype, int num_seqs, cudaStream_t st) {
    switch (dtype) {
        case PA_F32: return pa::merge_f32(p, num_seqs, st);
        case PA_BF16: return pa::merge_bf16(p, num_seqs, st);
        default: return pa::merge_f16(p, num_seqs, st);
    }
}

// Cluster split of one (sequence, KV head) when the caller leaves it open:
// enough thread blocks to fill the GPU a few times over, and no more than
// about 64 blocks (1024 tokens) of the longest possible sequence per split.
int auto_splits(int32_t num_seqs, int32_t num_kv_heads, int32_t max_blocks_per_seq) {
    int sms = pa::sm_count_of_current_device();
    if (sms <= 0) sms = 152;
    const int64_t units = (int64_t)num_seqs * num_kv_heads;
    const int64_t slots = (int64_t)sms * 2;        // resident thread blocks at 2 per SM
    int c = 1;
    while (c < 8 && (units * c < 2 * slots || max_blocks_per_seq / c > 64)) c *= 2;
    return c;
}

int decode_common(void *out, const void *q, const void *k_cache, const void *v_cache,
                  const int32_t *block_tables, const int32_t *seq_lens, int32_t num_seqs,
                  int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                  int64_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                  int64_t q_seq_stride, float scale, int32_t dtype, int32_t splits,
                  void *stream) {
    int rc = check_decode_args(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                               num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                               max_blocks_per_seq, q_seq_stride, scale, dtype);
    if (rc != PA_OK || num_seqs == 0) return rc;
    if (splits < 0 || splits > 8 || (splits & (splits - 1))) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.out = out; p.q = q; p.k_cache = k_cache; p.v_cache = v_cache;
    p.block_tables = block_tables; p.seq_lens = seq_lens;
    p.num_blocks = num_blocks; p.q_seq_stride = q_seq_stride;
    p.num_seqs = num_seqs; p.num_heads = num_heads; p.num_kv_heads = num_kv_heads;
    p.max_blocks = max_blocks_per_seq;
    p.scale_log2 = scale * pa::LOG2E;
    if (pa::device_error_ptr(&p.err) != cudaSuccess) return PA_ERR_CUDA;
    const int G = num_heads / num_kv_heads;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    cudaError_t e = cudaErrorNotSupported;
    if (splits == 0 && q_rows_aligned(q, q_seq_stride, dtype) && aligned16(out) &&
        prepare_maps(p, dtype, head_dim)) {
        e = run_persistent(p, dtype, head_dim, G, false, (long long)num_seqs * num_kv_heads, st);
        if (e != cudaErrorNotSupported) return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
    }
    if (splits == 0) splits = auto_splits(num_seqs, num_kv_heads, max_blocks_per_seq);
    dim3 grid((unsigned)splits, (unsigned)num_kv_heads, (unsigned)num_seqs);
    e = run_split(p, dtype, head_dim, G, grid, splits, st);
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

struct WorkspaceLayout {
    size_t o, m, l, total;
};

bool workspace_layout(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                      int32_t max_seq_len, int32_t partition_size, WorkspaceLayout *w) {
    if (num_seqs <= 0 || num_heads <= 0 || head_dim <= 0 || max_seq_len < 0 ||
        partition_size <= 0 || partition_size % 16)
        return false;
    const size_t P = (size_t)((max_seq_len + (int64_t)partition_size - 1) / partition_size);
    // Every product and sum is checked: the arguments allow about 2^71 bytes,
    // and a wrapped size would pass the workspace checks.
    size_t rows = 0, o_bytes = 0, ml_bytes = 0;
    if (__builtin_mul_overflow((size_t)num_seqs, (size_t)num_heads, &rows) ||
        __builtin_mul_overflow(rows, P > 0 ? P : (size_t)1, &rows) ||
        __builtin_mul_overflow(rows, (size_t)head_dim * sizeof(float), &o_bytes) ||
        __builtin_mul_overflow(rows, sizeof(float), &ml_bytes) ||
        o_bytes > (SIZE_MAX >> 2) || ml_bytes > (SIZE_MAX >> 2))
        return false;
    w->o = 0;
    w->m = align_up(o_bytes);
    w->l = w->m + align_up(ml_bytes);
    w->total = w->l + align_up(ml_bytes);
    return true;
}

}  // namespace

extern "C" {

int pa_abi_version(void) { return 4; }

int pa_test_stall_next_decode(void) {
    g_test_stall.store(1, std::memory_order_release);
    return PA_OK;
}

const char *pa_status_string(int status) {
    switch (status) {
        case PA_OK: return "ok";
        case PA_ERR_INVALID_ARG: return "invalid argument";
        case PA_ERR_UNSUPPORTED: return "unsupported shape or dtype";
        case PA_ERR_WORKSPACE: return "workspace missing or too small";
        case PA_ERR_CUDA: return "CUDA error";
        default: return "unknown status";
    }
}

int pa_reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int64_t num_tokens,
                         int32_t num_kv_heads, int32_t head_dim, int64_t k_token_stride,
                         int64_t v_token_stride, int64_t num_blocks, int32_t block_size,
                         int32_t dtype, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    if (es == 0) return PA_ERR_UNSUPPORTED;
    if (block_size != 16) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (k_token_stride < row || v_token_stride < row) return PA_ERR_INVALID_ARG;
    const int64_t row_bytes = (int64_t)head_dim * es;
    if (row_bytes % 16 || row_bytes > INT32_MAX) return PA_ERR_UNSUPPORTED;
    if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
         reinterpret_cast<uintptr_t>(k_cache) | reinterpret_cast<uintptr_t>(v_cache)) %
        es)
        return PA_ERR_INVALID_ARG;
    cudaError_t e = pa::reshape_and_cache(
        k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, (int)row_bytes,
        k_token_stride * es, v_token_stride * es, num_blocks * block_size,
        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, const int32_t *seq_lens, int32_t num_seqs,
              int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
              int32_t block_size, int32_t max_blocks_per_seq, int64_t q_seq_stride,
              float scale, int32_t dtype, void *stream) {
    return decode_common(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                         num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                         max_blocks_per_seq, q_seq_stride, scale, dtype, 0, stream);
}

int pa_decode_split(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, const int32_t *seq_lens, int32_t num_seqs,
                    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int64_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                    int64_t q_seq_stride, float scale, int32_t dtype, int32_t splits,
                    void *stream) {
    return decode_common(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                         num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                         max_blocks_per_seq, q_seq_stride, scale, dtype, splits, stream);
}

size_t pa_decode_partitioned_workspace_size(int32_t num_seqs, int32_t num_heads,
                                            int32_t head_dim, int32_t max_seq_len,
                                            int32_t partition_size) {
    WorkspaceLayout w;
    if (!workspace_layout(num_seqs, num_heads, head_dim, max_seq_len, partition_size, &w))
        return 0;
    return w.total;
}

int pa_decode_partitioned(void *out, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *block_tables,
                          const int32_t *seq_lens, int32_t num_seqs, int32_t num_heads,
                          int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                          int32_t block_size, int32_t max_blocks_per_seq,
                          int64_t q_seq_stride, float scale, int32_t dtype,
                          int32_t partition_size, int32_t max_seq_len, void *workspace,
                          size_t workspace_bytes, void *stream) {
    int rc = check_decode_args(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                               num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                               max_blocks_per_seq, q_seq_stride, scale, dtype);
    if (rc != PA_OK) return rc;
    if (partition_size <= 0 || partition_size % 16 || max_seq_len < 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    WorkspaceLayout w;
    if (!workspace_layout(num_seqs, num_heads, head_dim, max_seq_len, partition_size, &w))
        return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < w.total ||
        (reinterpret_cast<uintptr_t>(workspace) % kAlign))
        return PA_ERR_WORKSPACE;
    const int64_t P64 = ((int64_t)max_seq_len + partition_size - 1) / partition_size;
    const int P = (int)(P64 > 0 ? P64 : 1);
    if (P64 > INT32_MAX) return PA_ERR_UNSUPPORTED;
    unsigned char *ws = static_cast<unsigned char *>(workspace);

    pa::DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.out = out; p.q = q; p.k_cache = k_cache; p.v_cache = v_cache;
    p.block_tables = block_tables; p.seq_lens = seq_lens;
    p.part_o = reinterpret_cast<float *>(ws + w.o);
    p.part_m = reinterpret_cast<float *>(ws + w.m);
    p.part_l = reinterpret_cast<float *>(ws + w.l);
    p.num_blocks = num_blocks; p.q_seq_stride = q_seq_stride;
    p.num_seqs = num_seqs; p.num_heads = num_heads; p.num_kv_heads = num_kv_heads;
    p.max_blocks = max_blocks_per_seq;
    p.partition_blocks = partition_size / 16;
    p.max_parts = P;
    p.max_seq_len = max_seq_len;
    p.scale_log2 = scale * pa::LOG2E;
    if (pa::device_error_ptr(&p.err) != cudaSuccess) return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int G = num_heads / num_kv_heads;
    if (!q_rows_aligned(q, q_seq_stride, dtype)) return PA_ERR_UNSUPPORTED;
    if (!prepare_maps(p, dtype, head_dim)) return PA_ERR_CUDA;
    cudaError_t e = run_persistent(p, dtype, head_dim, G, true,
                                   (long long)num_seqs * num_kv_heads * P, st);
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return PA_ERR_CUDA;

    pa::MergeParams mp;
    std::memset(&mp, 0, sizeof mp);
    mp.out = out;
    mp.part_o = p.part_o; mp.part_m = p.part_m; mp.part_l = p.part_l;
    mp.seq_lens = seq_lens;
    mp.num_heads = num_heads; mp.head_dim = head_dim;
    mp.max_parts = P; mp.partition_size = partition_size;
    const int64_t cap = (int64_t)max_blocks_per_seq * 16;
    mp.seq_cap = (int)(max_seq_len < cap ? max_seq_len : cap);
    e = run_merge(mp, dtype, num_seqs, st);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_decode_multi(void *out, const void *q, const void *k_cache, const void *v_cache,
                    const int32_t *block_tables, const int32_t *seq_lens,
                    const int32_t *query_start, int32_t num_seqs, int32_t num_q_rows,
                    int32_t max_query_len, int32_t num_heads, int32_t num_kv_heads,
                    int32_t head_dim, int64_t num_blocks, int32_t block_size,
                    int32_t max_blocks_per_seq, int64_t q_row_stride, float scale,
                    int32_t dtype, void *stream) {
    int rc = check_decode_args(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                               num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                               max_blocks_per_seq, q_row_stride, scale, dtype);
    if (rc != PA_OK) return rc;
    if (num_q_rows < 0 || max_query_len < 0) return PA_ERR_INVALID_ARG;
    if (num_seqs == 0 || num_q_rows == 0) return PA_OK;
    if (!query_start) return PA_ERR_INVALID_ARG;
    if (dtype == PA_F32) return PA_ERR_UNSUPPORTED;
    if (!q_rows_aligned(q, q_row_stride, dtype) || !aligned16(out)) return PA_ERR_INVALID_ARG;
    const int G = num_heads / num_kv_heads;
    // Sequences with at least PREFILL_GROUP_ROWS (token, head) rows go to the prefill
    // kernel (blocks of 64 rows sharing one K/V ring), the others to the persistent
    // kernel's work units: (sequence, KV head, 16-row tile of the rows).
    const int64_t rows = (int64_t)(max_query_len < num_q_rows ? max_query_len : num_q_rows) * G;
    const bool split = rows >= pa::PREFILL_GROUP_ROWS;
    const int64_t small_rows = split ? pa::PREFILL_GROUP_ROWS - 1 : rows;
    const int64_t tiles = (small_rows + 15) / 16;
    if (rows == 0) return PA_OK;
    pa::DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.out = out; p.q = q; p.k_cache = k_cache; p.v_cache = v_cache;
    p.block_tables = block_tables; p.seq_lens = seq_lens;
    p.query_start = query_start;
    p.max_query_len = max_query_len;
    p.num_q_rows = num_q_rows;
    p.num_blocks = num_blocks; p.q_seq_stride = q_row_stride;
    p.num_seqs = num_seqs; p.num_heads = num_heads; p.num_kv_heads = num_kv_heads;
    p.max_blocks = max_blocks_per_seq;
    p.scale_log2 = scale * pa::LOG2E;
    p.mq_split_rows = split ? pa::PREFILL_GROUP_ROWS : 0;
    if (pa::device_error_ptr(&p.err) != cudaSuccess) return PA_ERR_CUDA;
    if (!prepare_maps(p, dtype, head_dim)) return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    if (split) {
        cudaError_t e;
        if (PA_PREFILL_TC) {                       // tcgen05: items of 128 rows
            const int groups = (int)((rows + pa::PREFILL_TC_ROWS - 1) / pa::PREFILL_TC_ROWS);
            CUtensorMap tmap_q;
            if (!encode_q_map(&tmap_q, q, num_q_rows, num_heads, head_dim, q_row_stride, G, dtype))
                return PA_ERR_CUDA;
            e = dtype == PA_BF16 ? pa::prefill_tc_bf16(p, tmap_q, head_dim, G, groups, st)
                                 : pa::prefill_tc_f16(p, tmap_q, head_dim, G, groups, st);
        } else {                                   // warp-level MMAs: items of 64 rows
            const int groups = (int)((rows + pa::PREFILL_GROUP_ROWS - 1) / pa::PREFILL_GROUP_ROWS);
            e = dtype == PA_BF16 ? pa::prefill_bf16(p, head_dim, G, groups, st)
                                 : pa::prefill_f16(p, head_dim, G, groups, st);
        }
        if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    const long long unit_bound = (long long)num_seqs * num_kv_heads * tiles;
    cudaError_t e = dtype == PA_BF16
                        ? pa::decode_multi_bf16(p, head_dim, G, unit_bound, PA_MULTI_CLUSTER, st)
                        : pa::decode_multi_f16(p, head_dim, G, unit_bound, PA_MULTI_CLUSTER, st);
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// ---- block copies for copy-on-write ---------------------------------------

int pa_copy_blocks(void *const *caches, int32_t num_caches, const int64_t *block_mapping,
                   int64_t num_pairs, int64_t num_blocks, int64_t block_bytes, void *stream) {
    if (num_pairs < 0 || num_blocks < 0 || block_bytes <= 0 || num_caches < 0)
        return PA_ERR_INVALID_ARG;
    if (block_bytes % 16) return PA_ERR_UNSUPPORTED;
    if (num_caches > pa::COPY_MAX_CACHES) return PA_ERR_UNSUPPORTED;
    if (num_pairs == 0 || num_caches == 0) return PA_OK;
    if (!caches || !block_mapping) return PA_ERR_INVALID_ARG;
    if (num_blocks > INT64_MAX / block_bytes) return PA_ERR_INVALID_ARG;
    pa::CopyParams p;
    std::memset(&p, 0, sizeof p);
    for (int32_t c = 0; c < num_caches; ++c) {
        if (!caches[c] || !aligned16(caches[c])) return PA_ERR_INVALID_ARG;
        p.caches[c] = static_cast<unsigned char *>(caches[c]);
    }
    p.num_caches = num_caches;
    p.mapping = block_mapping;
    p.num_pairs = num_pairs;
    p.num_blocks = num_blocks;
    p.block_bytes = block_bytes;
    if (pa::device_error_ptr(&p.err) != cudaSuccess) return PA_ERR_CUDA;
    cudaError_t e = pa::copy_blocks(p, static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// ---- FP8 (E4M3) KV cache --------------------------------------------------

int pa_reshape_and_cache_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                             const float *k_scale, const float *v_scale,
                             const int64_t *slot_mapping, int64_t num_tokens,
                             int32_t num_kv_heads, int32_t head_dim, int64_t k_token_stride,
                             int64_t v_token_stride, int64_t num_blocks, int32_t block_size,
                             int32_t dtype, void *stream) {
    if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks < 0)
        return PA_ERR_INVALID_ARG;
    const int es = elem_size(dtype);
    if (es == 0) return PA_ERR_UNSUPPORTED;
    if (block_size != 16) return PA_ERR_UNSUPPORTED;
    if (head_dim % 16) return PA_ERR_UNSUPPORTED;
    if (num_tokens == 0) return PA_OK;
    if (!k || !v || !k_cache || !v_cache || !slot_mapping || !k_scale || !v_scale)
        return PA_ERR_INVALID_ARG;
    const int64_t row = (int64_t)num_kv_heads * head_dim;
    if (k_token_stride < row || v_token_stride < row) return PA_ERR_INVALID_ARG;
    // 8 source elements per thread, read with 16-byte loads
    if (!aligned16(k) || !aligned16(v) || (k_token_stride * es) % 16 ||
        (v_token_stride * es) % 16 || !aligned16(k_cache) || !aligned16(v_cache))
        return PA_ERR_INVALID_ARG;
    cudaError_t e = pa::reshape_and_cache_fp8(
        k, v, k_cache, v_cache, slot_mapping, num_tokens, num_kv_heads, head_dim,
        k_token_stride, v_token_stride, num_blocks * block_size, dtype, k_scale, v_scale,
        static_cast<cudaStream_t>(stream));
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"

namespace {

// Shared by the FP8 decode entry points: checks, parameters, launch of the
// persistent kernel (and, for partitions, the merge).
int decode_fp8_common(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const float *k_scale, const float *v_scale,
                      const int32_t *block_tables, const int32_t *seq_lens, int32_t num_seqs,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int64_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                      int64_t q_seq_stride, float scale, int32_t dtype, bool partial,
                      int32_t partition_size, int32_t max_seq_len, void *workspace,
                      size_t workspace_bytes, void *stream) {
    int rc = check_decode_args(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                               num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                               max_blocks_per_seq, q_seq_stride, scale, dtype);
    if (rc != PA_OK) return rc;
    if (partial && (partition_size <= 0 || partition_size % 16 || max_seq_len < 0))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (dtype != PA_BF16 && dtype != PA_F16) return PA_ERR_UNSUPPORTED;
    if (!k_scale || !v_scale) return PA_ERR_INVALID_ARG;
    if (!q_rows_aligned(q, q_seq_stride, dtype) || !aligned16(out)) return PA_ERR_INVALID_ARG;
    pa::DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.out = out; p.q = q; p.k_cache = k_cache; p.v_cache = v_cache;
    p.k_scale = k_scale; p.v_scale = v_scale;
    p.block_tables = block_tables; p.seq_lens = seq_lens;
    p.num_blocks = num_blocks; p.q_seq_stride = q_seq_stride;
    p.num_seqs = num_seqs; p.num_heads = num_heads; p.num_kv_heads = num_kv_heads;
    p.max_blocks = max_blocks_per_seq;
    p.scale_log2 = scale * pa::LOG2E;
    long long unit_bound = (long long)num_seqs * num_kv_heads;
    int P = 1;
    WorkspaceLayout w{};
    if (partial) {
        if (!workspace_layout(num_seqs, num_heads, head_dim, max_seq_len, partition_size, &w))
            return PA_ERR_INVALID_ARG;
        if (!workspace || workspace_bytes < w.total ||
            (reinterpret_cast<uintptr_t>(workspace) % kAlign))
            return PA_ERR_WORKSPACE;
        const int64_t P64 = ((int64_t)max_seq_len + partition_size - 1) / partition_size;
        if (P64 > INT32_MAX) return PA_ERR_UNSUPPORTED;
        P = (int)(P64 > 0 ? P64 : 1);
        unsigned char *ws = static_cast<unsigned char *>(workspace);
        p.part_o = reinterpret_cast<float *>(ws + w.o);
        p.part_m = reinterpret_cast<float *>(ws + w.m);
        p.part_l = reinterpret_cast<float *>(ws + w.l);
        p.partition_blocks = partition_size / 16;
        p.max_parts = P;
        p.max_seq_len = max_seq_len;
        unit_bound *= P;
    }
    if (pa::device_error_ptr(&p.err) != cudaSuccess) return PA_ERR_CUDA;
    if (!prepare_maps(p, PA_E4M3, head_dim)) return PA_ERR_CUDA;
    cudaStream_t st = static_cast<cudaStream_t>(stream);
    const int G = num_heads / num_kv_heads;
    const int cluster = partial ? 1 : PA_F8_CLUSTER;
    cudaError_t e = dtype == PA_BF16
                        ? pa::decode_fp8_bf16(p, head_dim, G, partial, unit_bound, cluster, st)
                        : pa::decode_fp8_f16(p, head_dim, G, partial, unit_bound, cluster, st);
    if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
    if (e != cudaSuccess) return PA_ERR_CUDA;
    if (!partial) return PA_OK;
    pa::MergeParams mp;
    std::memset(&mp, 0, sizeof mp);
    mp.out = out;
    mp.part_o = p.part_o; mp.part_m = p.part_m; mp.part_l = p.part_l;
    mp.seq_lens = seq_lens;
    mp.num_heads = num_heads; mp.head_dim = head_dim;
    mp.max_parts = P; mp.partition_size = partition_size;
    const int64_t cap = (int64_t)max_blocks_per_seq * 16;
    mp.seq_cap = (int)(max_seq_len < cap ? max_seq_len : cap);
    e = run_merge(mp, dtype, num_seqs, st);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // namespace

extern "C" {

int pa_decode_fp8(void *out, const void *q, const void *k_cache, const void *v_cache,
                  const float *k_scale, const float *v_scale, const int32_t *block_tables,
                  const int32_t *seq_lens, int32_t num_seqs, int32_t num_heads,
                  int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                  int32_t block_size, int32_t max_blocks_per_seq, int64_t q_seq_stride,
                  float scale, int32_t dtype, void *stream) {
    return decode_fp8_common(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                             seq_lens, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks,
                             block_size, max_blocks_per_seq, q_seq_stride, scale, dtype,
                             false, 0, 0, nullptr, 0, stream);
}

int pa_decode_partitioned_fp8(void *out, const void *q, const void *k_cache,
                              const void *v_cache, const float *k_scale,
                              const float *v_scale, const int32_t *block_tables,
                              const int32_t *seq_lens, int32_t num_seqs, int32_t num_heads,
                              int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
                              int32_t block_size, int32_t max_blocks_per_seq,
                              int64_t q_seq_stride, float scale, int32_t dtype,
                              int32_t partition_size, int32_t max_seq_len, void *workspace,
                              size_t workspace_bytes, void *stream) {
    return decode_fp8_common(out, q, k_cache, v_cache, k_scale, v_scale, block_tables,
                             seq_lens, num_seqs, num_heads, num_kv_heads, head_dim, num_blocks,
                             block_size, max_blocks_per_seq, q_seq_stride, scale, dtype, true,
                             partition_size, max_seq_len, workspace, workspace_bytes, stream);
}

}  // extern "C"

// ---- split-KV decode without any allocation ---------------------------------
//
// Some callers cannot call cudaMalloc at the point where they decode: code
// running while a CUDA graph is being captured on another stream, allocators
// that forbid allocations after warm-up, or plug-ins handed device buffers
// by a host program that owns all memory.  For them this entry point runs
// the split-KV decode with its partition workspace in a fixed array compiled
// into the library instead of a caller buffer.

// The built-in workspace.  Every GPU that loads the library holds these
// PA_NOALLOC_SCRATCH_BYTES until the process exits; every call on a device
// shares them.
static __device__ __align__(256) unsigned char noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];

namespace {

// Device address of noalloc_scratch on the current device, looked up once
// per device (with that device current) and cached.  In host code the
// array's name is only a host-side stand-in, never a device address.
cudaError_t noalloc_scratch_ptr(void **out) {
    static std::mutex mu;
    static void *cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    std::lock_guard<std::mutex> lock(mu);
    if (dev >= 0 && dev < 64 && cache[dev]) {
        *out = cache[dev];
        return cudaSuccess;
    }
    void *ptr = nullptr;
    e = cudaGetSymbolAddress(&ptr, noalloc_scratch);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) cache[dev] = ptr;
    *out = ptr;
    return cudaSuccess;
}

}  // namespace

extern "C" int pa_decode_partitioned_noalloc(
    void *out, const void *q, const void *k_cache, const void *v_cache,
    const int32_t *block_tables, const int32_t *seq_lens, int32_t num_seqs,
    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
    int32_t block_size, int32_t max_blocks_per_seq, int64_t q_seq_stride, float scale,
    int32_t dtype, int32_t partition_size, int32_t max_seq_len, void *stream) {
    // The same checks, in the same order, as pa_decode_partitioned, so that
    // both calls give the same status for the same bad input.
    int rc = check_decode_args(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                               num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                               max_blocks_per_seq, q_seq_stride, scale, dtype);
    if (rc != PA_OK) return rc;
    if (partition_size <= 0 || partition_size % 16 || max_seq_len < 0)
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    const size_t need = pa_decode_partitioned_workspace_size(num_seqs, num_heads, head_dim,
                                                             max_seq_len, partition_size);
    if (need == 0) return PA_ERR_INVALID_ARG;
    if (need > (size_t)PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_WORKSPACE;
    void *scratch = nullptr;
    if (noalloc_scratch_ptr(&scratch) != cudaSuccess) return PA_ERR_CUDA;
    return pa_decode_partitioned(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                                 num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                                 max_blocks_per_seq, q_seq_stride, scale, dtype,
                                 partition_size, max_seq_len, scratch,
                                 (size_t)PA_NOALLOC_SCRATCH_BYTES, stream);
}

extern "C" {

int pa_device_error(uint32_t *flags, int clear) {
    if (!flags) return PA_ERR_INVALID_ARG;
    unsigned int f = 0;
    cudaError_t e = pa::read_device_error(&f, clear != 0);
    *flags = f;
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"

// ---- cascade decode over a shared prefix -----------------------------------
//
// Sequences whose block tables begin with the same physical blocks (a shared
// prompt, prefix caching) attend to those blocks once: the prefix's keys and
// values are read once per KV head and multiplied against the query heads
// of every sequence at once (128 (sequence, head) rows per tensor-core tile),
// then each sequence's own blocks are decoded as split-KV partitions, and the
// two are merged by log-sum-exp.

namespace {

// Prefix chunks of the cascade: at least 32 blocks (512 keys, eight steps of
// the tensor-core kernel) each, at most 16 chunks; the sequences' own blocks
// in partitions of 512 tokens.  (On the 2048-token shared prefix, chunks of
// 8, 16, 32, 64 and 128 blocks measured 74.8, 66.6, 62.5, 68.6 and 76.8 us
// per call: shorter items pay their start-up and write more partials, longer
// ones leave SMs idle.)
constexpr int32_t kCascadeSuffixPart = 512;

int32_t cascade_chunk_blocks(int32_t num_prefix_blocks) {
    int32_t c = (num_prefix_blocks + 15) / 16;
    c = (c + 3) / 4 * 4;
    return c < 32 ? 32 : c;
}

// Partitions of the cascade workspace: the prefix chunks, then the sequence's.
bool cascade_parts(int32_t num_prefix_blocks, int32_t max_blocks_per_seq, int32_t *nch,
                   int32_t *parts) {
    if (num_prefix_blocks <= 0 || max_blocks_per_seq < 0) return false;
    const int32_t cb = cascade_chunk_blocks(num_prefix_blocks);
    *nch = (num_prefix_blocks + cb - 1) / cb;
    const int64_t ps = ((int64_t)max_blocks_per_seq * 16 + kCascadeSuffixPart - 1) / kCascadeSuffixPart;
    const int64_t total = *nch + (ps > 0 ? ps : 1);
    if (total * kCascadeSuffixPart > INT32_MAX) return false;
    *parts = (int32_t)total;
    return true;
}

}  // namespace

extern "C" {

size_t pa_decode_cascade_workspace_size(int32_t num_seqs, int32_t num_heads, int32_t head_dim,
                                        int32_t num_prefix_blocks, int32_t max_blocks_per_seq) {
    int32_t nch = 0, P = 0;
    if (!cascade_parts(num_prefix_blocks, max_blocks_per_seq, &nch, &P)) return 0;
    WorkspaceLayout w;
    if (!workspace_layout(num_seqs, num_heads, head_dim, P * kCascadeSuffixPart,
                          kCascadeSuffixPart, &w))
        return 0;
    return w.total;
}

int pa_decode_cascade(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *prefix_blocks, int32_t num_prefix_blocks,
                      const int32_t *block_tables, const int32_t *seq_lens, int32_t num_seqs,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int64_t num_blocks, int32_t block_size, int32_t max_blocks_per_seq,
                      int64_t q_seq_stride, float scale, int32_t dtype, void *workspace,
                      size_t workspace_bytes, void *stream) {
    int rc = check_decode_args(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                               num_heads, num_kv_heads, head_dim, num_blocks, block_size,
                               max_blocks_per_seq, q_seq_stride, scale, dtype);
    if (rc != PA_OK) return rc;
    if (num_prefix_blocks < 0 || (num_prefix_blocks > 0 && !prefix_blocks))
        return PA_ERR_INVALID_ARG;
    if (num_seqs == 0) return PA_OK;
    if (num_prefix_blocks == 0)                              // nothing shared: plain decode
        return pa_decode(out, q, k_cache, v_cache, block_tables, seq_lens, num_seqs, num_heads,
                         num_kv_heads, head_dim, num_blocks, block_size, max_blocks_per_seq,
                         q_seq_stride, scale, dtype, stream);
    if (dtype == PA_F32) return PA_ERR_UNSUPPORTED;         // the prefix runs on 16-bit MMAs
    if (!q_rows_aligned(q, q_seq_stride, dtype) || !aligned16(out)) return PA_ERR_INVALID_ARG;
    int32_t nch = 0, P = 0;
    if (!cascade_parts(num_prefix_blocks, max_blocks_per_seq, &nch, &P)) return PA_ERR_UNSUPPORTED;
    // the prefix kernel numbers its items (chunk, KV head, 128-row group) in an int
    const int G = num_heads / num_kv_heads;
    const int64_t row_groups = ((int64_t)num_seqs * G + pa::PREFILL_TC_ROWS - 1) / pa::PREFILL_TC_ROWS;
    if ((int64_t)nch * num_kv_heads * row_groups > INT32_MAX) return PA_ERR_UNSUPPORTED;
    WorkspaceLayout w;
    if (!workspace_layout(num_seqs, num_heads, head_dim, P * kCascadeSuffixPart,
                          kCascadeSuffixPart, &w))
        return PA_ERR_INVALID_ARG;
    if (!workspace || workspace_bytes < w.total ||
        (reinterpret_cast<uintptr_t>(workspace) % kAlign))
        return PA_ERR_WORKSPACE;
    unsigned char *ws = static_cast<unsigned char *>(workspace);
    cudaStream_t st = static_cast<cudaStream_t>(stream);

    pa::DecodeParams p;
    std::memset(&p, 0, sizeof p);
    p.out = out; p.q = q; p.k_cache = k_cache; p.v_cache = v_cache;
    p.block_tables = block_tables; p.seq_lens = seq_lens;
    p.part_o = reinterpret_cast<float *>(ws + w.o);
    p.part_m = reinterpret_cast<float *>(ws + w.m);
    p.part_l = reinterpret_cast<float *>(ws + w.l);
    p.num_blocks = num_blocks; p.q_seq_stride = q_seq_stride;
    p.num_seqs = num_seqs; p.num_heads = num_heads; p.num_kv_heads = num_kv_heads;
    p.max_blocks = max_blocks_per_seq;
    p.max_parts = P;
    p.scale_log2 = scale * pa::LOG2E;
    if (pa::device_error_ptr(&p.err) != cudaSuccess) return PA_ERR_CUDA;
    if (!prepare_maps(p, dtype, head_dim)) return PA_ERR_CUDA;

    // 1. the shared prefix: partitions 0 .. nch-1, on the tcgen05 kernel
    {
        pa::DecodeParams pp = p;
        pp.prefix_blocks = prefix_blocks;
        pp.prefix_nblocks = num_prefix_blocks;
        pp.prefix_chunk_blocks = cascade_chunk_blocks(num_prefix_blocks);
        CUtensorMap tmap_q;
        if (!encode_q_map(&tmap_q, q, num_seqs, num_heads, head_dim, q_seq_stride, G, dtype))
            return PA_ERR_CUDA;
        cudaError_t e = dtype == PA_BF16 ? pa::prefill_tc_bf16(pp, tmap_q, head_dim, G, 1, st)
                                         : pa::prefill_tc_f16(pp, tmap_q, head_dim, G, 1, st);
        if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    // 2. each sequence's own blocks: split-KV partitions nch .. P-1
    {
        pa::DecodeParams ps = p;
        ps.part_o = p.part_o + (size_t)nch * head_dim;
        ps.part_m = p.part_m + nch;
        ps.part_l = p.part_l + nch;
        ps.partition_blocks = kCascadeSuffixPart / 16;
        ps.max_seq_len = max_blocks_per_seq * 16;
        cudaError_t e = run_persistent(ps, dtype, head_dim, G, true,
                                       (long long)num_seqs * num_kv_heads * (P - nch), st);
        if (e == cudaErrorNotSupported) return PA_ERR_UNSUPPORTED;
        if (e != cudaSuccess) return PA_ERR_CUDA;
    }
    // 3. log-sum-exp merge of the prefix chunks and the sequence's partitions
    pa::MergeParams mp;
    std::memset(&mp, 0, sizeof mp);
    mp.out = out;
    mp.part_o = p.part_o; mp.part_m = p.part_m; mp.part_l = p.part_l;
    mp.seq_lens = seq_lens;
    mp.num_heads = num_heads; mp.head_dim = head_dim;
    mp.max_parts = P; mp.partition_size = kCascadeSuffixPart;
    mp.seq_cap = max_blocks_per_seq * 16;
    mp.prefix_parts = nch;
    cudaError_t e = run_merge(mp, dtype, num_seqs, st);
    return e == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

}  // extern "C"
