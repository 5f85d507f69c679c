// pa_cache.cu -- the cache write (reshape_and_cache) and the device error word.
//
// "vLLM: Architecture, PagedAttention & Internals", *The forward step in
// detail*: for each token being written the runner computes the physical slot
// (block * block_size + offset); inside the attention layer the fresh K and V
// are scattered into the cache at those slots before attention reads it.
// This is a pure copy: every (token, KV head) row of head_dim elements moves
// bit for bit, in 16-byte pieces when the addresses allow it.
#include "pa_common.cuh"
#include "pa_fp8.cuh"
#include "pa_internal.h"

namespace pa {

__device__ unsigned int g_device_error = 0;

// Address of the error word on the current device (looked up once per device).
cudaError_t device_error_ptr(unsigned int **out) {
    static unsigned int *cache[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64 && cache[dev]) {
        *out = cache[dev];
        return cudaSuccess;
    }
    void *p = nullptr;
    e = cudaGetSymbolAddress(&p, g_device_error);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) cache[dev] = static_cast<unsigned int *>(p);
    *out = static_cast<unsigned int *>(p);
    return cudaSuccess;
}

// One thread per U-sized piece of one (token, KV head) row, for K and V.
template <typename U>
__global__ void __launch_bounds__(256)
reshape_and_cache_kernel(const unsigned char *__restrict__ k,
                         const unsigned char *__restrict__ v,
                         unsigned char *__restrict__ k_cache,
                         unsigned char *__restrict__ v_cache,
                         const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                         int num_kv_heads, int row_bytes, int64_t k_tok_stride_bytes,
                         int64_t v_tok_stride_bytes, int64_t num_slots,
                         unsigned int *err) {
    launch_dependents();      // a decode launched next may set up meanwhile
    const int per_row = row_bytes / (int)sizeof(U);
    const int64_t per_tok = (int64_t)num_kv_heads * per_row;
    const int64_t total = num_tokens * per_tok;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_tok;
        const int64_t rem = i - t * per_tok;
        const int jh = (int)(rem / per_row);
        const int piece = (int)(rem - (int64_t)jh * per_row);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;                        // padding token
        if (slot >= num_slots) {
            if (jh == 0 && piece == 0) set_error(err, ERR_SLOT);
            continue;
        }
        const int64_t blk = slot >> 4, row = slot & 15;  // block_size 16
        const int64_t dst = ((blk * num_kv_heads + jh) * 16 + row) * row_bytes +
                            (int64_t)piece * sizeof(U);
        const int64_t sk = t * k_tok_stride_bytes + (int64_t)jh * row_bytes +
                           (int64_t)piece * sizeof(U);
        const int64_t sv = t * v_tok_stride_bytes + (int64_t)jh * row_bytes +
                           (int64_t)piece * sizeof(U);
        *reinterpret_cast<U *>(k_cache + dst) = *reinterpret_cast<const U *>(k + sk);
        *reinterpret_cast<U *>(v_cache + dst) = *reinterpret_cast<const U *>(v + sv);
    }
}

static int largest_piece(uintptr_t a) {
    if ((a & 15) == 0) return 16;
    if ((a & 7) == 0) return 8;
    if ((a & 3) == 0) return 4;
    return 2;
}

cudaError_t reshape_and_cache(const void *k, const void *v, void *k_cache, void *v_cache,
                              const int64_t *slot_mapping, int64_t num_tokens,
                              int num_kv_heads, int row_bytes, int64_t k_tok_stride_bytes,
                              int64_t v_tok_stride_bytes, int64_t num_slots,
                              cudaStream_t st) {
    if (num_tokens == 0) return cudaSuccess;
    unsigned int *err = nullptr;
    cudaError_t ee = device_error_ptr(&err);
    if (ee != cudaSuccess) return ee;
    // the widest copy unit every address and stride allows
    const uintptr_t bits = (uintptr_t)k | (uintptr_t)v | (uintptr_t)k_cache |
                           (uintptr_t)v_cache | (uintptr_t)row_bytes |
                           (uintptr_t)k_tok_stride_bytes | (uintptr_t)v_tok_stride_bytes;
    const int unit = largest_piece(bits);
    const int64_t total = num_tokens * num_kv_heads * (row_bytes / unit);
    int sms = sm_count_of_current_device();
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 16;
    if (blocks > cap) blocks = cap;
    const auto *kb = static_cast<const unsigned char *>(k);
    const auto *vb = static_cast<const unsigned char *>(v);
    auto *kc = static_cast<unsigned char *>(k_cache);
    auto *vc = static_cast<unsigned char *>(v_cache);
#define PA_RC(U)                                                                     \
    prefer_shared_carveout<reshape_and_cache_kernel<U>>();                            \
    reshape_and_cache_kernel<U><<<(unsigned)blocks, 256, 0, st>>>(                    \
        kb, vb, kc, vc, slot_mapping, num_tokens, num_kv_heads, row_bytes,            \
        k_tok_stride_bytes, v_tok_stride_bytes, num_slots, err)
    switch (unit) {
        case 16: PA_RC(uint4); break;
        case 8: PA_RC(uint2); break;
        case 4: PA_RC(uint32_t); break;
        default: PA_RC(uint16_t); break;
    }
#undef PA_RC
    return cudaGetLastError();
}

// ---- FP8 (E4M3) cache write ---------------------------------------------
//
// The same scatter into an E4M3 cache: element d of KV head j of a new row
// is stored as E4M3(x / scale_j), the quotient rounded once to binary32
// (IEEE division) and then to E4M3 by the conversion instruction (nearest,
// ties to even, saturating to +-448, NaN to NaN).  One thread per 8 elements
// of one (token, KV head) row, for K and V.

template <typename TS>
__device__ __forceinline__ void load8(const TS *src, float *x) {
    if constexpr (sizeof(TS) == 2) {
        Elem<TS>::to_f32(*reinterpret_cast<const uint4 *>(src), x);
    } else {
        Elem<float>::to_f32(*reinterpret_cast<const uint4 *>(src), x);
        Elem<float>::to_f32(*reinterpret_cast<const uint4 *>(src + 4), x + 4);
    }
}

template <typename TS>
__device__ __forceinline__ uint2 quantise8(const TS *src, float scale) {
    float x[8];
    load8<TS>(src, x);
    uint2 r;
    r.x = e4m3x2_from_f32(__fdiv_rn(x[0], scale), __fdiv_rn(x[1], scale)) |
          (e4m3x2_from_f32(__fdiv_rn(x[2], scale), __fdiv_rn(x[3], scale)) << 16);
    r.y = e4m3x2_from_f32(__fdiv_rn(x[4], scale), __fdiv_rn(x[5], scale)) |
          (e4m3x2_from_f32(__fdiv_rn(x[6], scale), __fdiv_rn(x[7], scale)) << 16);
    return r;
}

template <typename TS>
__global__ void __launch_bounds__(256)
reshape_and_cache_fp8_kernel(const TS *__restrict__ k, const TS *__restrict__ v,
                             unsigned char *__restrict__ k_cache,
                             unsigned char *__restrict__ v_cache,
                             const int64_t *__restrict__ slot_mapping, int64_t num_tokens,
                             int num_kv_heads, int head_dim, int64_t k_tok_stride,
                             int64_t v_tok_stride, int64_t num_slots,
                             const float *__restrict__ k_scale,
                             const float *__restrict__ v_scale, unsigned int *err) {
    launch_dependents();      // a decode launched next may set up meanwhile
    const int per_row = head_dim / 8;
    const int64_t per_tok = (int64_t)num_kv_heads * per_row;
    const int64_t total = num_tokens * per_tok;
    for (int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x; i < total;
         i += (int64_t)gridDim.x * blockDim.x) {
        const int64_t t = i / per_tok;
        const int64_t rem = i - t * per_tok;
        const int jh = (int)(rem / per_row);
        const int piece = (int)(rem - (int64_t)jh * per_row);
        const int64_t slot = slot_mapping[t];
        if (slot < 0) continue;                        // padding token
        if (slot >= num_slots) {
            if (jh == 0 && piece == 0) set_error(err, ERR_SLOT);
            continue;
        }
        const int64_t blk = slot >> 4, row = slot & 15;  // block_size 16
        const int64_t dst = ((blk * num_kv_heads + jh) * 16 + row) * head_dim + piece * 8;
        const int64_t e = (int64_t)jh * head_dim + piece * 8;
        *reinterpret_cast<uint2 *>(k_cache + dst) =
            quantise8<TS>(k + t * k_tok_stride + e, __ldg(k_scale + jh));
        *reinterpret_cast<uint2 *>(v_cache + dst) =
            quantise8<TS>(v + t * v_tok_stride + e, __ldg(v_scale + jh));
    }
}

cudaError_t reshape_and_cache_fp8(const void *k, const void *v, void *k_cache, void *v_cache,
                                  const int64_t *slot_mapping, int64_t num_tokens,
                                  int num_kv_heads, int head_dim, int64_t k_tok_stride,
                                  int64_t v_tok_stride, int64_t num_slots, int src_dtype,
                                  const float *k_scale, const float *v_scale,
                                  cudaStream_t st) {
    if (num_tokens == 0) return cudaSuccess;
    unsigned int *err = nullptr;
    cudaError_t ee = device_error_ptr(&err);
    if (ee != cudaSuccess) return ee;
    const int64_t total = num_tokens * num_kv_heads * (head_dim / 8);
    int sms = sm_count_of_current_device();
    int64_t blocks = (total + 255) / 256;
    const int64_t cap = (int64_t)(sms > 0 ? sms : 152) * 16;
    if (blocks > cap) blocks = cap;
    auto *kc = static_cast<unsigned char *>(k_cache);
    auto *vc = static_cast<unsigned char *>(v_cache);
#define PA_RC8(TS)                                                                       \
    prefer_shared_carveout<reshape_and_cache_fp8_kernel<TS>>();                           \
    reshape_and_cache_fp8_kernel<TS><<<(unsigned)blocks, 256, 0, st>>>(                   \
        static_cast<const TS *>(k), static_cast<const TS *>(v), kc, vc, slot_mapping,      \
        num_tokens, num_kv_heads, head_dim, k_tok_stride, v_tok_stride, num_slots, k_scale, \
        v_scale, err)
    switch (src_dtype) {
        case 0: PA_RC8(float); break;
        case 1: PA_RC8(__nv_bfloat16); break;
        default: PA_RC8(__half); break;
    }
#undef PA_RC8
    return cudaGetLastError();
}

cudaError_t read_device_error(unsigned int *flags, bool clear) {
    cudaError_t e = cudaDeviceSynchronize();
    if (e != cudaSuccess) return e;
    e = cudaMemcpyFromSymbol(flags, g_device_error, sizeof(unsigned int));
    if (e != cudaSuccess) return e;
    if (clear) {
        const unsigned int zero = 0;
        e = cudaMemcpyToSymbol(g_device_error, &zero, sizeof(unsigned int));
    }
    return e;
}

}  // namespace pa
