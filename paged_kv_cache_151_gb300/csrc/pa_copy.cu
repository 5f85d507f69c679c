// pa_copy.cu -- block copies for copy-on-write.
//
// "vLLM: Architecture, PagedAttention & Internals", *Copy-on-write for shared
// blocks*: when a sequence must write into a block that another still reads
// (refcount > 1), the block manager hands it a fresh block and the GPU copies
// the shared block's contents there before the write.  The copies of one step
// come as a list of (src, dst) pairs and apply to every cache (K and V of
// every layer), so one launch serves the whole step.
//
// Each work item is a 16 KiB piece of one block of one cache for one pair:
// 256 threads x four 16-byte loads in flight each, then the four stores.
// Loads bypass L1 and stores are marked streaming, so the copy passes
// through L2 without displacing the blocks decode is about to read.
#include "pa_common.cuh"
#include "pa_internal.h"

namespace pa {

constexpr int COPY_THREADS = 256;
constexpr int COPY_VEC = 4;                                   // uint4 per thread per item
constexpr int64_t COPY_PIECE = (int64_t)COPY_THREADS * COPY_VEC * 16;   // 16 KiB

__device__ __forceinline__ uint4 ld_stream(const uint4 *p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "l"(p));
    return v;
}

__device__ __forceinline__ void st_stream(uint4 *p, uint4 v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};"
                 :: "l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w) : "memory");
}

__global__ void __launch_bounds__(COPY_THREADS)
copy_blocks_kernel(const __grid_constant__ CopyParams p) {
    const int64_t pieces = (p.block_bytes + COPY_PIECE - 1) / COPY_PIECE;
    const int64_t per_pair = pieces * p.num_caches;
    const int64_t items = p.num_pairs * per_pair;
    for (int64_t it = blockIdx.x; it < items; it += gridDim.x) {
        const int64_t pair = it / per_pair;
        const int64_t rem = it - pair * per_pair;
        const int c = (int)(rem / pieces);
        const int64_t piece = rem - (int64_t)c * pieces;
        const int64_t src = p.mapping[2 * pair], dst = p.mapping[2 * pair + 1];
        if (src < 0 || src >= p.num_blocks || dst < 0 || dst >= p.num_blocks) {
            if (c == 0 && piece == 0 && threadIdx.x == 0) set_error(p.err, ERR_BLOCK_ID);
            continue;
        }
        const unsigned char *s = p.caches[c] + src * p.block_bytes + piece * COPY_PIECE;
        unsigned char *d = p.caches[c] + dst * p.block_bytes + piece * COPY_PIECE;
        const int64_t n = min(COPY_PIECE, p.block_bytes - piece * COPY_PIECE) / 16;
        uint4 v[COPY_VEC];
#pragma unroll
        for (int u = 0; u < COPY_VEC; ++u) {
            const int64_t i = threadIdx.x + (int64_t)u * COPY_THREADS;
            if (i < n) v[u] = ld_stream(reinterpret_cast<const uint4 *>(s) + i);
        }
#pragma unroll
        for (int u = 0; u < COPY_VEC; ++u) {
            const int64_t i = threadIdx.x + (int64_t)u * COPY_THREADS;
            if (i < n) st_stream(reinterpret_cast<uint4 *>(d) + i, v[u]);
        }
    }
}

cudaError_t copy_blocks(const CopyParams &p, cudaStream_t st) {
    const int64_t pieces = (p.block_bytes + COPY_PIECE - 1) / COPY_PIECE;
    const int64_t items = p.num_pairs * p.num_caches * pieces;
    if (items == 0) return cudaSuccess;
    int sms = sm_count_of_current_device();
    int64_t grid = (int64_t)(sms > 0 ? sms : 152) * 8;        // 8 blocks of 256 per SM
    if (grid > items) grid = items;
    copy_blocks_kernel<<<(unsigned)grid, COPY_THREADS, 0, st>>>(p);
    return cudaGetLastError();
}

}  // namespace pa
