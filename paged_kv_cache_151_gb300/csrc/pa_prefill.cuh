// pa_prefill.cuh -- multi-token queries with many rows per sequence (a chunk
// of a long prompt): the rows of one (sequence, KV head) are cut into groups
// of 16*NWC, one group per thread block, and the block's NWC warps -- 16
// rows each -- consume ONE ring of K/V tiles that a producer warp fills with
// tensor-map copies.  Every tile read from L2 or HBM thus serves 16*NWC
// query rows instead of 16.
//
// "vLLM: Architecture, PagedAttention & Internals", *Prefill, decode, and
// chunked prefill*: one forward pass carries a slice of a long prompt next
// to one-token decodes.  Row r of sequence s's slice (token i = r / G, head
// r % G of the KV head's group) attends over positions 0 .. L - n + i of
// the paged cache, like the rows of pa_decode_multi's other path; a block
// handles the rows of one group from their first block to the block of the
// group's last visible position, and each warp masks its rows' limits.
//
// Work items: (row group, sequence, KV head) of the sequences whose runs have
// at least p.mq_split_rows rows (the others are the persistent kernel's).
// Every block lists them in the same order -- sequences by length, longest
// first (up to 256 sequences; in index order beyond), and within a sequence
// the last row groups (which see the most keys) first -- and takes item
// blockIdx.x, blockIdx.x + gridDim.x, ...: with one item per block the
// hardware starts the costliest items first and gives the cheap ones to the
// blocks that finish early.
#pragma once

#include <atomic>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_internal.h"
#include "pa_math.cuh"
#include "pa_mma.cuh"

namespace pa {

template <typename T, int D, int NWC, int S>
struct PrefillLayout {
    static constexpr int TILE = 16 * D * (int)sizeof(T);
    static constexpr size_t STAGES = (size_t)S * 2 * TILE;
    static constexpr size_t OFF_BARS = STAGES;                       // full[S], empty[S]
    static constexpr size_t OFF_OK = OFF_BARS + (size_t)2 * S * 8;    // int valid[S]
    static constexpr size_t BYTES = (OFF_OK + (size_t)S * 4 + 15) / 16 * 16 + 1024;
    static_assert(STAGES % 1024 == 0, "1024-byte aligned tiles");
};

#ifndef PA_PREFILL_BLOCKS_PER_SM
#define PA_PREFILL_BLOCKS_PER_SM 3
#endif

// The schedule of the prefill work items, in shared memory: up to 256
// sequences are sorted by length, longest first; beyond, index order.
struct PrefillSched {
    uint32_t keys[256];      // sort input
    uint32_t order[256];     // sequences, longest first (low 16 bits)
    int first[257];          // items before sorted position i
    int groups[256];         // row groups of sequence s
};

// Row groups (of ROWS rows) of sequence s if its run goes to a prefill
// kernel, else 0 (a run with a bad range is flagged, by block 0, and
// skipped).  Reads only query_start and seq_lens, which the kernel before
// this one must not write.
template <int G, int ROWS>
__device__ __forceinline__ int prefill_groups_of(const DecodeParams &p, int groups, int s) {
    const int q0 = p.query_start[s], q1 = p.query_start[s + 1];
    const int nq = q1 - q0, L = p.seq_lens[s];
    // sequences with fewer rows are the persistent kernel's, which flags bad ranges
    if (nq < 0 || nq * G < p.mq_split_rows) return 0;
    if (q0 < 0 || q1 > p.num_q_rows || nq > p.max_query_len || L < nq || L > p.max_blocks * 16) {
        if (blockIdx.x == 0) set_error(p.err, ERR_SEQ_LEN);
        return 0;
    }
    return min(groups, (nq * G + ROWS - 1) / ROWS);
}

// All threads of the block: build the schedule; returns the number of items.
template <int G, int ROWS>
__device__ int prefill_schedule(const DecodeParams &p, int groups, PrefillSched &sc) {
    const int B = p.num_seqs, Hkv = p.num_kv_heads;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (B > 256) {
        int sum = 0;
        for (int s = lane; s < B; s += 32) sum += prefill_groups_of<G, ROWS>(p, groups, s) * Hkv;
        return __reduce_add_sync(0xffffffffu, sum);
    }
    if (warp == 0) {
        for (int s = lane; s < 256; s += 32) {
            uint32_t key = 0xffffffffu;
            const int gs = s < B ? prefill_groups_of<G, ROWS>(p, groups, s) : 0;
            if (s < B) sc.groups[s] = gs;
            if (gs > 0) {
                const int nb = min(0xffff, (p.seq_lens[s] + 15) >> 4);
                key = ((uint32_t)(0xffff - nb) << 16) | (uint32_t)s;
            }
            sc.keys[s] = key;
        }
        __syncwarp();
        warp_bitonic_sort<8>(sc.keys, sc.order);
        __syncwarp();
        // items before each sorted position: lane holds positions 8*lane .. 8*lane+7
        int c[8], sum = 0;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            const uint32_t k = sc.order[8 * lane + e];
            c[e] = k == 0xffffffffu ? 0 : sc.groups[k & 0xffffu] * Hkv;
            sum += c[e];
        }
        int x = sum;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int y = __shfl_up_sync(0xffffffffu, x, o);
            if (lane >= o) x += y;
        }
        int run = x - sum;
#pragma unroll
        for (int e = 0; e < 8; ++e) {
            sc.first[8 * lane + e] = run;
            run += c[e];
        }
        if (lane == 31) sc.first[256] = run;
    }
    __syncthreads();
    return sc.first[256];
}

// Item r -> (sequence s, KV head j, row group grp), last row groups first
// within a sequence.  All lanes of the calling warp, convergent.
template <int G, int ROWS>
__device__ void prefill_item(const DecodeParams &p, int groups, const PrefillSched &sc, int r,
                             int &s, int &j, int &grp) {
    const int B = p.num_seqs, Hkv = p.num_kv_heads, lane = threadIdx.x & 31;
    int local;
    if (B <= 256) {
        int lo = 0, hi = 255;                      // last position with first <= r
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (sc.first[mid] <= r) lo = mid; else hi = mid - 1;
        }
        s = (int)(sc.order[lo] & 0xffffu);
        local = r - sc.first[lo];
    } else {
        // index order: the warp walks the sequences 32 at a time
        int base = 0;
        s = -1;
        local = 0;
        for (int s0 = 0; s0 < B && s < 0; s0 += 32) {
            const int n = (s0 + lane < B) ? prefill_groups_of<G, ROWS>(p, groups, s0 + lane) * Hkv : 0;
            int x = n;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int y = __shfl_up_sync(0xffffffffu, x, o);
                if (lane >= o) x += y;
            }
            const uint32_t hit = __ballot_sync(0xffffffffu, n > 0 && base + x - n <= r && r < base + x);
            if (hit) {
                const int l = __ffs(hit) - 1;
                s = s0 + l;
                local = r - (base + __shfl_sync(0xffffffffu, x - n, l));
            }
            base += __shfl_sync(0xffffffffu, x, 31);
        }
    }
    const int q0 = p.query_start[s], nq = p.query_start[s + 1] - q0;
    const int gs = min(groups, (nq * G + ROWS - 1) / ROWS);
    j = local % Hkv;
    grp = gs - 1 - local / Hkv;                    // last row groups first
}

template <typename T, int D, int G, int NWC, int S>
__global__ void __launch_bounds__((NWC + 1) * 32, PA_PREFILL_BLOCKS_PER_SM)
prefill_kernel(const __grid_constant__ DecodeParams p, int groups) {
    static_assert(sizeof(T) == 2, "16-bit caches");
    using W = WarpAttnTC16<T, D>;
    using Lay = PrefillLayout<T, D, NWC, S>;
    constexpr int TILE = Lay::TILE;
    constexpr int ROWS = 16 * NWC;                 // query rows of one work item

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::OFF_BARS);
    uint64_t *empty = full + S;
    int *valid = reinterpret_cast<int *>(smem + Lay::OFF_OK);
    __shared__ int abort_flag;                     // a wait timed out: everyone stops
    __shared__ PrefillSched sched;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hkv = p.num_kv_heads, H = p.num_heads;

    if (tid == 0) {
        prefetch_tensormap(&p.tmap_k);
        prefetch_tensormap(&p.tmap_v);
        for (int i = 0; i < S; ++i) {
            mbar_init(&full[i], 1);
            mbar_init(&empty[i], NWC);
        }
        fence_mbar_init();
        abort_flag = 0;
    }
    __syncthreads();
    const int total = prefill_schedule<G, ROWS>(p, groups, sched);

    // the caches (and q, out) only after the kernel before this one is done
    grid_dependency_wait();

    // The ring of stages runs on across the items of a block, so the producer
    // streams the next item while the consumers finish one.
    long long kglob = 0;                           // blocks through the ring so far
    const uint64_t pol = policy_evict_last();      // the sequence's other groups reread them
    W wa;
    wa.init(lane);
    for (int x = blockIdx.x; x < total; x += gridDim.x) {
        if (*(volatile int *)&abort_flag) break;
        int s, j, grp;
        prefill_item<G, ROWS>(p, groups, sched, x, s, j, grp);
        const int q0 = p.query_start[s], q1 = p.query_start[s + 1];
        const int nq = q1 - q0;
        const int L = p.seq_lens[s];
        const int last_row = min(grp * ROWS + ROWS, nq * G) - 1;
        const int nb = (L - nq + last_row / G) / 16 + 1;   // through the group's last position

        if (warp == NWC) {
            // ---- producer: one lane streams the item's blocks through the ring
            if (lane == 0) {
                const int32_t *tab = p.block_tables + (long long)s * p.max_blocks;
                for (int k = 0; k < nb; ++k) {
                    const long long kk = kglob + k;
                    const int st = (int)(kk % S);
                    if (kk >= S &&
                        !mbar_wait_bounded(&empty[st], (uint32_t)(((kk / S) - 1) & 1), p.err)) {
                        abort_flag = 1;
                        kglob += k;                // what was issued
                        goto producer_done;
                    }
                    const int pb = tab[k];
                    if (pb < 0 || (long long)pb >= p.num_blocks) {
                        set_error(p.err, ERR_BLOCK_ID);
                        valid[st] = 0;
                        mbar_arrive(&full[st]);
                        continue;
                    }
                    valid[st] = 1;
                    unsigned char *dst = smem + (size_t)st * 2 * TILE;
                    const int z = pb * Hkv + j;
                    mbar_arrive_expect_tx(&full[st], 2 * TILE);
#pragma unroll
                    for (int h = 0; h < D / 64; ++h) {
                        tma_load_3d(dst + h * 2048, &p.tmap_k, h * 64, 0, z, &full[st], pol);
                        tma_load_3d(dst + TILE + h * 2048, &p.tmap_v, h * 64, 0, z, &full[st], pol);
                    }
                }
            }
        } else {
            // ---- consumers: rows g and g+8 of this warp's 16-row tile
            const int r_lo = grp * ROWS + warp * 16 + (lane >> 2), r_hi = r_lo + 8;
            auto qrow = [&](int r) -> const T * {
                if (r >= nq * G) return nullptr;
                return reinterpret_cast<const T *>(p.q) + (long long)(q0 + r / G) * p.q_seq_stride +
                       (long long)(j * G + r % G) * D;
            };
            wa.reset();
            wa.load_q(qrow(r_lo), qrow(r_hi), L - nq + r_lo / G, L - nq + r_hi / G);
            bool ok = true;
            for (int k = 0; k < nb; ++k) {
                const long long kk = kglob + k;
                const int st = (int)(kk % S);
                const bool got = mbar_wait_bounded(&full[st], (uint32_t)((kk / S) & 1), p.err);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                if (valid[st]) {
                    const unsigned char *kt = smem + (size_t)st * 2 * TILE;
                    wa.block(smem_u32(kt), smem_u32(kt + TILE), 16 * k, p.scale_log2,
                             min(16, L - 16 * k));
                }
                __syncwarp();
                if (lane == 0) mbar_arrive(&empty[st]);
            }
            if (!ok) {
                if (lane == 0) abort_flag = 1;
                break;
            }
            wa.finish();
            wa.for_each_result([&](int row, int d, float v0, float v1, bool, float, float) {
                const int rr = grp * ROWS + warp * 16 + row;
                T *o = reinterpret_cast<T *>(p.out) +
                       ((long long)(q0 + rr / G) * H + j * G + rr % G) * D + d;
                store_pair<T>(o, v0, v1);
            });
        }
        kglob += nb;
    }
    if (warp == NWC && lane == 0) {
    producer_done:
        // no copy may still be landing when the block exits: wait (bounded) for
        // the last stages issued
        for (long long i = (kglob > S ? kglob - S : 0); i < kglob; ++i)
            mbar_wait_bounded(&full[i % S], (uint32_t)((i / S) & 1), p.err);
    }
    __syncthreads();
}

// Consumer warps and ring stages of the prefill path (16 rows per warp).
constexpr int PREFILL_NWC = PREFILL_GROUP_ROWS / 16;
template <typename T, int D>
__host__ __device__ constexpr int prefill_stages() {
    return (16 * 1024 * 4) / (2 * 16 * D * (int)sizeof(T));   // 64 KiB of K/V in flight
}

template <typename T, int D, int G>
cudaError_t launch_prefill(const DecodeParams &p, int groups, cudaStream_t st) {
    constexpr int S = prefill_stages<T, D>();
    using Lay = PrefillLayout<T, D, PREFILL_NWC, S>;
    constexpr size_t smem = Lay::BYTES;
    static_assert(smem <= 227 * 1024, "shared memory");
    auto kern = prefill_kernel<T, D, G, PREFILL_NWC, S>;
    static std::atomic<bool> attr_set[64];    // per device, read by any host thread
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
    }
    // One block per item.  The items are at most the worst case (every
    // sequence with `groups` row groups), and at most 2 * ceil(rows / 64) row
    // groups per KV head over all runs together, since every run taken here
    // has at least 64 rows; blocks past the real count return at once.
    const long long worst = (long long)groups * p.num_seqs * p.num_kv_heads;
    const long long rows_all = (long long)p.num_q_rows * G;
    const long long bound =
        (long long)p.num_kv_heads * 2 * ((rows_all + PREFILL_GROUP_ROWS - 1) / PREFILL_GROUP_ROWS);
    long long blocks = worst < bound ? worst : bound;
    if (blocks <= 0) return cudaSuccess;
    if (blocks > 0x7fffffffLL) blocks = 0x7fffffffLL;   // then blocks take several items
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3((PREFILL_NWC + 1) * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, groups);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_prefill(const DecodeParams &p, int D, int G, int groups, cudaStream_t st) {
#define PA_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_prefill<T, DD, GG>(p, groups, st);
    PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 4) PA_CASE(64, 8)
    PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 4) PA_CASE(128, 8)
#undef PA_CASE
    return cudaErrorNotSupported;
}

}  // namespace pa
