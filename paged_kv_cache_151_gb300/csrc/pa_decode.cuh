// pa_decode.cuh -- decode-step paged attention kernels for sm_103a.
//
// One thread block handles one (sequence, KV head) -- or one split of it --
// and all G query heads that share that KV head ("vLLM: Architecture,
// PagedAttention & Internals", *PagedAttention in one paragraph*: the kernel
// gathers K and V block by block through the block table; the arithmetic of
// attention is unchanged).
//
// Data movement.  Each warp owns a ring of S stages.  For each 16-token block
// of its share, lane 0 issues two 1-D bulk copies (cp.async.bulk, the TMA
// engine without a tensor map) of the block's K and V tiles -- each a
// contiguous run of rows*head_dim elements in the [block][kv_head][row][d]
// cache -- into the stage, completing on the stage's mbarrier.  Only the
// valid rows of a partial last block are copied.  Blocks are dealt to the
// warps of all CTAs of a cluster round-robin by logical block index, so the
// reduction order depends only on logical positions, never on where the
// blocks sit in the pool.
//
// Arithmetic per block (fp32):
//   scores   lane (r, c) reads 16-byte chunk c of row r + RPW*i of the K tile
//            and multiplies it with the matching slice of the G query
//            vectors held in registers; the per-lane partial dot products are
//            summed across the NCH lanes of a row by a shuffle
//            reduce-scatter (recursive halving), leaving each lane a few
//            complete scores.  Scores carry scale*log2(e) so that the
//            softmax can use exp2.
//   softmax  online: per head a running maximum m and sum l (fp32);
//            m_new = max(m, block max), alpha = 2^(m - m_new),
//            p_t = 2^(s_t - m_new), l = alpha*l + sum p_t  ("vLLM"
//            (stanleyjacob.dev), Part IV, *Stage 6: The forward pass*: the
//            kernel streams through a sequence it never holds in one piece).
//   P.V      acc[g][:] = alpha[g]*acc[g][:] + sum_t p[g][t] V[t][:], lane (r, c)
//            owning chunk c of the output for the rows of its row group.
// At the end the warps' (m, l, acc) are merged in shared memory and, when the
// (sequence, KV head) is split over a cluster, across the cluster through
// distributed shared memory; out = acc / l, rounded to the storage type.
// (The arithmetic is WarpAttn in pa_math.cuh; pa_persistent.cuh holds the
// persistent kernel that pa_decode and pa_decode_partitioned use by default.)
//
// This file also holds the log-sum-exp merge of split-KV partitions.
#pragma once

#include <cuda.h>   // CUtensorMap (a plain 128-byte descriptor; no driver calls here)

#include "pa_common.cuh"
#include "pa_math.cuh"

namespace pa {

struct DecodeParams {
    void *out;
    const void *q;
    const void *k_cache;
    const void *v_cache;
    const int32_t *block_tables;
    const int32_t *seq_lens;
    float *part_o;            // PARTIAL: [B][H][max_parts][D]
    float *part_m;            // PARTIAL: [B][H][max_parts]
    float *part_l;            // PARTIAL: [B][H][max_parts]
    long long num_blocks;
    long long q_seq_stride;   // elements
    int num_seqs;
    int num_heads;
    int num_kv_heads;
    int max_blocks;           // block-table row length
    int partition_blocks;     // PARTIAL: 16-token blocks per partition
    int max_parts;            // PARTIAL: partitions the workspace holds
    int max_seq_len;          // PARTIAL: bound on seq_len
    const int32_t *query_start;  // multi-token queries: [num_seqs + 1] row offsets
    int max_query_len;        // multi-token queries: bound on a sequence's rows
    int num_q_rows;           // multi-token queries: rows of q and out
    int mq_split_rows;        // multi-token queries: > 0: sequences with at least this
                              // many (token, head) rows are left to the prefill kernel
    // cascade prefix (prefill_tc_kernel): prefix_nblocks > 0 attends the G
    // heads of every sequence to the shared prefix blocks prefix_blocks[0..n),
    // in chunks of prefix_chunk_blocks blocks; chunk c's (m, l, o) per
    // (sequence, head) go to partition c of part_o / part_m / part_l
    const int32_t *prefix_blocks;
    int prefix_nblocks;
    int prefix_chunk_blocks;
    const float *k_scale;     // E4M3 caches: [num_kv_heads] dequantisation scales
    const float *v_scale;
    float scale_log2;         // scale * log2(e)
    int test_stall = 0;       // test hook (pa_test_stall_next_decode): each warp's
                              // first copy expects 16 bytes it never gets
    unsigned int *err;        // device error word
    // 16-bit and E4M3 caches, persistent kernel: the caches as 3-D tensors
    // [num_blocks*num_kv_heads][16 rows][head_dim], read in swizzled boxes
    // of 16 rows x 128 bytes (16-bit) or 16 rows x head_dim bytes (E4M3)
    CUtensorMap tmap_k;
    CUtensorMap tmap_v;
    // 16-bit caches: the same tensors read in boxes of 8 rows, for blocks
    // holding at most 8 valid tokens (the last block of a sequence)
    CUtensorMap tmap_k8;
    CUtensorMap tmap_v8;
};

// Stages per warp: about 24 KiB of K+V in flight per warp, at least 2.
template <typename T, int D>
__host__ __device__ constexpr int stages_for() {
    constexpr int per = 2 * Shape<T, D>::TILE_BYTES;
    constexpr int s = 24576 / per;
    return s < 2 ? 2 : (s > 8 ? 8 : s);
}

// The stage buffers; after the block loop the same bytes hold the merge data.
template <typename T, int D, int G, int NW, int S>
__host__ __device__ constexpr size_t stage_region_bytes() {
    constexpr size_t stages = (size_t)NW * S * 2 * Shape<T, D>::TILE_BYTES;
    constexpr size_t merge = (size_t)(NW * (2 * G + G * D) + 2 * G + G * D) * 4;
    constexpr size_t region = stages > merge ? stages : merge;
    return (region + 127) / 128 * 128;
}

// stage region | mbarriers [NW*S] | q [G*D] fp32 | per-warp scratch
template <typename T, int D, int G, int NW, int S>
__host__ __device__ constexpr size_t decode_smem_bytes() {
    return stage_region_bytes<T, D, G, NW, S>() + (size_t)NW * S * 8 +
           (size_t)G * D * 4 + (size_t)NW * warp_scratch_floats<G>() * 4;
}

// One thread block per (split, KV head, sequence); the splits of one
// (sequence, KV head) form a thread-block cluster and merge through
// distributed shared memory.
template <typename T, int D, int G, int NW, int S>
__global__ void __launch_bounds__(NW * 32)
decode_split_kernel(const DecodeParams p) {
    using W = WarpAttn<T, D, G>;
    using Sh = Shape<T, D>;
    constexpr int ROWB = Sh::ROW_BYTES, TILE = Sh::TILE_BYTES;
    constexpr int WS = warp_scratch_floats<G>();
    static_assert(S <= 32, "stage count");

    extern __shared__ __align__(128) unsigned char smem[];
    constexpr size_t STAGE_REGION = stage_region_bytes<T, D, G, NW, S>();
    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + STAGE_REGION);
    float *qs = reinterpret_cast<float *>(bars + NW * S);
    float *wscr_all = qs + G * D;

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int j = blockIdx.y, s = blockIdx.z;
    const int H = p.num_heads, Hkv = p.num_kv_heads;

    // ---- which tokens this block handles ----------------------------------
    int L = p.seq_lens[s];
    const int cap = p.max_blocks * 16;
    if (L < 0 || L > cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0) set_error(p.err, ERR_SEQ_LEN);
        L = L < 0 ? 0 : cap;
    }
    const int nb = (L + 15) >> 4;
    const int rank = (int)cluster_ctarank();
    const int nrank = (int)cluster_nctarank();

    // ---- set-up: barriers and the G query vectors (pre-scaled) -------------
    if (threadIdx.x == 0) {
        for (int i = 0; i < NW * S; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    {
        const T *qp = reinterpret_cast<const T *>(p.q) + (long long)s * p.q_seq_stride +
                      (long long)j * G * D;
        for (int i = threadIdx.x; i < G * D; i += NW * 32)
            qs[i] = Elem<T>::load1(qp + i) * p.scale_log2;
    }
    __syncthreads();

    W wa;
    wa.init(lane);
    wa.load_q_smem(qs);
    float *Sc = wscr_all + warp * WS;
    float *Pb = Sc + 16 * G;
    float *Al = Pb + 16 * G;

    // ---- this warp's share of the blocks: logical blocks worker, worker +
    // nwk, ... (dealt round-robin over the warps of all CTAs of the cluster)
    const int worker = rank * NW + warp, nwk = nrank * NW;
    const int n_mine = nb > worker ? (nb - worker + nwk - 1) / nwk : 0;
    const int32_t *bt_row = p.block_tables + (long long)s * p.max_blocks;
    auto table_entry = [&](int k) -> int {
        return k < n_mine ? bt_row[worker + k * nwk] : 0;
    };
    int c0 = 0;
    int tab_cur = table_entry(lane), tab_nxt = table_entry(32 + lane);
    auto pb_of = [&](int k) -> int {                  // warp-uniform k
        const int kk = k - c0;
        const int a = __shfl_sync(0xffffffffu, tab_cur, kk & 31);
        const int b = __shfl_sync(0xffffffffu, tab_nxt, kk & 31);
        return kk < 32 ? a : b;
    };
    unsigned char *my_stages = stages + (size_t)warp * S * 2 * TILE;
    uint64_t *my_bars = bars + warp * S;
    const uint64_t pol = policy_evict_first();
    const unsigned char *kbase = reinterpret_cast<const unsigned char *>(p.k_cache);
    const unsigned char *vbase = reinterpret_cast<const unsigned char *>(p.v_cache);
    auto rows_of = [&](int k) -> int { return min(16, L - (worker + k * nwk) * 16); };
    auto issue = [&](int k, int pbk) {                // lane 0 only
        uint64_t *bar = &my_bars[k % S];
        if (pbk < 0 || (long long)pbk >= p.num_blocks) {
            set_error(p.err, ERR_BLOCK_ID);
            mbar_arrive(bar);                          // completes the phase, no data
            return;
        }
        const uint32_t bytes = (uint32_t)(rows_of(k) * ROWB);
        const size_t off = ((size_t)pbk * Hkv + j) * TILE;
        unsigned char *dst = my_stages + (size_t)(k % S) * 2 * TILE;
        mbar_arrive_expect_tx(bar, 2 * bytes);
        bulk_g2s(dst, kbase + off, bytes, bar, pol);
        bulk_g2s(dst + TILE, vbase + off, bytes, bar, pol);
    };

    const int pre = n_mine < S ? n_mine : S;
    for (int k = 0; k < pre; ++k) {
        const int pbk = pb_of(k);
        if (lane == 0) issue(k, pbk);
    }

    int k_done = 0;
    bool ok = true;
    for (int k = 0; k < n_mine; ++k) {
        if (k - c0 == 32) {
            c0 += 32;
            tab_cur = tab_nxt;
            tab_nxt = table_entry(c0 + 32 + lane);
        }
        const int st = k % S;
        const int pbk = pb_of(k);
        const bool waited = mbar_wait_bounded(&my_bars[st], (uint32_t)((k / S) & 1), p.err);
        if (!__all_sync(0xffffffffu, waited)) { ok = false; break; }
        k_done = k + 1;
        if (pbk >= 0 && (long long)pbk < p.num_blocks) {
            const unsigned char *Kt = my_stages + (size_t)st * 2 * TILE;
            wa.block(Kt, Kt + TILE, rows_of(k), Sc, Pb, Al);
        }
        __syncwarp();
        const int kn = k + S;
        if (kn < n_mine) {
            const int pbn = pb_of(kn);
            if (lane == 0) {
                fence_proxy_async_smem();
                issue(kn, pbn);
            }
        }
    }

    // ---- after a timeout: wait (bounded) for this warp's copies in flight ----
    bool drained = true;
    if (!ok) {
        const int issued = min(n_mine, k_done + S);
        for (int k = k_done; k < issued; ++k)
            drained &= mbar_wait_bounded(&my_bars[k % S], (uint32_t)((k / S) & 1), p.err);
        drained = __all_sync(0xffffffffu, drained);
    }
    const bool cta_ok = __syncthreads_and(drained ? 1 : 0) != 0;
    wa.finish();

    // merge region (reuses the stage buffers: every copy has landed)
    float *Mw = reinterpret_cast<float *>(stages);      // [NW][G]
    float *Lw = Mw + NW * G;                            // [NW][G]
    float *Aw = Lw + NW * G;                            // [NW][G][D]
    float *Mc = Aw + NW * G * D;                        // [G]
    float *Lc = Mc + G;                                 // [G]
    float *Oc = Lc + G;                                 // [G][D]
    if (cta_ok) wa.store_partial(Mw + warp * G, Lw + warp * G, Aw + warp * G * D);
    __syncthreads();

    const int h0 = j * G;
    for (int idx = threadIdx.x; idx < G * D && cta_ok; idx += NW * 32) {
        const int g = idx / D, d = idx % D;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < NW; ++w) M = fmaxf(M, Mw[w * G + g]);
        float O = 0.f, Ls = 0.f;
        if (M != -INFINITY) {
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const float mw = Mw[w * G + g];
                const float f = mw == -INFINITY ? 0.f : ex2(mw - M);
                O = fmaf(f, Aw[(w * G + g) * D + d], O);
                Ls = fmaf(f, Lw[w * G + g], Ls);
            }
        }
        if (nrank == 1) {
            T *o = reinterpret_cast<T *>(p.out) + ((long long)s * H + h0 + g) * D + d;
            Elem<T>::store1(o, Ls > 0.f ? O / Ls : 0.f);
        } else {
            Oc[idx] = O;
            if (d == 0) { Mc[g] = M; Lc[g] = Ls; }
        }
    }

    if (nrank > 1) {
        // rank q finalises outputs [q*G*D/n, (q+1)*G*D/n) from every rank's (M, L, O)
        cluster_sync();
        const int per = (G * D + nrank - 1) / nrank;
        const int beg = rank * per, end = min(G * D, beg + per);
        for (int idx = beg + threadIdx.x; idx < end; idx += NW * 32) {
            const int g = idx / D, d = idx % D;
            float M = -INFINITY;
            for (int q = 0; q < nrank; ++q) M = fmaxf(M, ld_dsmem_f32(map_to_rank(&Mc[g], q)));
            float O = 0.f, Ls = 0.f;
            if (M != -INFINITY) {
                for (int q = 0; q < nrank; ++q) {
                    const float mq = ld_dsmem_f32(map_to_rank(&Mc[g], q));
                    const float f = mq == -INFINITY ? 0.f : ex2(mq - M);
                    O = fmaf(f, ld_dsmem_f32(map_to_rank(&Oc[idx], q)), O);
                    Ls = fmaf(f, ld_dsmem_f32(map_to_rank(&Lc[g], q)), Ls);
                }
            }
            if (cta_ok) {
                T *o = reinterpret_cast<T *>(p.out) + ((long long)s * H + h0 + g) * D + d;
                Elem<T>::store1(o, Ls > 0.f ? O / Ls : 0.f);
            }
        }
        cluster_sync();     // keep this CTA's shared memory alive for the peers
    }
}

// ---- log-sum-exp merge of the partitions -----------------------------------
struct MergeParams {
    void *out;
    const float *part_o;
    const float *part_m;
    const float *part_l;
    const int32_t *seq_lens;
    int num_heads;
    int head_dim;
    int max_parts;
    int partition_size;
    int seq_cap;              // min(max_seq_len, max_blocks*16)
    int prefix_parts;         // cascade: leading parts of the shared prefix, always
                              // present; the sequence's own partitions follow them
};

// One block of 128 threads per (head, sequence) row.  The weight of
// partition q, c_q = l_q * 2^((m_q - M) log2 e) with M the largest m_q, is
// formed once (threads over partitions, 128 at a time) into shared memory;
// thread d then sums c_q * o_q[d] and c_q over the partitions in partition
// order, eight loads in flight.
template <typename T>
__global__ void __launch_bounds__(128) lse_merge_kernel(const MergeParams p) {
    constexpr int NT = 128, UNR = 8;
    __shared__ float cw[NT];
    __shared__ float wmax[NT / 32];
    const int h = blockIdx.x, s = blockIdx.y, tid = threadIdx.x;
    // launched right behind the split-KV kernel that writes the partials, which
    // lets it start early: wait for that kernel before reading anything
    grid_dependency_wait();
    int L = p.seq_lens[s];
    L = L < 0 ? 0 : (L > p.seq_cap ? p.seq_cap : L);
    const int n = p.prefix_parts + (L + p.partition_size - 1) / p.partition_size;
    const long long row = ((long long)s * p.num_heads + h) * p.max_parts;
    const float *m = p.part_m + row;
    const float *l = p.part_l + row;
    const int D = p.head_dim;                      // <= NT
    const bool dv = tid < D;
    const float *o = p.part_o + row * D + tid;
    float mx = -INFINITY;
    for (int q = tid; q < n; q += NT) mx = fmaxf(mx, m[q]);
#pragma unroll
    for (int k = 16; k > 0; k >>= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, k));
    if ((tid & 31) == 0) wmax[tid >> 5] = mx;
    __syncthreads();
    const float M = fmaxf(fmaxf(wmax[0], wmax[1]), fmaxf(wmax[2], wmax[3]));
    float O = 0.f, S = 0.f;
    for (int q0 = 0; q0 < n; q0 += NT) {
        const int q = q0 + tid;
        const float c = q < n ? l[q] * ex2((m[q] - M) * LOG2E) : 0.f;
        __syncthreads();                           // the previous weights are used up
        cw[tid] = c;
        __syncthreads();
        const int nc = min(NT, n - q0);
        const float *oq = o + (long long)q0 * D;
        int j = 0;
        for (; j + UNR <= nc; j += UNR) {
            float ov[UNR];
#pragma unroll
            for (int u = 0; u < UNR; ++u) ov[u] = dv ? oq[(long long)(j + u) * D] : 0.f;
#pragma unroll
            for (int u = 0; u < UNR; ++u) {
                S += cw[j + u];
                O = fmaf(cw[j + u], ov[u], O);
            }
        }
        for (; j < nc; ++j) {
            const float ov = dv ? oq[(long long)j * D] : 0.f;
            S += cw[j];
            O = fmaf(cw[j], ov, O);
        }
    }
    T *out = reinterpret_cast<T *>(p.out) + ((long long)s * p.num_heads + h) * D;
    if (dv) Elem<T>::store1(out + tid, n > 0 ? O / S : 0.f);
}

// ---- host-side launch helpers ------------------------------------------------
int sm_count_of_current_device();

template <typename T, int D, int G>
cudaError_t launch_split(const DecodeParams &p, dim3 grid, int splits, cudaStream_t st) {
    constexpr int NW = 4;
    constexpr int S = stages_for<T, D>();
    constexpr size_t smem = decode_smem_bytes<T, D, G, NW, S>();
    auto kern = decode_split_kernel<T, D, G, NW, S>;
    static_assert(smem <= 227 * 1024, "shared memory");
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem);
    if (e != cudaSuccess) return e;
    if (splits <= 1) {
        kern<<<grid, NW * 32, smem, st>>>(p);
        return cudaGetLastError();
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = dim3(NW * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T>
cudaError_t launch_merge(const MergeParams &p, int num_seqs, cudaStream_t st) {
    // programmatic dependent launch: the blocks may become resident while the
    // split-KV kernel (which signals its dependents at entry) still runs
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)p.num_heads, (unsigned)num_seqs, 1);
    cfg.blockDim = dim3(128, 1, 1);
    cfg.dynamicSmemBytes = 0;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, lse_merge_kernel<T>, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Dispatch of the cluster-split kernel over (head_dim, group size) for one
// storage type.  Returns cudaErrorNotSupported for shapes that are not built.
template <typename T>
cudaError_t dispatch_split(const DecodeParams &p, int D, int G, dim3 grid, int splits,
                           cudaStream_t st) {
#define PA_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_split<T, DD, GG>(p, grid, splits, st);
    PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 4) PA_CASE(64, 8)
    PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 4) PA_CASE(128, 8)
#undef PA_CASE
    return cudaErrorNotSupported;
}

}  // namespace pa
