// pa_prefill_tc.cuh -- the prefill path (multi-token queries with many rows
// per sequence: a chunk of a long prompt) on the fifth-generation tensor
// cores.
//
// "vLLM: Architecture, PagedAttention & Internals", *Prefill, decode, and
// chunked prefill*: one forward pass carries a slice of a long prompt next
// to one-token decodes.  Row r of sequence s's slice (token i = r / G, head
// r % G of the KV head's group) attends over positions 0 .. L - n + i of the
// paged cache.
//
// A work item is 128 such rows of one (sequence, KV head) -- the M side of
// one tcgen05 MMA -- in the order of prefill_schedule (longest sequences
// first, one item per block).  Per step of 64 keys (four 16-token cache
// blocks):
//   1. S = Q K^T: tcgen05.mma, M = 128, N = 64, K = head_dim, both operands
//      K-major from shared memory (128-byte swizzle): Q written once per item
//      by the block's threads, the K tiles by tensor-map copies, the four
//      blocks of a step stacked into one 64-row operand; S lands in TMEM.
//   2. Each thread owns one row: it reads its 64 scores from TMEM
//      (tcgen05.ld), masks positions past its causal limit, updates the
//      online softmax in fp32 (lazy rescaling, as in the warp-level paths),
//      rescales its row of O in TMEM when its reference level moved, and
//      writes its probabilities, rounded to the cache type, back into TMEM
//      (two per 32-bit column, its lane = its row).
//   3. O += P V: tcgen05.mma, M = 128, N = head_dim, K = 64, P read from TMEM,
//      V from shared memory MN-major (its rows are keys, head_dim
//      contiguous); O accumulates in TMEM over the whole item and is read
//      back, normalised, at the end.
// A producer warp (lane 0) follows the same item order and keeps a ring of
// K/V stages filled with tensor-map copies, each stage freed by a commit after
// its P.V; one consumer thread issues the MMAs; completion comes back through
// mbarriers (tcgen05.commit); the four consumer warps synchronise among
// themselves on a named barrier.  The MMAs of one thread run in order, so when
// S of step c+1 is complete, P.V of step c is too: its P tile, its K/V stage
// and O are then free.  A ring of two K/V stages runs ahead of the MMAs;
// two blocks share an SM (about 100 KB of shared memory and 256 TMEM columns
// each), so one block's softmax overlaps the other's MMAs.  The grid is
// persistent (two blocks per SM); block b takes the items b, 2R-1-b, 2R+b, ...
// of the cost-sorted list (R blocks), which deals the long items out first.
// Every wait is bounded; on a timeout the block stops and the error word
// says so.
#pragma once

#include <climits>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_internal.h"
#include "pa_mma.cuh"
#include "pa_prefill.cuh"
#include "pa_tc5.cuh"

namespace pa {

constexpr int TC_ROWS = PREFILL_TC_ROWS;   // query rows of one item (the MMA's M)
constexpr int TC_KEYS = 64;    // keys per step (the S tile's N): four cache blocks

template <typename T, int D>
struct PrefillTcLayout {
    static constexpr int NH = D / 64;                                  // 128-byte groups of a row
    static constexpr size_t Q_BYTES = (size_t)TC_ROWS * D * 2;         // [NH][128 rows][128 B]
    static constexpr size_t KV_BYTES = (size_t)TC_KEYS * D * 2;        // [NH][64 keys][128 B]
    static constexpr int STAGES = 2;
    static constexpr size_t OFF_Q = 0;
    static constexpr size_t OFF_KV = OFF_Q + Q_BYTES;                  // stage st: K, then V
    static constexpr size_t OFF_BARS = OFF_KV + (size_t)STAGES * 2 * KV_BYTES;
    static constexpr size_t OFF_TMEM = OFF_BARS + (size_t)(2 * STAGES + 2) * 8;
    static constexpr size_t BYTES = OFF_TMEM + 16 + 1024;              // + alignment of the base
    static_assert(Q_BYTES % 1024 == 0 && KV_BYTES % 1024 == 0,
                  "1024-byte aligned swizzle atoms");
};

// TMEM columns of a block: S 0..63, P 64..95 (bf16/f16 pairs), O 128..128+D-1
constexpr uint32_t TC_TMEM_COLS = 256;
constexpr int TC_BLOCKS_PER_SM = 2;
constexpr int TC_CONSUMERS = 4;          // warps of the softmax (one row per thread)

// The consumer warps' own barrier (named barrier 1), plain and with an AND
// of a predicate.
__device__ __forceinline__ void tc_consumers_sync() {
    asm volatile("bar.sync 1, 128;" ::: "memory");
}
__device__ __forceinline__ bool tc_consumers_sync_and(bool pred) {
    uint32_t r;
    asm volatile("{\n\t.reg .pred p, q;\n\tsetp.ne.u32 p, %1, 0;\n\t"
                 "bar.red.and.pred q, 1, 128, p;\n\tselp.u32 %0, 1, 0, q;\n\t}"
                 : "=r"(r) : "r"((uint32_t)pred) : "memory");
    return r != 0;
}

template <typename T, int D, int G>
__global__ void __launch_bounds__((TC_CONSUMERS + 1) * 32, TC_BLOCKS_PER_SM)
prefill_tc_kernel(const __grid_constant__ DecodeParams p, int groups) {
    static_assert(sizeof(T) == 2 && (D == 64 || D == 128), "16-bit caches, head_dim 64 or 128");
    using Lay = PrefillTcLayout<T, D>;
    constexpr int NH = Lay::NH, S = Lay::STAGES;
    constexpr uint32_t KVB = (uint32_t)Lay::KV_BYTES;
    constexpr uint32_t ID_S = tc5_idesc<T>(TC_ROWS, TC_KEYS, 0);    // Q K^T: both K-major
    constexpr uint32_t ID_O = tc5_idesc<T>(TC_ROWS, D, 1);          // P V: V MN-major

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sQ = smem + Lay::OFF_Q;
    unsigned char *sKV = smem + Lay::OFF_KV;
    uint64_t *full = reinterpret_cast<uint64_t *>(smem + Lay::OFF_BARS);   // [S]: a stage landed
    uint64_t *empty = full + S;                    // [S]: a stage's P.V is done
    uint64_t *s_done = full + 2 * S;               // S of a step is in TMEM
    uint64_t *pv_done = full + 2 * S + 1;          // the item's last P.V is done
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay::OFF_TMEM);
    __shared__ PrefillSched sched;

    const int tid = threadIdx.x, warp = tid >> 5;
    const int Hkv = p.num_kv_heads, H = p.num_heads;

    if (tid == 0) {
        prefetch_tensormap(&p.tmap_k);
        prefetch_tensormap(&p.tmap_v);
        for (int i = 0; i < 2 * S; ++i) mbar_init(&full[i], 1);   // full and empty
        mbar_init(s_done, 1);
        mbar_init(pv_done, 1);
        fence_mbar_init();
    }
    if (warp == 0) tc5_alloc(tmem_slot, TC_TMEM_COLS);
    tc5_fence_before_sync();
    __syncthreads();
    tc5_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t lane_off = (uint32_t)(warp * 32) << 16;   // this warp's TMEM lanes
    const uint32_t tS = tmem, tP = tmem + 64, tO = tmem + 128;

    const int total = prefill_schedule<G, TC_ROWS>(p, groups, sched);

    // the caches (and q, out) only after the kernel before this one is done
    grid_dependency_wait();

    const uint64_t pol = policy_evict_last();      // the sequence's other items reread them
    // a box past the end of the tensor fills with zeros
    const int z_none = (int)min((long long)INT_MAX, p.num_blocks * (long long)Hkv);
    long long kglob = 0;                           // steps through the K/V ring so far
    uint32_t n_s = 0, n_pv = 0;                    // phases of s_done and pv_done so far
    bool ok = true;

    const int R = (int)gridDim.x, me = (int)blockIdx.x;
    // The geometry of an item; the producer and the consumers compute it alike.
    struct Item {
        int s, j, grp, q0, nq, L, nrows, nsteps, nb_seq;
    };
    auto item_at = [&](int k, Item &it) -> bool {  // all lanes of a warp
        const long long xl = (long long)k * R + ((k & 1) ? (R - 1 - me) : me);   // snake
        if (xl >= total) return false;
        prefill_item<G, TC_ROWS>(p, groups, sched, (int)xl, it.s, it.j, it.grp);
        it.q0 = p.query_start[it.s];
        it.nq = p.query_start[it.s + 1] - it.q0;
        it.L = p.seq_lens[it.s];
        it.nrows = min(TC_ROWS, it.nq * G - it.grp * TC_ROWS);   // >= 1
        const int last_tok = (it.grp * TC_ROWS + it.nrows - 1) / G;
        const int n_keys = it.L - it.nq + last_tok + 1;          // keys any row sees
        it.nsteps = (n_keys + TC_KEYS - 1) / TC_KEYS;
        it.nb_seq = (it.L + 15) >> 4;                            // blocks of the sequence
        return true;
    };

    if (warp == TC_CONSUMERS) {
        // ---- producer: step kk of the block's items into stage kk % S once its
        // previous use is done (lane 0 issues)
        long long kk = 0;
        bool pok = true;
        Item it;
        for (int k = 0; pok && item_at(k, it); ++k) {
            for (int c = 0; pok && c < it.nsteps; ++c, ++kk) {
                const int st = (int)(kk % S);
                bool w = true;
                if (threadIdx.x % 32 == 0) {
                    w = kk < S || mbar_wait_bounded(&empty[st], (uint32_t)(((kk / S) - 1) & 1), p.err);
                    if (w) {
                        int pbs[TC_KEYS / 16];
#pragma unroll
                        for (int b = 0; b < TC_KEYS / 16; ++b) {   // independent loads
                            const int lb = (TC_KEYS / 16) * c + b;
                            pbs[b] = lb < it.nb_seq ? p.block_tables[(long long)it.s * p.max_blocks + lb] : -1;
                        }
                        unsigned char *dK = sKV + (size_t)st * 2 * KVB, *dV = dK + KVB;
                        mbar_arrive_expect_tx(&full[st], 2 * KVB);
#pragma unroll
                        for (int b = 0; b < TC_KEYS / 16; ++b) {
                            const int lb = (TC_KEYS / 16) * c + b;
                            int z = z_none;                // past the sequence: zeros
                            if (lb < it.nb_seq) {
                                if (pbs[b] >= 0 && (long long)pbs[b] < p.num_blocks) z = pbs[b] * Hkv + it.j;
                                else set_error(p.err, ERR_BLOCK_ID);
                            }
#pragma unroll
                            for (int h = 0; h < NH; ++h) {
                                tma_load_3d(dK + h * (TC_KEYS * 128) + b * 2048, &p.tmap_k, h * 64, 0, z,
                                            &full[st], pol);
                                tma_load_3d(dV + h * (TC_KEYS * 128) + b * 2048, &p.tmap_v, h * 64, 0, z,
                                            &full[st], pol);
                            }
                        }
                    }
                }
                pok = __shfl_sync(0xffffffffu, w, 0);
            }
        }
        // copies still landing when the block exits: wait (bounded) for the last S
        if (threadIdx.x % 32 == 0)
            for (long long i = (kk > S ? kk - S : 0); i < kk; ++i)
                mbar_wait_bounded(&full[i % S], (uint32_t)((i / S) & 1), p.err);
    } else {
        // ---- consumers (thread 0 also issues the MMAs)
        Item it;
        for (int k = 0; ok && item_at(k, it); ++k) {
            const int s = it.s, j = it.j, grp = it.grp, q0 = it.q0, nq = it.nq, L = it.L;
            const int nrows = it.nrows, nsteps = it.nsteps, nb_seq = it.nb_seq;
            // this thread's row
            const int r = tid;
            const bool row_ok = r < nrows;
            const int rr = grp * TC_ROWS + r;
            const int tok = rr / G, head = rr % G;
            const int lim = L - nq + tok;                         // last visible position
            (void)s;

            // -- Q rows into sQ ([NH][128 rows][128 B], 128-byte swizzle); zeros past the run
            {
                const uint4 *qr = reinterpret_cast<const uint4 *>(
                    reinterpret_cast<const T *>(p.q) + (long long)(q0 + (row_ok ? tok : 0)) * p.q_seq_stride +
                    (long long)(j * G + head) * D);
#pragma unroll
                for (int c = 0; c < D / 8; ++c) {
                    const uint4 v = row_ok ? __ldg(qr + c) : make_uint4(0, 0, 0, 0);
                    const int h = c >> 3, cc = c & 7;
                    *reinterpret_cast<uint4 *>(sQ + h * (TC_ROWS * 128) + r * 128 + ((cc ^ (r & 7)) << 4)) = v;
                }
            }
            fence_proxy_async_smem();              // before the MMAs read sQ

            // -- S of step c (thread 0, after its stage landed); false on a timeout
            auto issue_s = [&](int c) -> bool {
                const long long kk = kglob + c;
                const int st = (int)(kk % S);
                if (!mbar_wait_bounded(&full[st], (uint32_t)((kk / S) & 1), p.err)) return false;
                const uint32_t kaddr = smem_u32(sKV + (size_t)st * 2 * KVB);
#pragma unroll
                for (int ks = 0; ks < D / 16; ++ks) {
                    const uint32_t off = (uint32_t)((ks & 3) * 32);   // 16 elements = 32 bytes
                    tc5_mma(tS,
                            tc5_desc_sw128(smem_u32(sQ) + (ks >> 2) * (TC_ROWS * 128) + off, 16, 1024),
                            tc5_desc_sw128(kaddr + (ks >> 2) * (TC_KEYS * 128) + off, 16, 1024),
                            ID_S, ks > 0);
                }
                tc5_commit(s_done);
                return true;
            };

            float m_run = -INFINITY, l_run = 0.f;
            tc5_fence_before_sync();
            tc_consumers_sync();                   // sQ written
            bool issued = true;
            if (tid == 0) {
                tc5_fence_after_sync();
                issued = issue_s(0);
            }

            for (int c = 0; c < nsteps; ++c) {
                const bool got = issued && mbar_wait_bounded(s_done, n_s & 1, p.err);
                ++n_s;
                if (!tc_consumers_sync_and(got)) { ok = false; break; }
                tc5_fence_after_sync();

                // -- this row's 64 scores
                float sv[TC_KEYS];
                tc5_ld32(tS + lane_off, *reinterpret_cast<float(*)[32]>(&sv[0]));
                tc5_ld32(tS + lane_off + 32, *reinterpret_cast<float(*)[32]>(&sv[32]));
                const int kb = c * TC_KEYS;
                float mx = -INFINITY;
#pragma unroll
                for (int e = 0; e < TC_KEYS; ++e) {
                    sv[e] = (row_ok && kb + e <= lim) ? sv[e] * p.scale_log2 : -INFINITY;
                    mx = fmaxf(mx, sv[e]);
                }
                // lazy rescaling: the reference level moves only by more than 2^RESCALE_LOG2
                const float m_new = mx > m_run + RESCALE_LOG2 ? mx : m_run;
                const float ms = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = m_new == m_run ? 1.f : ex2(m_run - ms);
                uint32_t pw[TC_KEYS / 2];
                float psum = 0.f;
#pragma unroll
                for (int e = 0; e < TC_KEYS / 2; ++e) {
                    pw[e] = Mma<T>::pack(ex2(sv[2 * e] - ms), ex2(sv[2 * e + 1] - ms));
                    float a, b;
                    Mma<T>::unpack(pw[e], a, b);
                    psum += a + b;
                }
                l_run = l_run * alpha + psum;
                m_run = m_new;
                // this row of O to the new level (O holds nothing before the first P.V)
                if (__any_sync(0xffffffffu, c > 0 && alpha != 1.f)) {
                    const float f = c > 0 ? alpha : 1.f;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        float o[32];
                        tc5_ld32(tO + lane_off + c0, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= f;
                        tc5_st32(tO + lane_off + c0, o);
                    }
                }
                // P row r into TMEM: 64 keys, two per column
                tc5_st32u(tP + lane_off, pw);
                // V rows of the sequence's last block past L hold other tokens' data
                // (zero-weighted, but 0 * NaN is NaN): clear them
                {
                    const int st = (int)((kglob + c) % S);
                    unsigned char *dV = sKV + (size_t)st * 2 * KVB + KVB;
                    const int tail = L & 15, lb_last = nb_seq - 1;
                    const int b = lb_last - (TC_KEYS / 16) * c;
                    if (tail != 0 && b >= 0 && b < TC_KEYS / 16) {
                        const int nclr = (16 - tail) * NH * 8;    // 16-byte pieces
                        for (int i = tid; i < nclr; i += 128) {
                            const int h = i / ((16 - tail) * 8), rem = i % ((16 - tail) * 8);
                            const int row = 16 * b + tail + rem / 8;
                            *reinterpret_cast<uint4 *>(dV + h * (TC_KEYS * 128) + row * 128 + (rem % 8) * 16) =
                                make_uint4(0, 0, 0, 0);
                        }
                    }
                }
                fence_proxy_async_smem();          // the cleared rows before the MMA
                tc5_fence_before_sync();
                tc_consumers_sync();
                if (tid == 0) {
                    tc5_fence_after_sync();
                    const int st = (int)((kglob + c) % S);
                    const uint32_t vaddr = smem_u32(sKV + (size_t)st * 2 * KVB + KVB);
#pragma unroll
                    for (int ks = 0; ks < TC_KEYS / 16; ++ks)
                        tc5_mma_ta(tO, tP + 8 * ks,
                                   tc5_desc_sw128(vaddr + ks * 2048, TC_KEYS * 128, 1024), ID_O,
                                   (c > 0 || ks > 0) ? 1u : 0u);
                    tc5_commit(&empty[st]);        // the stage is free once P.V is done
                    if (c + 1 < nsteps) issued = issue_s(c + 1);
                    else tc5_commit(pv_done);
                }
            }
            if (!ok) break;

            // -- O / l into out (this thread's row)
            const bool got = mbar_wait_bounded(pv_done, n_pv & 1, p.err);
            ++n_pv;
            if (!tc_consumers_sync_and(got)) { ok = false; break; }
            tc5_fence_after_sync();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            T *o = reinterpret_cast<T *>(p.out) + ((long long)(q0 + tok) * H + j * G + head) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float v[32];
                tc5_ld32(tO + lane_off + c0, v);
                if (row_ok) {
#pragma unroll
                    for (int e = 0; e < 32; e += 8) {
                        uint4 w;
                        w.x = Mma<T>::pack(v[e] * inv, v[e + 1] * inv);
                        w.y = Mma<T>::pack(v[e + 2] * inv, v[e + 3] * inv);
                        w.z = Mma<T>::pack(v[e + 4] * inv, v[e + 5] * inv);
                        w.w = Mma<T>::pack(v[e + 6] * inv, v[e + 7] * inv);
                        *reinterpret_cast<uint4 *>(o + c0 + e) = w;
                    }
                }
            }
            kglob += nsteps;
            tc5_fence_before_sync();
            tc_consumers_sync();                   // sQ and TMEM free for the next item
        }
    }

    tc5_fence_before_sync();
    __syncthreads();
    if (warp == 0) tc5_dealloc(tmem, TC_TMEM_COLS);
}

template <typename T, int D, int G>
cudaError_t launch_prefill_tc(const DecodeParams &p, int groups, cudaStream_t st) {
    using Lay = PrefillTcLayout<T, D>;
    constexpr size_t smem = Lay::BYTES;
    static_assert(smem + sizeof(PrefillSched) <= 227 * 1024, "shared memory");
    auto kern = prefill_tc_kernel<T, D, G>;
    static bool attr_set[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev]) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev] = true;
    }
    // persistent: the resident blocks (two per SM), but no more than the items
    // can be: the worst case, and at most 2 * ceil(rows / 64) items per KV head
    // over all runs together (each run has at least 64 rows)
    const long long worst = (long long)groups * p.num_seqs * p.num_kv_heads;
    const long long rows_all = (long long)p.num_q_rows * G;
    const long long bound =
        (long long)p.num_kv_heads * 2 * ((rows_all + PREFILL_GROUP_ROWS - 1) / PREFILL_GROUP_ROWS);
    const int sms = sm_count_of_current_device();
    long long blocks = (long long)(sms > 0 ? sms : 152) * TC_BLOCKS_PER_SM;
    if (blocks > worst) blocks = worst;
    if (blocks > bound) blocks = bound;
    if (blocks <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3((TC_CONSUMERS + 1) * 32, 1, 1);
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
cudaError_t dispatch_prefill_tc(const DecodeParams &p, int D, int G, int groups, cudaStream_t st) {
#define PA_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_prefill_tc<T, DD, GG>(p, groups, st);
    PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 4) PA_CASE(64, 8)
    PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 4) PA_CASE(128, 8)
#undef PA_CASE
    return cudaErrorNotSupported;
}

}  // namespace pa
