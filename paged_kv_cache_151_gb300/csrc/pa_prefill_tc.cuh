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
// first).  Per step of 64 keys (four 16-token cache blocks):
//   1. S = Q K^T: tcgen05.mma, M = 128, N = 64, K = head_dim, both operands
//      K-major in shared memory (128-byte swizzle): Q by one tensor-map copy
//      per item, the four K blocks of the step by tensor-map copies stacked
//      into one 64-row operand.  S lands in the block's S buffer in TMEM.
//   2. Each softmax thread owns one row (TMEM lane = row): it reads its 64
//      scores (tcgen05.ld) -- after which S of the next step may overwrite
//      the buffer -- masks positions past its causal limit (only on the
//      steps that reach past some row's limit), updates the online softmax
//      in fp32 (lazy rescaling, as in the warp-level paths; two lanes per
//      instruction where the arithmetic allows), rescales its row of O in
//      TMEM when its reference level moved, and writes its probabilities,
//      rounded to the cache type, into the step's P buffer (two per column;
//      even and odd steps alternate between two buffers).
//   3. O += P V: tcgen05.mma, M = 128, N = head_dim, K = 64, P read from TMEM,
//      V from shared memory MN-major (rows = keys, head_dim contiguous).  O
//      accumulates in TMEM over the whole item and is read back, normalised,
//      at the end.
// Roles: warps 0-3 run the softmax (warp w reaches TMEM lanes 32w..32w+31);
// warps 4 and 6 keep the copies going -- Q once per item and a ring of two K
// stages (warp 4; a K stage is free once its S is done), a ring of two V
// stages (warp 6; free once its P.V is done); lane 0 of warp 5 issues the
// S MMAs (S(g+1) once the softmax has read S(g) and K(g+1) has landed) and
// lane 0 of warp 7 the P.V MMAs (PV(g) once P(g) is written).  An MMA issue
// blocks while the tensor pipe, which the SM's two blocks share, is busy;
// with two issuers a P.V that is ready never waits behind S MMAs, or the
// reverse.  S and P.V write disjoint TMEM columns, and each issuer's
// commits track its own MMAs.  Completion comes back through tcgen05.commit
// on mbarriers; neither MMA thread waits on an MMA's completion (the
// softmax waits for PV(g-2) before reusing its P buffer, the copy warps for
// S(g-2) and PV(g-2) before reusing a stage).  Two blocks share
// an SM (about 104 KB of shared memory and 256 TMEM columns each).  The
// grid is persistent; block b takes the items b, 2R-1-b, 2R+b, ... of the
// sorted list (R blocks), which deals the long items out first.  Every wait
// is bounded; on a timeout the block stops and the error word says so.
#pragma once

#include <atomic>
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
    static constexpr int STAGES = 2;                                   // of K, and of V
    static constexpr size_t OFF_Q = 0;
    static constexpr size_t OFF_K = OFF_Q + Q_BYTES;
    static constexpr size_t OFF_V = OFF_K + (size_t)STAGES * KV_BYTES;
    static constexpr size_t OFF_BARS = OFF_V + (size_t)STAGES * KV_BYTES;
    static constexpr int NBARS = 14;
    static constexpr size_t OFF_TMEM = OFF_BARS + (size_t)NBARS * 8;
    static constexpr size_t BYTES = OFF_TMEM + 16 + 1024;              // + alignment of the base
    static_assert(Q_BYTES % 1024 == 0 && KV_BYTES % 1024 == 0,
                  "1024-byte aligned swizzle atoms");
};

// TMEM columns of a block: S 0..63, P of even steps 64..95, of odd steps
// 96..127 (two 16-bit probabilities per column), O 128..128+D-1
constexpr uint32_t TC_TMEM_COLS = 256;
constexpr int TC_BLOCKS_PER_SM = 2;
constexpr int TC_SOFTMAX_WARPS = 4;      // one row per thread
constexpr int TC_COPY_WARP = 4;        // Q and K copies
constexpr int TC_MMA_WARP = 5;        // S MMAs
constexpr int TC_PV_WARP = 7;         // P.V MMAs
constexpr int TC_VCOPY_WARP = 6;       // V copies
constexpr int TC_THREADS = 8 * 32;

template <typename T, int D, int G>
__global__ void __launch_bounds__(TC_THREADS, TC_BLOCKS_PER_SM)
prefill_tc_kernel(const __grid_constant__ DecodeParams p, const __grid_constant__ CUtensorMap tmap_q,
                  int groups) {
    static_assert(sizeof(T) == 2 && (D == 64 || D == 128), "16-bit caches, head_dim 64 or 128");
    static_assert(TC_ROWS % G == 0, "an item holds whole tokens");
    using Lay = PrefillTcLayout<T, D>;
    constexpr int NH = Lay::NH;
    constexpr uint32_t KVB = (uint32_t)Lay::KV_BYTES;
    constexpr int TOKS = TC_ROWS / G;                               // tokens of one item
    constexpr uint32_t ID_S = tc5_idesc<T>(TC_ROWS, TC_KEYS, 0);    // Q K^T: both K-major
    constexpr uint32_t ID_O = tc5_idesc<T>(TC_ROWS, D, 1);          // P V: V MN-major

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *sQ = smem + Lay::OFF_Q;
    unsigned char *sK = smem + Lay::OFF_K;
    unsigned char *sV = smem + Lay::OFF_V;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::OFF_BARS);
    uint64_t *kfull = bars;          // [2] K of step g landed in stage g % 2
    uint64_t *vfull = bars + 2;      // [2] V of step g landed
    uint64_t *pv_done = bars + 4;    // [2] P.V of step g (and every MMA before it) done:
                                     //     V stage g % 2 and P buffer g % 2 free
    uint64_t *kfree = bars + 6;      // [2] S of step g done: K stage g % 2 free
    uint64_t *p_full = bars + 8;     // [2] P of step g written (four warp arrivals)
    uint64_t *q_full = bars + 10;    // Q of the item landed
    uint64_t *mma_idle = bars + 11;  // the block's MMAs are all done
    uint64_t *s_full = bars + 12;    // S of a step in TMEM (one phase per step)
    uint64_t *s_free = bars + 13;    // S of a step read by the softmax (four warp arrivals)
    uint32_t *tmem_slot = reinterpret_cast<uint32_t *>(smem + Lay::OFF_TMEM);
    __shared__ PrefillSched sched;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int Hkv = p.num_kv_heads, H = p.num_heads;

    // the decode kernel launched after this one (the rows of the short runs)
    // may set up on SMs this grid leaves; it waits for this grid before it
    // touches the caches or out
    launch_dependents();
    if (tid == 0) {
        prefetch_tensormap(&p.tmap_k);
        prefetch_tensormap(&p.tmap_v);
        prefetch_tensormap(&tmap_q);
        for (int i = 0; i < 8; ++i) mbar_init(&bars[i], 1);
        mbar_init(&p_full[0], TC_SOFTMAX_WARPS);
        mbar_init(&p_full[1], TC_SOFTMAX_WARPS);
        mbar_init(q_full, 1);
        mbar_init(mma_idle, 2);
        mbar_init(s_full, 1);
        mbar_init(s_free, TC_SOFTMAX_WARPS);
        fence_mbar_init();
    }
    if (warp == 0) tc5_alloc(tmem_slot, TC_TMEM_COLS);
    tc5_fence_before_sync();
    __syncthreads();
    tc5_fence_after_sync();
    const uint32_t tmem = *tmem_slot;
    const uint32_t tS = tmem, tP = tmem + 64, tO = tmem + 128;

    // Cascade prefix (p.prefix_nblocks > 0): an item is (prefix chunk, KV
    // head, 128 rows of (sequence, head) pairs) -- row r of row group grp is
    // head (grp*128 + r) % G of sequence (grp*128 + r) / G, every row sees
    // every key of the chunk, and the item writes the rows' (m, l, o) of the
    // chunk as a partition of the split-KV workspace.  Row groups of one
    // (chunk, KV head) are consecutive items, so their K/V come from L2.
    const bool cascade = p.prefix_nblocks > 0;
    const int nrg = (p.num_seqs * G + TC_ROWS - 1) / TC_ROWS;     // cascade row groups
    const int total = cascade
        ? ((p.prefix_nblocks + p.prefix_chunk_blocks - 1) / p.prefix_chunk_blocks) * Hkv * nrg
        : prefill_schedule<G, TC_ROWS>(p, groups, sched);

    // the caches (and q, out) only after the kernel before this one is done
    grid_dependency_wait();

    const int R = (int)gridDim.x, me = (int)blockIdx.x;
    // The geometry of an item; every role computes it alike.
    struct Item {
        int s, j, grp, q0, nq, L, nrows, nsteps, nb_seq;
    };
    auto item_at = [&](int k, Item &it) -> bool {  // all lanes of a warp
        const long long xl = (long long)k * R + ((k & 1) ? (R - 1 - me) : me);   // snake
        if (xl >= total) return false;
        if (cascade) {
            // it.s: the chunk; rows: (sequence, head) pairs of all sequences
            const int per = Hkv * nrg, x = (int)xl;
            it.s = x / per;
            it.j = (x % per) / nrg;
            it.grp = (x % per) % nrg;
            const int b0 = it.s * p.prefix_chunk_blocks;
            const int nbk = min(p.prefix_chunk_blocks, p.prefix_nblocks - b0);
            it.q0 = 0;
            it.nq = p.num_seqs;
            it.L = 16 * nbk;                                         // keys of the chunk
            it.nrows = min(TC_ROWS, p.num_seqs * G - it.grp * TC_ROWS);
            it.nsteps = (it.L + TC_KEYS - 1) / TC_KEYS;
            it.nb_seq = nbk;
            return true;
        }
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

    if (warp == TC_COPY_WARP || warp == TC_VCOPY_WARP) {
        // ---- copies.  Warp TC_COPY_WARP: Q of item k once S of item k-1's
        // last step is done, and K of step g into stage g % 2 once S(g-2) is
        // done; warp TC_VCOPY_WARP: V of step g once P.V(g-2) is done.  Two
        // warps, so that a K copy never waits behind a V stage (S(g-2)
        // completes well before P.V(g-2)).
        const bool kside = warp == TC_COPY_WARP;
        const uint64_t pol = policy_evict_last();  // the sequence's other items reread them
        const CUtensorMap *tmap = kside ? &p.tmap_k : &p.tmap_v;
        unsigned char *const stage0 = kside ? sK : sV;
        uint64_t *const full = kside ? kfull : vfull;
        uint64_t *const empty = kside ? kfree : pv_done;
        // a box past the end of the tensor fills with zeros
        const int z_none = (int)min((long long)INT_MAX, p.num_blocks * (long long)Hkv);
        long long g = 0, ncopies = 0;              // steps so far; stages issued
        int nq_issued = 0;
        bool pok = true;
        Item it;
        for (int k = 0; pok && item_at(k, it); ++k) {
            bool w = true;
            if (kside && lane == 0) {
                if (g > 0) w = mbar_wait_bounded(&kfree[(g - 1) & 1], (uint32_t)(((g - 1) >> 1) & 1), p.err);
                if (w) {
                    mbar_arrive_expect_tx(q_full, (uint32_t)Lay::Q_BYTES);
#pragma unroll
                    for (int h = 0; h < NH; ++h)
                        tma_load_3d(sQ + h * (TC_ROWS * 128), &tmap_q, h * 64, it.j * G,
                                    it.q0 + it.grp * TOKS, q_full, pol);
                    ++nq_issued;
                }
            }
            pok = __shfl_sync(0xffffffffu, w, 0);
            // Lane i < 4 holds the block-table entry of block i of the step,
            // read one step ahead so that its latency passes while the warp
            // waits for a stage; lanes l < 4 * NH then issue one box each
            // (block l % 4, 64-element half l / 4).
            const int32_t *row = cascade
                ? p.prefix_blocks + (long long)it.s * p.prefix_chunk_blocks
                : p.block_tables + (long long)it.s * p.max_blocks;
            auto fetch = [&](int c) -> int {
                const int lb = (TC_KEYS / 16) * c + lane;
                return (lane < TC_KEYS / 16 && c < it.nsteps && lb < it.nb_seq) ? __ldg(row + lb) : -1;
            };
            int pb_next = fetch(0);
            for (int c = 0; pok && c < it.nsteps; ++c, ++g) {
                const int b = (int)(g & 1);
                const uint32_t ph_prev = (uint32_t)(((g >> 1) - 1) & 1);   // phase of step g - 2
                int zl = z_none;                       // past the sequence: zeros
                {
                    const int lb = (TC_KEYS / 16) * c + lane, pb = pb_next;
                    if (lane < TC_KEYS / 16 && lb < it.nb_seq) {
                        if (pb >= 0 && (long long)pb < p.num_blocks) zl = pb * Hkv + it.j;
                        else if (kside) set_error(p.err, ERR_BLOCK_ID);
                    }
                }
                pb_next = fetch(c + 1);
                const int blk = lane % (TC_KEYS / 16), h = lane / (TC_KEYS / 16);
                const int z = __shfl_sync(0xffffffffu, zl, blk);
                w = true;
                if (lane == 0) {
                    w = g < 2 || mbar_wait_bounded(&empty[b], ph_prev, p.err);
                    if (w) mbar_arrive_expect_tx(&full[b], KVB);
                }
                w = __shfl_sync(0xffffffffu, w, 0);
                if (w && lane < (TC_KEYS / 16) * NH)
                    tma_load_3d(stage0 + (size_t)b * KVB + h * (TC_KEYS * 128) + blk * 2048, tmap, h * 64, 0, z,
                                &full[b], pol);
                if (w) ++ncopies;
                pok = w;
            }
        }
        // copies still landing when the block exits: wait (bounded) for the
        // last Q and the last two stages issued
        if (lane == 0) {
            if (nq_issued > 0) mbar_wait_bounded(q_full, (uint32_t)((nq_issued - 1) & 1), p.err);
            for (long long i = (ncopies > 2 ? ncopies - 2 : 0); i < ncopies; ++i)
                mbar_wait_bounded(&full[i & 1], (uint32_t)((i >> 1) & 1), p.err);
        }
    } else if (warp == TC_MMA_WARP || warp == TC_PV_WARP) {
        // ---- MMAs, issued by lane 0 of two warps so that a P.V that is ready
        // never waits behind S MMAs blocked on the busy pipe (or the reverse).
        // Warp TC_MMA_WARP: S(g) once K(g) has landed and the softmax has read
        // S(g-1) (one S buffer).  Warp TC_PV_WARP: PV(g) once P(g) is written
        // (P alternates between two buffers).  S and P.V use disjoint TMEM
        // columns; each warp's commits track its own MMAs.
        const bool sside = warp == TC_MMA_WARP;
        long long g0 = 0;
        bool mok = true;
        Item it;
        // Descriptors of the operands' bases; an offset of a multiple of 16
        // bytes inside shared memory adds offset / 16 to the start-address
        // field (addresses stay below 2^18, so the field does not overflow).
        const uint64_t dq = tc5_desc_sw128(smem_u32(sQ), 16, 1024);
        const uint64_t dk0 = tc5_desc_sw128(smem_u32(sK), 16, 1024), dk1 = dk0 + (KVB >> 4);
        const uint64_t dv0 = tc5_desc_sw128(smem_u32(sV), TC_KEYS * 128, 1024), dv1 = dv0 + (KVB >> 4);
        for (int k = 0; mok && item_at(k, it); ++k) {
            const int n = it.nsteps;
            bool w = true;
            if (lane == 0 && sside) {
                // the item's Q has landed
                w = mbar_wait_bounded(q_full, (uint32_t)(k & 1), p.err);
                for (int c = 0; w && c < n; ++c) {
                    const long long g = g0 + c;
                    const int b = (int)(g & 1);
                    // the softmax has read S(g-1); K(g) has landed
                    w = (g == 0 || mbar_wait_bounded(s_free, (uint32_t)((g - 1) & 1), p.err)) &&
                        mbar_wait_bounded(&kfull[b], (uint32_t)((g >> 1) & 1), p.err);
                    if (!w) break;
                    tc5_fence_after_sync();
                    const uint64_t kb = b ? dk1 : dk0;
#pragma unroll
                    for (int ks = 0; ks < D / 16; ++ks) {
                        // 16 elements = 32 bytes along K inside a 128-byte row; 64 per row group
                        const uint32_t qo = (uint32_t)(((ks >> 2) * (TC_ROWS * 128) + (ks & 3) * 32) >> 4);
                        const uint32_t ko = (uint32_t)(((ks >> 2) * (TC_KEYS * 128) + (ks & 3) * 32) >> 4);
                        tc5_mma(tS, dq + qo, kb + ko, ID_S, ks > 0);
                    }
                    tc5_commit(s_full);
                    tc5_commit(&kfree[b]);
                }
            } else if (lane == 0) {
                for (int c = 0; w && c < n; ++c) {
                    const long long g = g0 + c;
                    const int b = (int)(g & 1);
                    const uint32_t ph = (uint32_t)((g >> 1) & 1);
                    w = mbar_wait_bounded(&p_full[b], ph, p.err) && mbar_wait_bounded(&vfull[b], ph, p.err);
                    if (!w) break;
                    tc5_fence_after_sync();
                    const uint64_t vb = b ? dv1 : dv0;
#pragma unroll
                    for (int ks = 0; ks < TC_KEYS / 16; ++ks)      // 16 keys = 2048 bytes
                        tc5_mma_ta(tO, tP + 32 * b + 8 * ks, vb + (uint32_t)(ks * 2048 >> 4), ID_O,
                                   (c > 0 || ks > 0) ? 1u : 0u);
                    tc5_commit(&pv_done[b]);
                }
            }
            mok = __shfl_sync(0xffffffffu, w, 0);
            g0 += n;
        }
        // MMAs may still be running (after a timeout): wait for them (both warps)
        if (lane == 0) {
            tc5_commit(mma_idle);
            mbar_wait_bounded(mma_idle, 0, p.err);
        }
    } else {
        // ---- softmax: thread tid owns row tid of every item
        const uint32_t lane_base = (uint32_t)(warp * 32) << 16;   // this warp's TMEM lanes
        const float sl2 = p.scale_log2;
        long long g = 0;
        bool ok = true;
        Item it;
        for (int k = 0; ok && item_at(k, it); ++k) {
            const int n = it.nsteps;
            const int r = tid;
            const bool row_ok = r < it.nrows;
            const int rr = it.grp * TC_ROWS + r;
            const int tok = rr / G, head = rr % G;
            // last visible position; rows past the run see what its last row
            // sees; in a cascade chunk every row sees every key
            const int lim = cascade ? it.L - 1 : it.L - it.nq + min(tok, it.nq - 1);
            float m_run = -INFINITY, l_run = 0.f;
            float m_max = -INFINITY;               // largest score (log2 units, scaled)
            for (int c = 0; c < n; ++c, ++g) {
                const int b = (int)(g & 1);
                const uint32_t ph = (uint32_t)((g >> 1) & 1);
                const bool got = mbar_wait_bounded(s_full, (uint32_t)(g & 1), p.err);
                if (!__all_sync(0xffffffffu, got)) { ok = false; break; }
                tc5_fence_after_sync();

                // -- this row's 64 scores (then the S buffer is free for the
                // next step's S); the causal mask only where some row needs it
                float sv[TC_KEYS];
                tc5_ld64u(tS + lane_base, *reinterpret_cast<uint32_t(*)[TC_KEYS]>(&sv[0]));
                tc5_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(s_free);
                const int nvis = lim - c * TC_KEYS + 1;      // positions of this step the row sees
                if (__any_sync(0xffffffffu, nvis < TC_KEYS)) {
#pragma unroll
                    for (int e = 0; e < TC_KEYS; ++e) sv[e] = e < nvis ? sv[e] : -INFINITY;
                }
                float m4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
                for (int e = 0; e < TC_KEYS; e += 8) {
                    m4[0] = max3f(m4[0], sv[e], sv[e + 1]);
                    m4[1] = max3f(m4[1], sv[e + 2], sv[e + 3]);
                    m4[2] = max3f(m4[2], sv[e + 4], sv[e + 5]);
                    m4[3] = max3f(m4[3], sv[e + 6], sv[e + 7]);
                }
                const float mxs = max3f(m4[0], m4[1], fmaxf(m4[2], m4[3])) * sl2;
                m_max = fmaxf(m_max, mxs);
                // lazy rescaling: the reference level moves only by more than 2^RESCALE_LOG2
                const float m_new = mxs > m_run + RESCALE_LOG2 ? mxs : m_run;
                const float ms = m_new == -INFINITY ? 0.f : m_new;
                const float alpha = m_new == m_run ? 1.f : ex2(m_run - ms);
                // probabilities 2^(s * scale_log2 - m), two lanes per instruction
                uint32_t pw[TC_KEYS / 2];
                float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f),
                                 make_float2(0.f, 0.f)};
                const float2 sc2 = make_float2(sl2, sl2), nm2 = make_float2(-ms, -ms);
#pragma unroll
                for (int e = 0; e < TC_KEYS / 2; ++e) {
                    const float2 x = fma2(make_float2(sv[2 * e], sv[2 * e + 1]), sc2, nm2);
                    const float2 pe = make_float2(ex2(x.x), ex2(x.y));
                    pw[e] = Mma<T>::pack(pe.x, pe.y);
                    acc[e & 3] = add2(acc[e & 3], pe);
                }
                const float2 a2 = add2(add2(acc[0], acc[1]), add2(acc[2], acc[3]));
                l_run = l_run * alpha + (a2.x + a2.y);
                m_run = m_new;
                // this row of O to the new level, once P.V(g-1) is done (O holds
                // nothing before the item's first P.V)
                if (__any_sync(0xffffffffu, c > 0 && alpha != 1.f)) {
                    const long long gp = g - 1;
                    const bool done = mbar_wait_bounded(&pv_done[gp & 1], (uint32_t)((gp >> 1) & 1), p.err);
                    if (!__all_sync(0xffffffffu, done)) { ok = false; break; }
                    tc5_fence_after_sync();
                    const float f = c > 0 ? alpha : 1.f;
#pragma unroll
                    for (int c0 = 0; c0 < D; c0 += 32) {
                        float o[32];
                        tc5_ld32(tO + lane_base + c0, o);
#pragma unroll
                        for (int e = 0; e < 32; ++e) o[e] *= f;
                        tc5_st32(tO + lane_base + c0, o);
                    }
                }
                // P into buffer b once P.V(g-2) has read it (waits for the store)
                if (g >= 2) {
                    const bool freed = mbar_wait_bounded(&pv_done[b], (uint32_t)(((g >> 1) - 1) & 1), p.err);
                    if (!__all_sync(0xffffffffu, freed)) { ok = false; break; }
                    tc5_fence_after_sync();
                }
                tc5_st32u(tP + 32 * b + lane_base, pw);
                // V rows of the sequence's last block past L hold other tokens' data
                // (zero-weighted, but 0 * NaN is NaN): clear them once V has landed
                const int tail = it.L & 15, bl = it.nb_seq - 1 - (TC_KEYS / 16) * c;
                if (tail != 0 && bl >= 0 && bl < TC_KEYS / 16) {
                    const bool landed = mbar_wait_bounded(&vfull[b], ph, p.err);
                    if (!__all_sync(0xffffffffu, landed)) { ok = false; break; }
                    unsigned char *dV = sV + (size_t)b * KVB;
                    const int nclr = (16 - tail) * NH * 8;     // 16-byte pieces
                    for (int i = tid; i < nclr; i += TC_SOFTMAX_WARPS * 32) {
                        const int h = i / ((16 - tail) * 8), rem = i % ((16 - tail) * 8);
                        const int row = 16 * bl + tail + rem / 8;
                        *reinterpret_cast<uint4 *>(dV + h * (TC_KEYS * 128) + row * 128 + (rem % 8) * 16) =
                            make_uint4(0, 0, 0, 0);
                    }
                    fence_proxy_async_smem();              // the cleared rows before the MMA
                }
                tc5_fence_before_sync();
                __syncwarp();
                if (lane == 0) mbar_arrive(&p_full[b]);
            }
            if (!ok) break;

            // -- O / l into out (this thread's row), once the item's last P.V is done
            const long long gl = g - 1;
            const bool done = mbar_wait_bounded(&pv_done[gl & 1], (uint32_t)((gl >> 1) & 1), p.err);
            if (!__all_sync(0xffffffffu, done)) { ok = false; break; }
            tc5_fence_after_sync();
            const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
            if (cascade) {
                // chunk it.s of (sequence tok, head j*G + head): o = O / l, and
                // (m, l) taken to the true maximum, m in natural units
                const long long prow = ((long long)tok * H + it.j * G + head) * p.max_parts + it.s;
#pragma unroll
                for (int c0 = 0; c0 < D; c0 += 32) {
                    float v[32];
                    tc5_ld32(tO + lane_base + c0, v);
                    if (row_ok) {
                        float *po = p.part_o + prow * D + c0;
#pragma unroll
                        for (int e = 0; e < 32; e += 4)
                            *reinterpret_cast<float4 *>(po + e) =
                                make_float4(v[e] * inv, v[e + 1] * inv, v[e + 2] * inv, v[e + 3] * inv);
                    }
                }
                if (row_ok) {
                    p.part_m[prow] = m_max * LN2;
                    p.part_l[prow] = l_run * ex2(m_run - m_max);
                }
                tc5_fence_before_sync();
                continue;
            }
            T *o = reinterpret_cast<T *>(p.out) + ((long long)(it.q0 + tok) * H + it.j * G + head) * D;
#pragma unroll
            for (int c0 = 0; c0 < D; c0 += 32) {
                float v[32];
                tc5_ld32(tO + lane_base + c0, v);
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
            // O read before the next item's first P.V overwrites it (that P.V
            // waits for this warp's next arrival)
            tc5_fence_before_sync();
        }
    }

    tc5_fence_before_sync();
    __syncthreads();
    if (warp == 0) tc5_dealloc(tmem, TC_TMEM_COLS);
}

template <typename T, int D, int G>
cudaError_t launch_prefill_tc(const DecodeParams &p, const CUtensorMap &tmap_q, int groups,
                              cudaStream_t st) {
    using Lay = PrefillTcLayout<T, D>;
    constexpr size_t smem = Lay::BYTES;
    static_assert(TC_BLOCKS_PER_SM * (smem + sizeof(PrefillSched) + 1024) <= 228 * 1024,
                  "two blocks per SM");
    auto kern = prefill_tc_kernel<T, D, G>;
    static std::atomic<bool> attr_set[64];    // per device, read by any host thread
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64 || !attr_set[dev].load(std::memory_order_acquire)) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (dev >= 0 && dev < 64) attr_set[dev].store(true, std::memory_order_release);
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
    if (p.prefix_nblocks > 0) {                    // cascade prefix: its items
        const long long nrg = ((long long)p.num_seqs * G + TC_ROWS - 1) / TC_ROWS;
        const long long nch = (p.prefix_nblocks + p.prefix_chunk_blocks - 1) / p.prefix_chunk_blocks;
        if (blocks > nch * p.num_kv_heads * nrg) blocks = nch * p.num_kv_heads * nrg;
    } else {
        if (blocks > worst) blocks = worst;
        if (blocks > bound) blocks = bound;
    }
    if (blocks <= 0) return cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)blocks, 1, 1);
    cfg.blockDim = dim3(TC_THREADS, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, kern, p, tmap_q, groups);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

template <typename T>
cudaError_t dispatch_prefill_tc(const DecodeParams &p, const CUtensorMap &tmap_q, int D, int G,
                                int groups, cudaStream_t st) {
#define PA_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_prefill_tc<T, DD, GG>(p, tmap_q, groups, st);
    PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 4) PA_CASE(64, 8)
    PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 4) PA_CASE(128, 8)
#undef PA_CASE
    return cudaErrorNotSupported;
}

}  // namespace pa
