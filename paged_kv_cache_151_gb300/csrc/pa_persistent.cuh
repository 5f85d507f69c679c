// pa_persistent.cuh -- persistent decode kernel: resident thread blocks,
// grouped in thread-block clusters, stream a balanced list of work units end
// to end.
//
// A work unit is (sequence, KV head) for pa_decode, or (sequence, KV head,
// token partition) for pa_decode_partitioned.  Every block:
//
//  1. reads all seq_lens and sorts the sequences by block count, longest
//     first (bitonic sort in shared memory; ties by index, so the order is
//     deterministic);
//  2. numbers the units in that order; cluster c of the NC clusters takes
//     ranks c, 2NC-1-c, 2NC+c, ... ("snake" order), which deals the longest
//     units out first and evens the per-cluster totals;
//  3. concatenates the 16-token blocks of its cluster's units into one
//     stream of F blocks and gives warp g of the cluster's C*NW warps the
//     contiguous range [g*F/(C*NW), (g+1)*F/(C*NW)): every warp gets the same
//     number of blocks (to one), and a long unit spreads over several warps
//     and SMs.  Each warp keeps a ring of S stages filled with bulk copies
//     (tensor-map copies of whole swizzled tiles for 16-bit caches, 1-D
//     copies of the valid rows for fp32) of its next blocks' K and V, running
//     ahead across unit boundaries;
//  4. a unit that lies inside one warp's range is finished by that warp
//     alone.  A unit that crosses range boundaries leaves one partial
//     (m, l, acc) per warp that touched it -- each warp has one slot for the
//     unit it starts in and one for the unit it ends in, so slots are never
//     reused -- and the last of those warps to arrive (an atomic counter of
//     the unit's first warp, in distributed shared memory when the warps
//     span several blocks) merges the partials in warp order and writes the
//     unit's output (pa_decode) or partition statistics
//     (pa_decode_partitioned).  No warp ever waits for another.
//
// Everything a unit's result depends on -- the unit order, the block ranges,
// the merge order -- is a function of seq_lens and logical block indices
// only, never of where the blocks sit in the pool, so outputs are
// bit-identical under any permutation of physical blocks and under prefix
// aliasing.
#pragma once

#include <atomic>
#include <type_traits>

#include "pa_common.cuh"
#include "pa_decode.cuh"
#include "pa_fp8.cuh"
#include "pa_math.cuh"
#include "pa_mma.cuh"

namespace pa {

// What a launch computes: whole-sequence decode (one query token per
// sequence), split-KV partitions, or several query tokens per sequence.
enum Mode : int { MODE_DECODE = 0, MODE_PARTITIONED = 1, MODE_MULTI = 2 };

// Rows of one unit's query tile: the G heads of one token, or for multi-token
// queries 16 (token, head) pairs.
__host__ __device__ constexpr int rows_of_mode(int mode, int G) { return mode == MODE_MULTI ? 16 : G; }

struct UnitRec {
    int s, j, lb0, nb, L, part;   // part: partition (partitioned) or row tile (multi)
    int q0, nq;                   // multi: first query row of the sequence, its count
};

// Shared-memory layout; KV is the cache's storage type (T itself, or E4M3).
template <typename T, typename KV, int D, int G, int NW, int S, int MODE>
struct PersistentLayout {
    static constexpr bool PARTIAL = MODE == MODE_PARTITIONED;
    static constexpr int ROWS = rows_of_mode(MODE, G);
    static constexpr size_t TILE_BYTES = (size_t)16 * D * sizeof(KV);
    static constexpr int NU_MAX = 128;                    // units per cluster
    static constexpr size_t STAGES = (size_t)NW * S * 2 * TILE_BYTES;
    // one partial: O[ROWS][D], M[ROWS], L[ROWS], padded to 16 bytes
    static constexpr size_t PART_FLOATS = ((size_t)ROWS * D + 2 * ROWS + 3) / 4 * 4;
    static constexpr size_t OFF_BARS = STAGES;
    static constexpr size_t OFF_SCR = OFF_BARS + (size_t)NW * S * 8;
    // per-warp score scratch of the CUDA-core path (16-bit caches use none)
    static constexpr size_t SCR_BYTES = sizeof(T) == 2 ? 0 : (size_t)NW * warp_scratch_floats<G>() * 4;
    static constexpr size_t OFF_PARTS = OFF_SCR + SCR_BYTES;
    static constexpr size_t OFF_UNITS = OFF_PARTS + (size_t)NW * PART_FLOATS * 4;
    static constexpr size_t OFF_CUM = OFF_UNITS + (size_t)NU_MAX * sizeof(UnitRec);
    static constexpr size_t OFF_CTL = (OFF_CUM + (size_t)(NU_MAX + 1) * 4 + 15) / 16 * 16;
    // control words: arrival counters [NW], scan scratch [2*NW] (64-bit
    // values), warp ranges of the cluster's stream [16*NW + 1] (clusters of up
    // to 16 blocks)
    static constexpr size_t CTL_BYTES = ((size_t)(3 * NW + 16 * NW + 1) * 4 + 15) / 16 * 16;
    static constexpr size_t BYTES = OFF_CTL + CTL_BYTES + 1024;   // + alignment of the base
    static_assert(STAGES % 1024 == 0, "stage buffers: 1024-byte aligned boxes");
    static_assert(S == 0 || (size_t)S * 2 * TILE_BYTES >= PART_FLOATS * 4,
                  "a warp's stages must hold one partial");
    static_assert(OFF_SCR % 16 == 0 && OFF_PARTS % 16 == 0 && OFF_UNITS % 16 == 0 &&
                      OFF_CTL % 16 == 0 && PART_FLOATS % 4 == 0,
                  "shared-memory regions must stay 16-byte aligned");
    // the sort scratch (keys padded to a power of two >= the thread count,
    // scan, lengths) lives in the stage region before streaming: at most 16
    // bytes per sequence
    static constexpr int MAX_SEQS = (int)(STAGES / 16) > 65535 ? 65535 : (int)(STAGES / 16);
};

// In-thread compare-exchange of a bitonic network stage with stride J < EPT
// (elements t*EPT .. t*EPT+EPT-1 in registers).
template <int EPT, int J>
__device__ __forceinline__ void bitonic_local(uint32_t (&v)[EPT], int t, int k) {
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        const int e2 = e ^ J;
        if (e2 > e) {
            const bool up = ((t * EPT + e) & k) == 0;
            const uint32_t a = v[e], b = v[e2];
            if ((a > b) == up) { v[e] = b; v[e2] = a; }
        }
    }
}

// Ascending bitonic sort of keys[0 .. EPT*NT) (distinct values), EPT per
// thread in registers: strides inside a thread are register swaps, strides
// inside a warp are shuffles, and only strides that cross warps go through
// shared memory.
template <int EPT, int NT>
__device__ __forceinline__ void bitonic_sort_regs(uint32_t *keys) {
    constexpr int N = EPT * NT;
    const int t = threadIdx.x;
    uint32_t v[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) v[e] = keys[t * EPT + e];
    for (int k = 2; k <= N; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            if (jj < EPT) {
                if constexpr (EPT > 1) { if (jj == 1) bitonic_local<EPT, 1>(v, t, k); }
                if constexpr (EPT > 2) { if (jj == 2) bitonic_local<EPT, 2>(v, t, k); }
                if constexpr (EPT > 4) { if (jj == 4) bitonic_local<EPT, 4>(v, t, k); }
            } else if (jj < 32 * EPT) {
                const int m = jj / EPT;
                const bool lower = (t & m) == 0;
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    const bool up = ((t * EPT + e) & k) == 0;
                    const uint32_t b = __shfl_xor_sync(0xffffffffu, v[e], m);
                    v[e] = (lower == up) ? min(v[e], b) : max(v[e], b);
                }
            } else {
#pragma unroll
                for (int e = 0; e < EPT; ++e) keys[t * EPT + e] = v[e];
                __syncthreads();
#pragma unroll
                for (int e = 0; e < EPT; ++e) {
                    const int i = t * EPT + e, ixj = i ^ jj;
                    const uint32_t b = keys[ixj];
                    const bool up = (i & k) == 0;
                    v[e] = ((i < ixj) == up) ? min(v[e], b) : max(v[e], b);
                }
                __syncthreads();
            }
        }
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) keys[t * EPT + e] = v[e];
    __syncthreads();
}

// Ascending sort of keys[0 .. N) (distinct values) by counting: each key's
// position is the number of smaller keys.  EPT keys per thread compared
// against all N (broadcast reads); out receives the sorted keys.
template <int EPT, int NT>
__device__ __forceinline__ void rank_sort(const uint32_t *keys, uint32_t *out) {
    constexpr int N = EPT * NT;
    const int t = threadIdx.x;
    uint32_t v[EPT];
    int rk[EPT];
#pragma unroll
    for (int e = 0; e < EPT; ++e) {
        v[e] = keys[t * EPT + e];
        rk[e] = 0;
    }
    const uint4 *k4 = reinterpret_cast<const uint4 *>(keys);
#pragma unroll 4
    for (int i = 0; i < N / 4; ++i) {
        const uint4 w = k4[i];
#pragma unroll
        for (int e = 0; e < EPT; ++e)
            rk[e] += (w.x < v[e]) + (w.y < v[e]) + (w.z < v[e]) + (w.w < v[e]);
    }
#pragma unroll
    for (int e = 0; e < EPT; ++e) out[rk[e]] = v[e];
    __syncthreads();
}

// Ascending bitonic sort of keys[0 .. Np) (Np a power of two >= NT).
template <int NT>
__device__ void sort_keys_bitonic(uint32_t *keys, int Np) {
    if (Np == NT) { bitonic_sort_regs<1, NT>(keys); return; }
    if (Np == 2 * NT) { bitonic_sort_regs<2, NT>(keys); return; }
    if (Np == 4 * NT) { bitonic_sort_regs<4, NT>(keys); return; }
    if (Np == 8 * NT) { bitonic_sort_regs<8, NT>(keys); return; }
    const int tid = threadIdx.x;                   // larger batches: shared memory only
    for (int k = 2; k <= Np; k <<= 1) {
        for (int jj = k >> 1; jj > 0; jj >>= 1) {
            for (int i = tid; i < Np; i += NT) {
                const int ixj = i ^ jj;
                if (ixj > i) {
                    const uint32_t a = keys[i], b = keys[ixj];
                    const bool up = (i & k) == 0;
                    if ((a > b) == up) { keys[i] = b; keys[ixj] = a; }
                }
            }
            __syncthreads();
        }
    }
}

// Ascending sort of keys[0 .. Np) (Np a power of two >= NT, distinct values);
// `tmp` has room for Np keys.  Returns the array holding the result.
template <int NT>
__device__ uint32_t *sort_keys(uint32_t *keys, uint32_t *tmp, int Np) {
    if (Np == NT) { rank_sort<1, NT>(keys, tmp); return tmp; }
    if (Np == 2 * NT) { rank_sort<2, NT>(keys, tmp); return tmp; }
    sort_keys_bitonic<NT>(keys, Np);
    return keys;
}

// Exclusive scan of one int per thread across the block; returns this
// thread's exclusive prefix and writes the total to *total.
template <int NT>
__device__ __forceinline__ int block_exclusive_scan(int v, int *wtot, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    int x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    int before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const int t = wtot[w];
        if (w < warp) before += t;
        all += t;
    }
    __syncthreads();
    *total = all;
    return before + x - v;
}

// The same for one 64-bit value per thread; wtot holds NT/32 values.
template <int NT>
__device__ __forceinline__ long long block_exclusive_scan64(long long v, long long *wtot,
                                                            long long *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    long long x = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const long long y = __shfl_up_sync(0xffffffffu, x, o);
        if (lane >= o) x += y;
    }
    if (lane == 31) wtot[warp] = x;
    __syncthreads();
    long long before = 0, all = 0;
#pragma unroll
    for (int w = 0; w < NT / 32; ++w) {
        const long long t = wtot[w];
        if (w < warp) before += t;
        all += t;
    }
    __syncthreads();
    *total = all;
    return before + x - v;
}

// 16-bit caches use the tensor cores (pa_mma.cuh) on swizzled tiles placed
// by tensor-map copies of whole 16-row blocks; fp32 caches use the CUDA-core
// path (pa_math.cuh) on tiles placed by 1-D copies of the valid rows.
template <typename T>
__host__ __device__ constexpr bool use_tc() { return sizeof(T) == 2; }

#ifndef PA_DECODE_PDL
#define PA_DECODE_PDL 1
#endif

#ifndef PA_F8_BLOCKS_PER_SM
#define PA_F8_BLOCKS_PER_SM 3
#endif

// What a warp pays to enter a unit (load its query, park or write its
// result), in quarters of one 16-token block; used to split the stream.
#ifndef PA_UNIT_COST_Q4
#define PA_UNIT_COST_Q4 4
#endif

// T: the type of q and out; KV: the caches' storage (T, or E4M3 codes with
// per-KV-head scales, 16-bit T only).
// Warps per block: whole-sequence decode and multi-token queries over 16-bit
// caches run one block of eight warps per SM (the set-up, done once per block,
// then serves all eight); partitions, fp32 and E4M3 caches run blocks of four.
#ifndef PA_DECODE_WARPS
#define PA_DECODE_WARPS 8
#endif
template <typename KV, int MODE>
__host__ __device__ constexpr int persistent_warps() {
    return (sizeof(KV) == 2 && (MODE == MODE_DECODE || MODE == MODE_MULTI)) ? PA_DECODE_WARPS : 4;
}

// Blocks per SM the kernel is built for: eight warps of 16-bit tiles per SM
// (one block of eight or two of four); E4M3 tiles are half the bytes, so
// three blocks of four fit and hide more latency.
template <typename KV, int NW>
__host__ __device__ constexpr int persistent_blocks_per_sm() {
    return sizeof(KV) == 1 ? PA_F8_BLOCKS_PER_SM : (NW >= 8 ? 1 : 2);
}

template <typename T, typename KV, int D, int G, int NW, int S, int MODE>
__global__ void __launch_bounds__(NW * 32, (persistent_blocks_per_sm<KV, NW>()))
decode_persistent_kernel(const __grid_constant__ DecodeParams p) {
    constexpr bool TC = use_tc<T>();
    constexpr bool F8 = std::is_same<KV, e4m3>::value;
    constexpr bool PARTIAL = MODE == MODE_PARTITIONED;
    constexpr bool MQ = MODE == MODE_MULTI;
    constexpr int ROWS = rows_of_mode(MODE, G);
    static_assert(!MQ || TC, "multi-token queries use the tensor-core path");
    static_assert(F8 || std::is_same<KV, T>::value, "cache type");
    static_assert(!F8 || (TC && !MQ), "E4M3 caches: 16-bit q, one query token per sequence");
    using W = std::conditional_t<
        F8, WarpAttnF8<T, D, G>,
        std::conditional_t<MQ, WarpAttnTC16<T, D>,
                           std::conditional_t<TC, WarpAttnTC<T, D, G>, WarpAttn<T, D, G>>>>;
    using Lay = PersistentLayout<T, KV, D, G, NW, S, MODE>;
    using Sh = Shape<T, D>;                        // chunks of q / out
    constexpr int E = Sh::E;
    constexpr int ROWB = D * (int)sizeof(KV), TILE = 16 * ROWB;   // cache rows and tiles
    constexpr int NT = NW * 32;
    constexpr int NU_MAX = Lay::NU_MAX;
    constexpr int WS = warp_scratch_floats<G>();
    constexpr int PF = (int)Lay::PART_FLOATS;
    constexpr int UNIT_COST = PA_UNIT_COST_Q4;     // quarter blocks charged per unit

    extern __shared__ __align__(1024) unsigned char smem_raw[];
    // the 128-byte swizzle pattern is tied to 1024-byte aligned addresses
    unsigned char *smem = smem_raw + ((1024 - (smem_u32(smem_raw) & 1023)) & 1023);
    unsigned char *stages = smem;
    uint64_t *bars = reinterpret_cast<uint64_t *>(smem + Lay::OFF_BARS);
    float *scr = reinterpret_cast<float *>(smem + Lay::OFF_SCR);
    float *parts = reinterpret_cast<float *>(smem + Lay::OFF_PARTS);   // [NW][PF]
    UnitRec *units = reinterpret_cast<UnitRec *>(smem + Lay::OFF_UNITS);
    int *cum = reinterpret_cast<int *>(smem + Lay::OFF_CUM);
    int *ctl = reinterpret_cast<int *>(smem + Lay::OFF_CTL);
    int *arrive = ctl;                       // [NW] warps done with the unit that
                                             //      starts in this warp's range
    int *wtot = ctl + NW;                    // [2*NW] scan scratch (NW 64-bit values)
    int *bound = ctl + 3 * NW;               // [C*NW + 1] warp ranges of the stream

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int B = p.num_seqs, Hkv = p.num_kv_heads, H = p.num_heads;
    const int cap = PARTIAL ? min(p.max_seq_len, p.max_blocks * 16) : p.max_blocks * 16;
    const int PB = PARTIAL ? p.partition_blocks : 1;
    const int C = (int)cluster_nctarank(), rank = (int)cluster_ctarank();
    const int NWC = C * NW;                  // warps of the cluster
    const int gw = rank * NW + warp;         // this warp's index in the cluster

    // split-KV partitions are always followed by their merge, which waits for
    // this whole grid before it reads anything: let it become resident early
    if constexpr (PARTIAL) launch_dependents();

    // ---- 0. barriers, and the first reads after the set-up started early -----
    if (tid == 0) {
        if constexpr (TC) {                        // fetch the descriptors early
            prefetch_tensormap(&p.tmap_k);
            prefetch_tensormap(&p.tmap_v);
            if constexpr (!F8) {
                prefetch_tensormap(&p.tmap_k8);
                prefetch_tensormap(&p.tmap_v8);
            }
        }
        for (int i = 0; i < NW * S; ++i) mbar_init(&bars[i], 1);
        fence_mbar_init();
    }
    if (tid < NW) arrive[tid] = 0;
    // this block's arrival counters are initialised; peers wait for that
    // (cluster_wait below) before their first access to them.  Arriving now,
    // before any other memory traffic, keeps the release cheap.
    if (C > 1) cluster_arrive();

    // ---- 1. sort the sequences by block count (longest first) ----------------
    // multi-token queries: rows query_start[s] .. query_start[s+1]-1 belong to
    // sequence s; a range outside its bounds is flagged and gets no rows
    auto mq_valid = [&](int s, int L) -> bool {
        const int a = p.query_start[s], b = p.query_start[s + 1];
        return a >= 0 && b >= a && b <= p.num_q_rows && b - a <= p.max_query_len && b - a <= L;
    };
    int Bp = NT;
    while (Bp < B) Bp <<= 1;
    uint32_t *keys = reinterpret_cast<uint32_t *>(stages);           // [Bp]
    int *start = reinterpret_cast<int *>(stages + (size_t)Bp * 4);   // [B]
    int *lens = start + B;                                           // [B], clamped
    uint32_t *sort_tmp = reinterpret_cast<uint32_t *>(lens + ((B + 3) & ~3));  // [Bp] if Bp <= 2*NT
    for (int i = tid; i < Bp; i += NT) {
        uint32_t key = 0xffffffffu;
        if (i < B) {
            const int L0 = p.seq_lens[i];
            if ((L0 < 0 || L0 > cap) && blockIdx.x == 0) set_error(p.err, ERR_SEQ_LEN);
            const int L = L0 < 0 ? 0 : (L0 > cap ? cap : L0);
            lens[i] = L;
            if constexpr (MQ) {
                if (blockIdx.x == 0 && !mq_valid(i, L)) set_error(p.err, ERR_SEQ_LEN);
            }
            const int nb = (L + 15) >> 4;
            key = ((uint32_t)(0xffff - nb) << 16) | (uint32_t)i;
        }
        keys[i] = key;
    }
    // block tables, and the queries, are read as soon as the set-up is done:
    // start bringing them into L2 now that seq_lens, which everything waits
    // for, has arrived (at most 4 MiB of each; L2 is coherent, so this is safe
    // even while the previous kernel may still write q)
    {
        constexpr size_t PF_MAX = (size_t)4 << 20;
        const size_t bt_bytes = (size_t)B * p.max_blocks * 4;
        const size_t q_rows = MQ ? (size_t)p.num_q_rows : (size_t)B;   // rows of H x D
        const size_t q_bytes =
            q_rows > 0 ? ((q_rows - 1) * p.q_seq_stride + (size_t)H * D) * sizeof(T) : 0;
        prefetch_l2_range(p.block_tables, bt_bytes < PF_MAX ? bt_bytes : PF_MAX);
        prefetch_l2_range(p.q, q_bytes < PF_MAX ? q_bytes : PF_MAX);
    }
    __syncthreads();
    static_assert(Lay::STAGES >= 16 * 256, "the stage region holds the sort's scratch");
    if (Bp <= 256) {
        // up to 256 sequences: one warp sorts in registers (the others wait)
        if (warp == 0) {
            if (Bp == 256) warp_bitonic_sort<8>(keys, sort_tmp);
            else if (Bp == 128) warp_bitonic_sort<4>(keys, sort_tmp);
            else warp_bitonic_sort<2>(keys, sort_tmp);
        }
        __syncthreads();
        keys = sort_tmp;
    } else {
        keys = sort_keys<NT>(keys, sort_tmp, Bp);
    }

    // ---- 2. number the units ------------------------------------------------
    // One-token decode gives every sequence Hkv units, so unit r belongs to
    // sorted position r / Hkv; otherwise an exclusive scan of the units per
    // sorted sequence, searched per unit below.
    constexpr bool UNIFORM = !PARTIAL && !MQ;
    auto units_of = [&](int pos) -> int {          // pos < B
        const int nb = 0xffff - (int)(keys[pos] >> 16);
        if constexpr (MQ) {
            const int s = (int)(keys[pos] & 0xffffu);
            int nq = mq_valid(s, lens[s]) ? p.query_start[s + 1] - p.query_start[s] : 0;
            if (p.mq_split_rows > 0 && nq * G >= p.mq_split_rows) nq = 0;   // the prefill path's
            return Hkv * ((nq * G + 15) / 16);
        }
        return PARTIAL ? Hkv * ((nb + PB - 1) / PB) : Hkv;
    };
    int U = 0;
    if constexpr (UNIFORM) {
        U = B * Hkv;
    } else {
        const int per = (B + NT - 1) / NT;
        const int lo = min(B, tid * per), hi = min(B, lo + per);
        int sum = 0;
        for (int i = lo; i < hi; ++i) sum += units_of(i);
        int run = block_exclusive_scan<NT>(sum, wtot, &U);
        for (int i = lo; i < hi; ++i) {
            start[i] = run;
            run += units_of(i);
        }
        __syncthreads();
    }

    // ---- 3. this cluster's units (snake over the ranks) -----------------------
    const int NC = gridDim.x / C, me = blockIdx.x / C;
    auto rank_of = [&](int q) -> long long {
        return (long long)q * NC + ((q & 1) ? (NC - 1 - me) : me);
    };
    // ranks q*NC + (q even ? me : NC-1-me) below U: every full round, and the
    // partial last round if this cluster's offset falls inside it
    int nu = U / NC;
    if (rank_of(nu) < U) ++nu;
    if (nu > NU_MAX) {                             // the host sizes the grid to avoid this
        if (tid == 0) set_error(p.err, ERR_SEQ_LEN);
        nu = NU_MAX;
    }
    static_assert(NU_MAX <= NT, "one thread per unit");
    int nb_q = 0;                                  // thread q builds unit q
    if (tid < nu) {
        const int r = (int)rank_of(tid);
        int pos, local;
        if constexpr (UNIFORM) {
            pos = r / Hkv;
            local = r - pos * Hkv;
        } else {
            int lo = 0, hi = B - 1;                // last pos with start[pos] <= r
            while (lo < hi) {
                const int mid = (lo + hi + 1) >> 1;
                if (start[mid] <= r) lo = mid; else hi = mid - 1;
            }
            pos = lo;
            local = r - start[lo];
        }
        const int s = (int)(keys[pos] & 0xffffu);
        const int nb = 0xffff - (int)(keys[pos] >> 16);
        UnitRec u;
        u.s = s;
        u.L = lens[s];
        u.q0 = 0;
        u.nq = 1;
        if constexpr (MQ) {
            const int q0 = p.query_start[s], nq = p.query_start[s + 1] - q0;   // valid: it has units
            const int tiles = (nq * G + 15) / 16;
            u.j = local / tiles;
            u.part = local % tiles;
            u.q0 = q0;
            u.nq = nq;
            u.lb0 = 0;
            // the tile's last row sees positions up to L - nq + its token
            const int last_tok = min(16 * u.part + 15, nq * G - 1) / G;
            const int lim = u.L - nq + last_tok;             // >= 0: nq <= L
            u.nb = lim >= 0 ? lim / 16 + 1 : 0;
        } else if (PARTIAL) {
            const int ps = (nb + PB - 1) / PB;
            u.j = local / ps;
            u.part = local % ps;
            u.lb0 = u.part * PB;
            u.nb = min(PB, nb - u.lb0);
        } else {
            u.j = local;
            u.part = 0;
            u.lb0 = 0;
            u.nb = nb;
        }
        units[tid] = u;
        nb_q = u.nb;
    }
    // cum[q] = blocks before unit q.  The stream is split into C*NW ranges of
    // equal cost, a block costing 4 and each unit a warp enters a further
    // UNIT_COST (quarter blocks): in a virtual stream where every unit with
    // blocks starts with UNIT_COST/4 header blocks, the cuts fall at equal
    // steps, and the thread of the unit a cut falls in moves it to a real block.
    long long tot;
    const long long ex = block_exclusive_scan64<NT>(((long long)(nb_q > 0) << 32) | (unsigned)nb_q,
                                                    reinterpret_cast<long long *>(wtot), &tot);
    const int cum_q = (int)(ex & 0xffffffffLL), nz_before = (int)(ex >> 32);
    const int run = (int)(tot & 0xffffffffLL), nz = (int)(tot >> 32);
    if (tid < nu) cum[tid] = cum_q;
    if (tid == 0) {
        cum[nu] = run;
        bound[0] = 0;
        bound[NWC] = run;
    }
    const long long vtot = 4LL * run + (long long)nz * UNIT_COST;
    if (tid < nu && nb_q > 0) {
        const long long vs = 4LL * cum_q + (long long)nz_before * UNIT_COST;
        const long long ve = vs + 4LL * nb_q + UNIT_COST;
        // cuts g with floor(g * vtot / NWC) in [vs, ve)
        int g = (int)((vs * NWC + vtot - 1) / vtot);
        const long long g_end = (ve * NWC + vtot - 1) / vtot;
        if (g < 1) g = 1;
        for (; g < g_end && g < NWC; ++g) {
            const long long o = (long long)g * vtot / NWC - vs;
            bound[g] = o < UNIT_COST ? cum_q : min(cum_q + nb_q, cum_q + (int)((o - UNIT_COST) / 4));
        }
    }
    if (nz == 0)
        for (int g = 1 + tid; g < NWC; g += NT) bound[g] = run;
    // the sort scratch in the stage region is overwritten by bulk copies next
    fence_proxy_async_smem();
    __syncthreads();

    // ---- 4. stream this warp's range of the cluster's blocks ------------------
    auto range_lo = [&](int g) -> int { return bound[g]; };
    auto owner = [&](int f) -> int {               // warp whose range holds position f
        int lo = 0, hi = NWC - 1;                  // last warp starting at or before f
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (bound[mid] <= f) lo = mid; else hi = mid - 1;
        }
        return lo;
    };
    const int my_lo = range_lo(gw), my_hi = range_lo(gw + 1);
    const int n_mine = my_hi - my_lo;
    auto locate = [&](int f) -> int {              // unit holding stream position f
        int lo = 0, hi = nu - 1;
        while (lo < hi) {
            const int mid = (lo + hi + 1) >> 1;
            if (cum[mid] <= f) lo = mid; else hi = mid - 1;
        }
        return lo;
    };
    // lane i holds (unit, physical block) of this warp's block c0 + i and c0 + 32 + i
    auto fetch = [&](int k, int &ui, int &pb) {
        ui = -1;
        pb = 0;
        if (k < n_mine) {
            const int f = my_lo + k;
            ui = locate(f);
            const UnitRec &u = units[ui];
            const int lb = u.lb0 + (f - cum[ui]);
            pb = p.block_tables[(long long)u.s * p.max_blocks + lb];
        }
    };
    int c0 = 0, ui_cur, pb_cur, ui_nxt, pb_nxt;
    fetch(lane, ui_cur, pb_cur);
    fetch(32 + lane, ui_nxt, pb_nxt);
    auto of = [&](int k, int &ui, int &pb) {      // warp-uniform k
        const int kk = k - c0;
        const int a = __shfl_sync(0xffffffffu, ui_cur, kk & 31);
        const int b = __shfl_sync(0xffffffffu, ui_nxt, kk & 31);
        const int x = __shfl_sync(0xffffffffu, pb_cur, kk & 31);
        const int y = __shfl_sync(0xffffffffu, pb_nxt, kk & 31);
        ui = kk < 32 ? a : b;
        pb = kk < 32 ? x : y;
    };
    auto pos_of = [&](int k, int ui) -> int {     // sequence position of block k's row 0
        const UnitRec &u = units[ui];
        return (u.lb0 + (my_lo + k - cum[ui])) * 16;
    };
    auto rows_of = [&](int k, int ui) -> int { return min(16, units[ui].L - pos_of(k, ui)); };

    unsigned char *my_stages = stages + (size_t)warp * S * 2 * TILE;
    uint64_t *my_bars = bars + warp * S;
    const uint64_t pol = policy_evict_first();
    const unsigned char *kbase = reinterpret_cast<const unsigned char *>(p.k_cache);
    const unsigned char *vbase = reinterpret_cast<const unsigned char *>(p.v_cache);
    // test hook: each warp's first stage never completes, so its wait runs out
    const uint32_t stall = p.test_stall ? 16u : 0u;
    auto issue = [&](int k, int ui, int pbk) {     // lane 0 only
        uint64_t *bar = &my_bars[k % S];
        const uint32_t extra = k == 0 ? stall : 0u;
        if (pbk < 0 || (long long)pbk >= p.num_blocks) {
            set_error(p.err, ERR_BLOCK_ID);
            mbar_arrive(bar);
            return;
        }
        unsigned char *dst = my_stages + (size_t)(k % S) * 2 * TILE;
        if constexpr (F8) {
            // whole 16-row tiles, one box of 16 rows x D bytes each
            const int z = pbk * Hkv + units[ui].j;
            mbar_arrive_expect_tx(bar, 2 * TILE + extra);
            tma_load_3d(dst, &p.tmap_k, 0, 0, z, bar, pol);
            tma_load_3d(dst + TILE, &p.tmap_v, 0, 0, z, bar, pol);
        } else if constexpr (TC) {
            // 16-row tiles, D/64 boxes each for K and V; a block with at most 8
            // valid tokens takes boxes of 8 rows (the rest of the stage keeps
            // stale rows, which the block math masks or clears)
            const int z = pbk * Hkv + units[ui].j;
            const bool half = rows_of(k, ui) <= 8;
            mbar_arrive_expect_tx(bar, (half ? TILE : 2 * TILE) + extra);
            const CUtensorMap *mk = half ? &p.tmap_k8 : &p.tmap_k;
            const CUtensorMap *mv = half ? &p.tmap_v8 : &p.tmap_v;
#pragma unroll
            for (int h = 0; h < D / 64; ++h) {
                tma_load_3d(dst + h * 2048, mk, h * 64, 0, z, bar, pol);
                tma_load_3d(dst + TILE + h * 2048, mv, h * 64, 0, z, bar, pol);
            }
        } else {
            const uint32_t bytes = (uint32_t)(rows_of(k, ui) * ROWB);
            const size_t off = ((size_t)pbk * Hkv + units[ui].j) * TILE;
            mbar_arrive_expect_tx(bar, 2 * bytes + extra);
            bulk_g2s(dst, kbase + off, bytes, bar, pol);
            bulk_g2s(dst + TILE, vbase + off, bytes, bar, pol);
        }
    };

    // Everything above reads only seq_lens, query_start and block_tables.
    // The caches (and q, out) are touched only after the kernel before this
    // one in the stream -- typically the cache write of the same step, which
    // lets this kernel start early -- has completed.
    grid_dependency_wait();

    // units with no tokens (pa_decode only): their output is zero
    if (!PARTIAL && !MQ && rank == 0 && warp == NW - 1) {
        for (int q = 0; q < nu; ++q) {
            const UnitRec u = units[q];
            if (u.nb != 0) continue;
            T *o = reinterpret_cast<T *>(p.out) + ((long long)u.s * H + u.j * G) * D;
            for (int i = lane; i < G * D / E; i += 32) {
                float z[E];
#pragma unroll
                for (int e = 0; e < E; ++e) z[e] = 0.f;
                store_chunk<T>(o + i * E, z);
            }
        }
    }

    const int pre = n_mine < S ? n_mine : S;
    for (int k = 0; k < pre; ++k) {
        int ui, pbk;
        of(k, ui, pbk);
        if (lane == 0) issue(k, ui, pbk);
    }

    W wa;
    wa.init(lane);
    float *Sc = scr + warp * WS;
    float *Pb = Sc + 16 * G;
    float *Al = Pb + 16 * G;

    // Partial slots of warp g (in block g / NW).  Slot 0 holds the unit the
    // warp's range starts inside of (shared with earlier warps and ending in
    // this range), written while the warp streams on, so it has its own
    // space.  Slot 1 holds the unit that runs past the end of the range: the
    // warp's last unit, written when its ring is idle, so it lives in the
    // warp's stage buffers.  (Units wholly inside the range are written from
    // registers.)
    auto part_of = [&](int g, int which) -> float * {
        return which == 0 ? parts + (size_t)(g % NW) * PF
                          : reinterpret_cast<float *>(stages + (size_t)(g % NW) * S * 2 * TILE);
    };

    // V's dequantisation scale of unit u (E4M3 caches), applied to results
    auto v_scale_of = [&](const UnitRec &u) -> float {
        if constexpr (F8) return __ldg(p.v_scale + u.j);
        else return 1.f;
    };

    // Output row (in units of D) of row r of unit u's query tile; -1 if the
    // tile's row is past the sequence's query rows.
    auto out_row = [&](const UnitRec &u, int r) -> long long {
        if constexpr (MQ) {
            const int rr = 16 * u.part + r;
            if (rr >= u.nq * G) return -1;
            return (long long)(u.q0 + rr / G) * H + u.j * G + rr % G;
        } else {
            return (long long)u.s * H + u.j * G + r;
        }
    };

    // Write the result of unit u from a merged (M, L, O) of chunk (g, d0).
    auto emit = [&](const UnitRec &u, int g, int d0, float M, float Ls, float *O) {
        const float inv = Ls > 0.f ? v_scale_of(u) / Ls : 0.f;
        if constexpr (PARTIAL) {
            const long long row = ((long long)u.s * H + u.j * G + g) * p.max_parts + u.part;
            float *po = p.part_o + row * D + d0;
#pragma unroll
            for (int e = 0; e < E; e += 4)
                *reinterpret_cast<float4 *>(po + e) =
                    make_float4(O[e] * inv, O[e + 1] * inv, O[e + 2] * inv, O[e + 3] * inv);
            if (d0 == 0) {
                p.part_m[row] = M * LN2;          // natural units
                p.part_l[row] = Ls;
            }
        } else {
#pragma unroll
            for (int e = 0; e < E; ++e) O[e] *= inv;
            T *o = reinterpret_cast<T *>(p.out) + out_row(u, g) * D + d0;
            store_chunk<T>(o, O);
        }
    };

    // Merge every partial of unit `ui` (in warp order) and write the unit's
    // result; run by the last of the unit's warps to arrive.
    auto merge_unit = [&](int ui) {
        const UnitRec u = units[ui];
        const int g_first = owner(cum[ui]), g_last = owner(cum[ui] + u.nb - 1);
        {
            // Merge the unit's partials in warp order with a running maximum.
            // A lane owns chunks lane, lane + 32, ... (E outputs each), taken
            // CG at a time; all loads of one partial for those chunks are
            // issued before any is used, so each partial costs one round trip
            // to cluster shared memory rather than one per load.
            constexpr int NCH = ROWS * (D / E);
            constexpr int CPL = (NCH + 31) / 32;
            constexpr int CG = CPL < 16 / E ? CPL : (16 / E > 0 ? 16 / E : 1);
#pragma unroll 1
            for (int c0g = 0; c0g < CPL; c0g += CG) {
                float M[CG], Ls[CG], O[CG][E];
                int gg[CG], dd[CG];
#pragma unroll
                for (int c = 0; c < CG; ++c) {
                    const int ch = lane + 32 * (c0g + c);
                    const int chv = ch < NCH ? ch : 0;     // out-of-range chunks read chunk 0
                    gg[c] = chv / (D / E);
                    dd[c] = (chv % (D / E)) * E;
                    M[c] = -INFINITY;
                    Ls[c] = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) O[c][e] = 0.f;
                }
                for (int w = g_first; w <= g_last; ++w) {
                    if (range_lo(w) == range_lo(w + 1)) continue;
                    const float *pw = part_of(w, (w == g_last && w != g_first) ? 0 : 1);
                    const uint32_t rw = (uint32_t)(w / NW);
                    float mw[CG], lw[CG];
                    float4 ow[CG][E / 4];
#pragma unroll
                    for (int c = 0; c < CG; ++c) {
                        mw[c] = ld_dsmem_f32(map_to_rank(pw + ROWS * D + gg[c], rw));
                        lw[c] = ld_dsmem_f32(map_to_rank(pw + ROWS * D + ROWS + gg[c], rw));
#pragma unroll
                        for (int e = 0; e < E / 4; ++e)
                            ow[c][e] = ld_dsmem_f32x4(map_to_rank(pw + gg[c] * D + dd[c] + 4 * e, rw));
                    }
#pragma unroll
                    for (int c = 0; c < CG; ++c) {
                        const float Mn = fmaxf(M[c], mw[c]);
                        if (Mn == -INFINITY) continue;     // nothing seen yet
                        const float a = M[c] == -INFINITY ? 0.f : ex2(M[c] - Mn);
                        const float b = mw[c] == -INFINITY ? 0.f : ex2(mw[c] - Mn);
                        Ls[c] = fmaf(b, lw[c], Ls[c] * a);
#pragma unroll
                        for (int e = 0; e < E / 4; ++e) {
                            O[c][4 * e] = fmaf(b, ow[c][e].x, O[c][4 * e] * a);
                            O[c][4 * e + 1] = fmaf(b, ow[c][e].y, O[c][4 * e + 1] * a);
                            O[c][4 * e + 2] = fmaf(b, ow[c][e].z, O[c][4 * e + 2] * a);
                            O[c][4 * e + 3] = fmaf(b, ow[c][e].w, O[c][4 * e + 3] * a);
                        }
                        M[c] = Mn;
                    }
                }
#pragma unroll
                for (int c = 0; c < CG; ++c) {
                    if (c0g + c >= CPL || lane + 32 * (c0g + c) >= NCH) continue;
                    if (MQ && out_row(u, gg[c]) < 0) continue;
                    emit(u, gg[c], dd[c], M[c], Ls[c], O[c]);
                }
            }
        }
        __syncwarp();
    };

    // Count this warp in at the first warp of unit `ui`; returns the old count.
    auto arrive_at = [&](int ui) -> int {          // lane 0 only
        const int g_first = owner(cum[ui]);
        return atom_add_acq_rel_dsmem(map_to_rank(&arrive[g_first % NW], g_first / NW), 1);
    };
    // Warps (with non-empty ranges) that hold a partial of unit `ui`.
    auto parts_of = [&](int ui) -> int {
        const int g_first = owner(cum[ui]), g_last = owner(cum[ui] + units[ui].nb - 1);
        int n = 0;
        for (int g = g_first; g <= g_last; ++g) n += range_lo(g) < range_lo(g + 1);
        return n;
    };

    // The unit this warp's range starts inside of, once this warp has parked
    // its partial of it: the arrival (a cluster-scope fence and an atomic) is
    // deferred to the end of the range, when no copies are in flight, so the
    // fence does not hold up the stream.
    int pending = -1;

    // Leave unit `ui`.  A unit only this warp touched is written from
    // registers; otherwise this warp parks its partial, and at the end of the
    // range (at_end) it arrives for the pending unit and this one; the last
    // warp of a unit to arrive merges it.
    auto leave_unit = [&](int ui, bool at_end) {
        wa.finish();
        const UnitRec u = units[ui];
        const int u_lo = cum[ui], u_hi = cum[ui] + u.nb;
        const bool from_before = u_lo < my_lo, to_after = u_hi > my_hi;
        int shared_unit = -1;
        if (!from_before && !to_after) {
            // a unit only this warp touched: write its result from registers
            const float vsc = v_scale_of(u);
            wa.for_each_result([&](int g, int d, float v0, float v1, bool first, float m,
                                   float l) {
                v0 *= vsc;
                v1 *= vsc;
                if constexpr (PARTIAL) {
                    const long long row =
                        ((long long)u.s * H + u.j * G + g) * p.max_parts + u.part;
                    *reinterpret_cast<float2 *>(p.part_o + row * D + d) = make_float2(v0, v1);
                    if (first) {
                        p.part_m[row] = m * LN2;      // natural units
                        p.part_l[row] = l;
                    }
                } else {
                    T *o = reinterpret_cast<T *>(p.out) + out_row(u, g) * D + d;
                    store_pair<T>(o, v0, v1);
                }
            });
        } else {
            float *mine = part_of(gw, (from_before && !to_after) ? 0 : 1);
            // partial layout: O[ROWS][D], M[ROWS], L[ROWS]
            wa.store_partial(mine + ROWS * D, mine + ROWS * D + ROWS, mine);
            shared_unit = ui;
        }
        __syncwarp();
        wa.reset();
        if (!at_end) {
            // only the range's first unit can be shared and end inside it
            if (shared_unit >= 0) pending = shared_unit;
            return;
        }
        if (pending < 0 && shared_unit < 0) return;
        int old_p = 0, old_u = 0;
        if (lane == 0) {
            fence_acq_rel_cluster();               // the parked partials are visible first
            if (pending >= 0) old_p = arrive_at(pending);
            if (shared_unit >= 0) old_u = arrive_at(shared_unit);
        }
        old_p = __shfl_sync(0xffffffffu, old_p, 0);
        old_u = __shfl_sync(0xffffffffu, old_u, 0);
        const bool last_p = pending >= 0 && old_p == parts_of(pending) - 1;
        const bool last_u = shared_unit >= 0 && old_u == parts_of(shared_unit) - 1;
        if (last_p || last_u) fence_acq_rel_cluster();
        if (last_p) merge_unit(pending);
        if (last_u) merge_unit(shared_unit);
        pending = -1;
    };

    int cur = -1, qnext = -1;                      // unit whose query is loaded ahead
    float unit_scale = p.scale_log2;               // score scale (x K's scale for E4M3)
    int k_done = 0;
    bool ok = true;
    for (int k = 0; k < n_mine; ++k) {
        if (k - c0 == 32) {
            c0 += 32;
            ui_cur = ui_nxt;
            pb_cur = pb_nxt;
            fetch(c0 + 32 + lane, ui_nxt, pb_nxt);
        }
        int ui, pbk;
        of(k, ui, pbk);
        if (ui != cur) {
            if (cur >= 0) leave_unit(cur, false);
            cur = ui;
            if constexpr (MQ) {
                // this lane's rows g and g + 8 of the unit's 16-row tile:
                // (token i, head) pairs, token i seeing positions up to L - nq + i
                const UnitRec &u = units[ui];
                const int r_lo = 16 * u.part + (lane >> 2), r_hi = r_lo + 8;
                auto qrow = [&](int r) -> const T * {
                    if (r >= u.nq * G) return nullptr;
                    return reinterpret_cast<const T *>(p.q) +
                           (long long)(u.q0 + r / G) * p.q_seq_stride +
                           (long long)(u.j * G + r % G) * D;
                };
                wa.load_q(qrow(r_lo), qrow(r_hi), u.L - u.nq + r_lo / G, u.L - u.nq + r_hi / G);
            } else {
                auto qptr = [&](int q) {
                    const UnitRec &u = units[q];
                    return reinterpret_cast<const T *>(p.q) + (long long)u.s * p.q_seq_stride +
                           (long long)u.j * G * D;
                };
                if (qnext != ui) wa.prefetch_q(qptr(ui));
                if constexpr (TC) wa.take_q();
                else wa.take_q(p.scale_log2);
                if constexpr (F8) unit_scale = p.scale_log2 * __ldg(p.k_scale + units[ui].j);
                // load the next unit's query while this one streams
                qnext = -1;
                if (ui + 1 < nu && cum[ui + 1] < my_hi && units[ui + 1].nb > 0) {
                    qnext = ui + 1;
                    wa.prefetch_q(qptr(qnext));
                }
            }
        }
        const int st = k % S;
        const bool waited = mbar_wait_bounded(&my_bars[st], (uint32_t)((k / S) & 1), p.err);
        if (!__all_sync(0xffffffffu, waited)) { ok = false; break; }
        k_done = k + 1;
        if (pbk >= 0 && (long long)pbk < p.num_blocks) {
            unsigned char *Kt = my_stages + (size_t)st * 2 * TILE;
            const int rows = rows_of(k, ui);
            if constexpr (TC) {
                // tail rows hold other tokens' data: the one-token block math
                // drops them in registers; the others clear them in the tile
                if (F8 || MQ) {
                    if (rows < 16) {
                        if constexpr (F8) W::zero_rows(Kt + TILE, rows, lane);
                        else WarpAttnTC<T, D, G>::zero_rows(Kt + TILE, rows, lane);
                        // these generic writes must be ordered before the next
                        // bulk copy into the stage
                        fence_proxy_async_smem();
                        __syncwarp();
                    }
                }
                if constexpr (MQ) wa.block(smem_u32(Kt), smem_u32(Kt + TILE), pos_of(k, ui), p.scale_log2);
                else wa.block(smem_u32(Kt), smem_u32(Kt + TILE), rows, unit_scale);
            } else {
                wa.block(Kt, Kt + TILE, rows, Sc, Pb, Al);
            }
        }
        __syncwarp();                              // every lane is done with the stage
        const int kn = k + S;
        if (kn < n_mine) {
            int uin, pbn;
            of(kn, uin, pbn);
            if (lane == 0) issue(kn, uin, pbn);
        }
    }
    // a timeout leaves the unit unmerged (its output is not written; the
    // error word says so); otherwise finish the last unit
    // every block of the cluster has initialised its counters (the only
    // accesses to peers' shared memory follow)
    if (C > 1) cluster_wait();
    if (ok && cur >= 0) leave_unit(cur, true);

    // after a timeout: wait (bounded) for this warp's copies still in flight
    if (!ok) {
        const int issued = min(n_mine, k_done + S);
        for (int k = k_done; k < issued; ++k)
            mbar_wait_bounded(&my_bars[k % S], (uint32_t)((k / S) & 1), p.err);
    }
    // keep this block's shared memory alive while peers may still read it
    __syncthreads();
    if (C > 1) cluster_sync();
}

// Stages per warp: as many as keep the blocks per SM the kernel is built for
// (two, or three for E4M3 tiles) within shared memory, up to about
// PA_STAGE_KB KiB of K+V in flight per warp.
#ifndef PA_STAGE_KB
#define PA_STAGE_KB 16
#endif
template <typename T, typename KV, int D, int G, int MODE, int NW>
__host__ __device__ constexpr int persistent_stages() {
    int s = PA_STAGE_KB * 1024 / (int)(2 * 16 * D * sizeof(KV));
    s = s < 2 ? 2 : (s > 6 ? 6 : s);
    const size_t cap = (size_t)(227 / persistent_blocks_per_sm<KV, NW>()) * 1024;
    while (s > 2 && PersistentLayout<T, KV, D, G, NW, 0, MODE>::BYTES +
                            (size_t)NW * s * (2 * 16 * D * sizeof(KV) + 8) > cap)
        --s;
    return s;
}

template <typename T, typename KV, int D, int G, int MODE>
struct PersistentConfig {
    static constexpr int NW = persistent_warps<KV, MODE>();
    static constexpr int S = persistent_stages<T, KV, D, G, MODE, NW>();
    using Lay = PersistentLayout<T, KV, D, G, NW, S, MODE>;
};

// Largest num_seqs the persistent kernel sorts in shared memory.
template <typename T, typename KV, int D, int G, int MODE>
constexpr int persistent_max_seqs() {
    return PersistentConfig<T, KV, D, G, MODE>::Lay::MAX_SEQS;
}

// Clusters of `cluster` blocks, as many as fit on the GPU at once (looked up
// once per device and cluster size), but at least enough that no cluster
// gets more than NU_MAX units.
template <typename T, typename KV, int D, int G, int MODE>
cudaError_t launch_persistent(const DecodeParams &p, long long unit_bound, int cluster,
                              cudaStream_t st) {
    using C = PersistentConfig<T, KV, D, G, MODE>;
    constexpr size_t smem = C::Lay::BYTES;
    static_assert(smem <= 227 * 1024, "shared memory");
    auto kern = decode_persistent_kernel<T, KV, D, G, C::NW, C::S, MODE>;
    if (p.num_seqs > C::Lay::MAX_SEQS) {
        // more sequences than one block sorts in shared memory: launch on
        // consecutive slices of the batch (sequences are independent)
        const int chunk = C::Lay::MAX_SEQS, B = p.num_seqs;
        for (int a = 0; a < B; a += chunk) {
            const int n = B - a < chunk ? B - a : chunk;
            DecodeParams q = p;
            q.num_seqs = n;
            q.seq_lens = p.seq_lens + a;
            q.block_tables = p.block_tables + (long long)a * p.max_blocks;
            if (MODE == MODE_MULTI) {
                q.query_start = p.query_start + a;        // rows stay absolute
            } else {
                q.q = reinterpret_cast<const T *>(p.q) + (long long)a * p.q_seq_stride;
                q.out = reinterpret_cast<T *>(p.out) + (long long)a * p.num_heads * D;
            }
            if (MODE == MODE_PARTITIONED) {
                const long long rows = (long long)a * p.num_heads * p.max_parts;
                q.part_o = p.part_o + rows * D;
                q.part_m = p.part_m + rows;
                q.part_l = p.part_l + rows;
            }
            const long long ub = (unit_bound * n + B - 1) / B;
            cudaError_t e = launch_persistent<T, KV, D, G, MODE>(q, ub > 0 ? ub : 1, cluster, st);
            if (e != cudaSuccess) return e;
        }
        return cudaSuccess;
    }
    if (cluster < 1 || cluster > 16 || (cluster & (cluster - 1))) return cudaErrorInvalidValue;
    // clusters resident per device, per size; written once per (device, size)
    // after the attributes are set, read by any host thread
    static std::atomic<int> fitted[64][5];
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    const int ci = cluster == 1 ? 0 : cluster == 2 ? 1 : cluster == 4 ? 2 : cluster == 8 ? 3 : 4;
    int nc = (dev >= 0 && dev < 64) ? fitted[dev][ci].load(std::memory_order_acquire) : 0;

    cudaLaunchConfig_t cfg = {};
    cfg.blockDim = dim3(C::NW * 32, 1, 1);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = st;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    // may start while the previous kernel in the stream finishes, if that
    // kernel allows it (the cache write does); see grid_dependency_wait()
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = PA_DECODE_PDL;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (nc <= 0) {
        e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
        if (e != cudaSuccess) return e;
        if (cluster > 8) {                         // 16 blocks: beyond the portable size
            e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            if (e != cudaSuccess) return e;
        }
        cfg.gridDim = dim3((unsigned)(cluster * 64), 1, 1);
        e = cudaOccupancyMaxActiveClusters(&nc, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (nc < 1) nc = 1;
        if (dev >= 0 && dev < 64) fitted[dev][ci].store(nc, std::memory_order_release);
    }
    long long NC = nc;
    const long long need = (unit_bound + C::Lay::NU_MAX - 1) / C::Lay::NU_MAX;
    if (need > NC) NC = need;
    if (NC > unit_bound) NC = unit_bound > 0 ? unit_bound : 1;
    if (NC * cluster > 0x7fffffffLL) return cudaErrorNotSupported;
    cfg.gridDim = dim3((unsigned)(NC * cluster), 1, 1);
    e = cudaLaunchKernelEx(&cfg, kern, p);
    if (e != cudaSuccess) return e;
    return cudaGetLastError();
}

// Launch mode MODE for the built shapes: D in {64, 128}, G in {1, 2, 4, 8}.
template <typename T, int MODE, typename KV = T>
cudaError_t dispatch_persistent(const DecodeParams &p, int D, int G, long long unit_bound,
                                int cluster, cudaStream_t st) {
#define PA_CASE(DD, GG) \
    if (D == DD && G == GG) return launch_persistent<T, KV, DD, GG, MODE>(p, unit_bound, cluster, st);
    PA_CASE(64, 1) PA_CASE(64, 2) PA_CASE(64, 4) PA_CASE(64, 8)
    PA_CASE(128, 1) PA_CASE(128, 2) PA_CASE(128, 4) PA_CASE(128, 8)
#undef PA_CASE
    return cudaErrorNotSupported;
}

}  // namespace pa
