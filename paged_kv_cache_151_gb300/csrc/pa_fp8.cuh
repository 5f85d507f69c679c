// pa_fp8.cuh -- FP8 (E4M3) KV cache: conversions and the per-warp decode
// arithmetic over E4M3 tiles.
//
// An FP8 KV cache halves the bytes of every block ("vLLM: Architecture,
// PagedAttention & Internals", *The knobs that actually matter*, item 5: it
// enlarges the pool).  The format read here is OCP E4M3 with one float scale
// per KV head for K and one for V: a stored code c of KV head j stands for
// value(c) * scale_j.
//
// Every E4M3 value is exactly an f16 value, so the block math converts the
// codes to f16 in registers (cvt.rn.f16x2.e4m3x2, exact) and runs the same
// two contractions as the 16-bit path on the f16 tensor cores; q is rounded
// to f16 once per unit, P is rounded to f16, accumulation is fp32.  K's scale
// folds into the score scale and V's into the final normalisation.
//
// The tiles arrive by tensor-map copies with the 128-byte (head_dim 128) or
// 64-byte (head_dim 64) swizzle.  Instead of ldmatrix, every lane reads its
// operand bytes with plain shared-memory loads, using three freedoms of the
// contractions:
//   - the order of d inside the score product is free (q and K use the same
//     one): lane t takes d = 32kk + 8t .. 8t+7 for k-steps 2kk and 2kk+1, one
//     8-byte load of a K row;
//   - the order of tokens is free (scores, P and V use the same one): column
//     n of the score tile nt holds token 8*nt + PERM[n], chosen so that every
//     half- or quarter-warp load below touches distinct banks, and the value
//     product's k index follows the score fragment, so P still never leaves
//     registers;
//   - the value product is taken transposed, O^T[d][head] += V^T[d][token]
//     P^T[token][head]: the heads (at most 8) fill the 8 columns of the MMA
//     tile instead of half of its 16 rows, so no accumulator is wasted, and
//     the probabilities of the score fragment are exactly its B operand;
//     its d order is free too (the output is unpermuted when written): lane
//     g owns d = (D/8)g .. (D/8)g + D/8-1, one contiguous run of each of its
//     four V rows.
#pragma once

#include <cuda_fp8.h>

#include <type_traits>

#include "pa_common.cuh"
#include "pa_math.cuh"
#include "pa_mma.cuh"

namespace pa {

using e4m3 = __nv_fp8_e4m3;

// Two binary32 values to E4M3 codes (round to nearest even, saturating to
// +-448; NaN stays NaN): lo in bits 0-7, hi in bits 8-15.
__device__ __forceinline__ uint32_t e4m3x2_from_f32(float lo, float hi) {
    unsigned short r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// Two E4M3 codes (bits 0-7 and 8-15 of c) to an f16x2 word (exact).
__device__ __forceinline__ uint32_t f16x2_from_e4m3x2(uint32_t c) {
    uint32_t r;
    const unsigned short h = (unsigned short)(c & 0xffffu);
    asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(r) : "h"(h));
    return r;
}

__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t sel) {
    uint32_t r;
    asm("prmt.b32 %0, %1, %2, %3;" : "=r"(r) : "r"(a), "r"(b), "r"(sel));
    return r;
}

__device__ __forceinline__ uint2 lds64(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
    return v;
}

__device__ __forceinline__ uint4 lds128(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
    return v;
}

// Token of column n (0..7) in each 8-column score tile.  Every group of four
// columns that one load instruction serves -- {0..3}, {4..7} (K rows read by
// lanes g = 0..3 and 4..7) and {0,2,4,6}, {1,3,5,7} (V rows read by lanes
// t = 0..3) -- maps to rows in four distinct bank groups under both swizzles
// (128-byte: row mod 8 >> 1; 64-byte: row bits 0 and 2).
__device__ __forceinline__ int fp8_tile_token(int n) {
    return (int)((0x26157340u >> (4 * n)) & 0xfu);   // 0 4 3 7 5 1 6 2
}

// Byte offset of byte `b` (0..ROWB-1) of row `row` in a swizzled E4M3 tile:
// 16-byte chunk c of the row lands at chunk c ^ (row & 7) (128-byte rows) or
// c ^ ((row >> 1) & 3) (64-byte rows).
template <int D>
__device__ __forceinline__ uint32_t fp8_swz(int row, int b) {
    const int c = b >> 4;
    const int x = D == 128 ? (row & 7) : ((row >> 1) & 3);
    return (uint32_t)(row * D + ((c ^ x) << 4) + (b & 15));
}

template <typename T, int D, int G>
struct WarpAttnF8 {
    static_assert(sizeof(T) == 2, "q and out are 16-bit");
    static_assert(D == 64 || D == 128, "head_dim");
    static_assert(G >= 1 && G <= 8, "group size");
    static constexpr int KK = D / 32;     // 32-wide d groups of the score product (two k-steps each)
    static constexpr int MT = D / 16;     // 16-row d tiles of the transposed value product
    static constexpr int DL = D / 8;      // d values of one lane in the value product
    static constexpr int TILE_BYTES = 16 * D;

    int lane, g, t;
    bool head_ok;                          // row g of the score tile is a real head
    uint32_t qa0[2 * KK], qa2[2 * KK];     // f16 A fragments of q (rows 0..7), d permuted
    uint4 qn[KK];                          // the next unit's q, raw (8 elements per kk)
    // O^T tiles: acc[mt][0], [1]: d = DL*g + 2mt for heads 2t, 2t+1;
    //            acc[mt][2], [3]: d = DL*g + 2mt + 1 for heads 2t, 2t+1
    float acc[MT][4];
    float m_run, l_run;                    // reference level and sum of head g (score layout)
    float m_max;                           // largest score of head g so far

    __device__ __forceinline__ void init(int lane_) {
        lane = lane_;
        g = lane >> 2;
        t = lane & 3;
        head_ok = g < G;
        reset();
    }

    __device__ __forceinline__ void reset() {
        m_run = m_max = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int j = 0; j < MT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    }

    // q points at the first of the G heads ([G][D] of T)
    __device__ __forceinline__ void prefetch_q(const T *q) {
        const uint4 *qw = reinterpret_cast<const uint4 *>(q + (head_ok ? g : 0) * D + 8 * t);
#pragma unroll
        for (int kk = 0; kk < KK; ++kk)
            qn[kk] = head_ok ? __ldg(qw + 4 * kk) : make_uint4(0, 0, 0, 0);
    }

    __device__ __forceinline__ static uint32_t to_f16x2(uint32_t w) {
        if constexpr (std::is_same<T, __half>::value) {
            return w;
        } else {
            float lo, hi;
            Elem<T>::pair(w, lo, hi);
            return Mma<__half>::pack(lo, hi);
        }
    }

    __device__ __forceinline__ void take_q() {
#pragma unroll
        for (int kk = 0; kk < KK; ++kk) {
            qa0[2 * kk] = to_f16x2(qn[kk].x);        // d 32kk+8t + {0,1}
            qa2[2 * kk] = to_f16x2(qn[kk].y);        //            {2,3}
            qa0[2 * kk + 1] = to_f16x2(qn[kk].z);    //            {4,5}
            qa2[2 * kk + 1] = to_f16x2(qn[kk].w);    //            {6,7}
        }
    }

    // The running statistics of heads 2t and 2t+1 (held by the lanes of
    // score rows 2t and 2t+1).
    __device__ __forceinline__ void head_stats(float v, float &a, float &b) const {
        a = __shfl_sync(0xffffffffu, v, (8 * t) & 31);
        b = __shfl_sync(0xffffffffu, v, (8 * t + 4) & 31);
    }

    // After finish(): f(head, d, v0, v1, first, m, l) for the normalised
    // outputs at d, d+1 of this lane's heads 2t and 2t+1.
    template <typename Fn>
    __device__ __forceinline__ void for_each_result(Fn &&f) const {
        float ma, mb, la, lb;
        head_stats(m_run, ma, mb);
        head_stats(l_run, la, lb);
        const int ha = 2 * t, hb = 2 * t + 1;
        const float ia = la > 0.f ? 1.f / la : 0.f, ib = lb > 0.f ? 1.f / lb : 0.f;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int d = DL * g + 2 * mt;
            if (ha < G) f(ha, d, acc[mt][0] * ia, acc[mt][2] * ia, g == 0 && mt == 0, ma, la);
            if (hb < G) f(hb, d, acc[mt][1] * ib, acc[mt][3] * ib, g == 0 && mt == 0, mb, lb);
        }
    }

    // One block of E4M3 tiles at shared addresses kt, vt; rows in 1..16.
    // scale_log2 already carries K's scale.
    __device__ __forceinline__ void block(uint32_t kt, uint32_t vt, int rows, float scale_log2) {
        // -- scores S[head][token]: tile 0 column n = token PERM[n], tile 1 = 8 + PERM[n];
        // the odd k-steps accumulate separately (shorter MMA chains)
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        float s2[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
        const int r0 = fp8_tile_token(g), r1 = 8 + r0;
#pragma unroll
        for (int kk = 0; kk < KK; ++kk) {
            const uint2 k0 = lds64(kt + fp8_swz<D>(r0, 32 * kk + 8 * t));
            const uint2 k1 = lds64(kt + fp8_swz<D>(r1, 32 * kk + 8 * t));
            Mma<__half>::run(s0, qa0[2 * kk], qa2[2 * kk], f16x2_from_e4m3x2(k0.x),
                             f16x2_from_e4m3x2(k0.x >> 16));
            Mma<__half>::run(s2, qa0[2 * kk + 1], qa2[2 * kk + 1], f16x2_from_e4m3x2(k0.y),
                             f16x2_from_e4m3x2(k0.y >> 16));
            Mma<__half>::run(s1, qa0[2 * kk], qa2[2 * kk], f16x2_from_e4m3x2(k1.x),
                             f16x2_from_e4m3x2(k1.x >> 16));
            Mma<__half>::run(s3, qa0[2 * kk + 1], qa2[2 * kk + 1], f16x2_from_e4m3x2(k1.y),
                             f16x2_from_e4m3x2(k1.y >> 16));
        }
        // this lane's four tokens: columns 2t, 2t+1 of both tiles
        const int ta = fp8_tile_token(2 * t), tb = fp8_tile_token(2 * t + 1);
        float sc[4] = {(s0[0] + s2[0]) * scale_log2, (s0[1] + s2[1]) * scale_log2,
                       (s1[0] + s3[0]) * scale_log2, (s1[1] + s3[1]) * scale_log2};
        const int tk[4] = {ta, tb, 8 + ta, 8 + tb};
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = tk[e] < rows ? sc[e] : -INFINITY;

        float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        m_max = fmaxf(m_max, mx);
        const float m_new = mx > m_run + RESCALE_LOG2 ? mx : m_run;   // lazy rescaling
        const float ms = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2(m_run - ms);
        // P[head g][tokens]: exactly the B fragments of the transposed value
        // product (k = the tokens of columns 2t, 2t+1 of tiles 0 and 1)
        const uint32_t pb0 = Mma<__half>::pack(ex2(sc[0] - ms), ex2(sc[1] - ms));
        const uint32_t pb1 = Mma<__half>::pack(ex2(sc[2] - ms), ex2(sc[3] - ms));
        float p0, p1, p2, p3;
        Mma<__half>::unpack(pb0, p0, p1);
        Mma<__half>::unpack(pb1, p2, p3);
        l_run = l_run * alpha + ((p0 + p1) + (p2 + p3));
        m_run = m_new;
        // the accumulator columns are heads 2t and 2t+1: rescale with theirs
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
            float aa, ab;
            head_stats(alpha, aa, ab);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                acc[mt][0] *= aa;
                acc[mt][1] *= ab;
                acc[mt][2] *= aa;
                acc[mt][3] *= ab;
            }
        }

        // -- O^T[d][head] += V^T[d][token] P^T[token][head]: A fragments from the
        // four V rows of this lane's tokens, bytes DL*g .. DL*g + DL-1, paired per d
        if constexpr (D == 128) {
            const uint4 va = lds128(vt + fp8_swz<D>(ta, 16 * g));
            const uint4 vb = lds128(vt + fp8_swz<D>(tb, 16 * g));
            const uint4 vc = lds128(vt + fp8_swz<D>(8 + ta, 16 * g));
            const uint4 vd = lds128(vt + fp8_swz<D>(8 + tb, 16 * g));
            const uint32_t wa[4] = {va.x, va.y, va.z, va.w}, wb[4] = {vb.x, vb.y, vb.z, vb.w};
            const uint32_t wc[4] = {vc.x, vc.y, vc.z, vc.w}, wd[4] = {vd.x, vd.y, vd.z, vd.w};
#pragma unroll
            for (int w = 0; w < 4; ++w) {
                // bytes 4w .. 4w+3 = d rows (g of tile 2w), (g+8 of 2w), (g of 2w+1), (g+8 of 2w+1)
                const uint32_t lo01 = prmt(wa[w], wb[w], 0x5140), lo23 = prmt(wa[w], wb[w], 0x7362);
                const uint32_t hi01 = prmt(wc[w], wd[w], 0x5140), hi23 = prmt(wc[w], wd[w], 0x7362);
                Mma<__half>::run4(acc[2 * w], f16x2_from_e4m3x2(lo01), f16x2_from_e4m3x2(lo01 >> 16),
                                  f16x2_from_e4m3x2(hi01), f16x2_from_e4m3x2(hi01 >> 16), pb0, pb1);
                Mma<__half>::run4(acc[2 * w + 1], f16x2_from_e4m3x2(lo23),
                                  f16x2_from_e4m3x2(lo23 >> 16), f16x2_from_e4m3x2(hi23),
                                  f16x2_from_e4m3x2(hi23 >> 16), pb0, pb1);
            }
        } else {
            const uint2 va = lds64(vt + fp8_swz<D>(ta, 8 * g));
            const uint2 vb = lds64(vt + fp8_swz<D>(tb, 8 * g));
            const uint2 vc = lds64(vt + fp8_swz<D>(8 + ta, 8 * g));
            const uint2 vd = lds64(vt + fp8_swz<D>(8 + tb, 8 * g));
            const uint32_t wa[2] = {va.x, va.y}, wb[2] = {vb.x, vb.y};
            const uint32_t wc[2] = {vc.x, vc.y}, wd[2] = {vd.x, vd.y};
#pragma unroll
            for (int w = 0; w < 2; ++w) {
                const uint32_t lo01 = prmt(wa[w], wb[w], 0x5140), lo23 = prmt(wa[w], wb[w], 0x7362);
                const uint32_t hi01 = prmt(wc[w], wd[w], 0x5140), hi23 = prmt(wc[w], wd[w], 0x7362);
                Mma<__half>::run4(acc[2 * w], f16x2_from_e4m3x2(lo01), f16x2_from_e4m3x2(lo01 >> 16),
                                  f16x2_from_e4m3x2(hi01), f16x2_from_e4m3x2(hi01 >> 16), pb0, pb1);
                Mma<__half>::run4(acc[2 * w + 1], f16x2_from_e4m3x2(lo23),
                                  f16x2_from_e4m3x2(lo23 >> 16), f16x2_from_e4m3x2(hi23),
                                  f16x2_from_e4m3x2(hi23 >> 16), pb0, pb1);
            }
        }
    }

    // Zero V rows [rows, 16) (whole rows: the swizzle stays inside a row).
    __device__ __forceinline__ static void zero_rows(unsigned char *vt, int rows, int lane) {
        const int n = (16 - rows) * D / 16;
        uint4 *p = reinterpret_cast<uint4 *>(vt + rows * D);
        for (int i = lane; i < n; i += 32) p[i] = make_uint4(0, 0, 0, 0);
    }

    // Bring the state to the true maximum, then sum the lanes of each row.
    __device__ __forceinline__ void finish() {
        const float f = m_max == -INFINITY ? 1.f : ex2((m_run == -INFINITY ? m_max : m_run) - m_max);
        if (__any_sync(0xffffffffu, f != 1.f)) {
            float fa, fb;
            head_stats(f, fa, fb);
#pragma unroll
            for (int mt = 0; mt < MT; ++mt) {
                acc[mt][0] *= fa;
                acc[mt][1] *= fb;
                acc[mt][2] *= fa;
                acc[mt][3] *= fb;
            }
        }
        l_run *= f;
        m_run = m_max;
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    }

    // merge slot: Mw[G], Lw[G], Aw[G][D] in natural d order
    __device__ __forceinline__ void store_partial(float *Mw, float *Lw, float *Aw) const {
        if (head_ok && t == 0) {
            Mw[g] = m_run;
            Lw[g] = l_run;
        }
        const int ha = 2 * t, hb = 2 * t + 1;
#pragma unroll
        for (int mt = 0; mt < MT; ++mt) {
            const int d = DL * g + 2 * mt;
            if (ha < G) *reinterpret_cast<float2 *>(Aw + ha * D + d) = make_float2(acc[mt][0], acc[mt][2]);
            if (hb < G) *reinterpret_cast<float2 *>(Aw + hb * D + d) = make_float2(acc[mt][1], acc[mt][3]);
        }
    }
};

}  // namespace pa
