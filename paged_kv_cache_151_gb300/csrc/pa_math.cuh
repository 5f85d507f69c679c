// pa_math.cuh -- the per-warp arithmetic of decode attention over one
// 16-token block held in shared memory: GQA-grouped scores, online softmax
// and P.V, all in fp32.
//
// Lane layout.  A K or V row of head_dim elements is NCH 16-byte chunks.
// Lane (r, c) = (lane / NCH, lane % NCH) reads chunk c of rows r, r + RPW,
// r + 2*RPW, ... so one warp-wide 16-byte load covers RPW whole rows and the
// warp never has two lanes on the same bank group.
//
//   scores   each lane multiplies its K chunk with the matching slice of the
//            G query vectors (kept in registers, pre-scaled by
//            scale*log2(e)) and the NCH partial sums of a row are combined
//            by a shuffle reduce-scatter (recursive halving): each level
//            halves the values a lane holds, so the warp ends with every
//            score exactly once.  Scores go to a small per-warp array.
//   softmax  online ("vLLM" (stanleyjacob.dev), Part IV, *Stage 6: The
//            forward pass*: the kernel streams through a sequence it never
//            holds in one piece): per head a running maximum m and sum l,
//            m' = max(m, block max), alpha = 2^(m - m'), p = 2^(s - m'),
//            l' = alpha*l + sum p.  Scores are in log2 units, so exp2 is the
//            exponential.
//   P.V      acc[g][:] = alpha[g]*acc[g][:] + sum_rows p[g][row] * V[row][:];
//            lane (r, c) owns output chunk c for the rows of its row group;
//            the row groups are summed once, when the warp is done.
#pragma once

#include "pa_common.cuh"

namespace pa {

template <typename T, int D>
struct Shape {
    static constexpr int E = Elem<T>::E;            // elements per 16-byte chunk
    static constexpr int NCH = D / E;               // chunks per row
    static constexpr int RPW = 32 / NCH;            // rows per warp-wide chunk load
    static constexpr int STEPS = 16 / RPW;          // chunk loads per 16-row tile
    static constexpr int ROW_BYTES = D * (int)sizeof(T);
    static constexpr int TILE_BYTES = 16 * ROW_BYTES;
    static constexpr int LOG_NCH = NCH == 8 ? 3 : NCH == 16 ? 4 : 5;
    static_assert(NCH == 8 || NCH == 16 || NCH == 32, "unsupported head_dim/type");
};

__host__ __device__ constexpr int ilog2(int x) { return x <= 1 ? 0 : 1 + ilog2(x / 2); }

template <int G>
__host__ __device__ constexpr int warp_scratch_floats() {   // scores[16][G], probs[16][G], alpha[G]
    return ((33 * G + 3) / 4) * 4;
}

// Shuffle reduce-scatter of N partial sums across the lanes whose chunk
// index c differs in the bits of MASK, MASK/2, ..., 1.  At each level a lane
// keeps half of its values (the upper half when its bit of c is set), adds
// the partner's copy of that half, and the count halves; once one value is
// left the remaining levels are a plain butterfly sum.
template <int N, int MASK>
struct ReduceScatter {
    static __device__ __forceinline__ void run(float *v, int c) {
        if constexpr (MASK == 0) {
            return;
        } else if constexpr (N > 1) {
            constexpr int H = N / 2;
            const bool upper = (c & MASK) != 0;
#pragma unroll
            for (int i = 0; i < H; ++i) {
                const float send = upper ? v[i] : v[i + H];
                const float keep = upper ? v[i + H] : v[i];
                v[i] = keep + __shfl_xor_sync(0xffffffffu, send, MASK);
            }
            ReduceScatter<H, MASK / 2>::run(v, c);
        } else {
            v[0] += __shfl_xor_sync(0xffffffffu, v[0], MASK);
            ReduceScatter<1, MASK / 2>::run(v, c);
        }
    }
};

// State and arithmetic of one warp attending with the G query heads of one
// KV head.
template <typename T, int D, int G>
struct WarpAttn {
    using Sh = Shape<T, D>;
    static constexpr int E = Sh::E, NCH = Sh::NCH, RPW = Sh::RPW, STEPS = Sh::STEPS;
    static constexpr int ROWB = Sh::ROW_BYTES;
    // score pass in sub-passes of SUB chunk loads: SUB*G partial sums a lane
    static constexpr int SUB = (STEPS * G <= 32) ? STEPS : (32 / G);
    static constexpr int NSUB = STEPS / SUB;
    static constexpr int NV = SUB * G;
    static constexpr int NVF = NV >= NCH ? NV / NCH : 1;    // scores a lane ends with
    static constexpr int NL = ilog2(NV / NVF);               // scatter levels
    static constexpr int LOWB = Sh::LOG_NCH - NL;            // c bits the scatter leaves
    // softmax layout: 16*G scores over 32 lanes, VPL rows of one head per lane
    static constexpr int VPL = (16 * G) / 32 >= 1 ? (16 * G) / 32 : 1;
    static constexpr int LPH = 16 / VPL;                     // lanes per head
    static_assert(STEPS % SUB == 0, "sub-pass split");

    int lane, r, c, g_sm, row0;
    float qreg[G][E];
    uint4 qraw[G];                  // the next unit's query chunks, loaded ahead
    float acc[G][E];
    float m_run, l_run;

    __device__ __forceinline__ void init(int lane_) {
        lane = lane_;
        r = lane / NCH;
        c = lane % NCH;
        const int idx0 = (lane * VPL) % (16 * G);
        g_sm = idx0 / 16;
        row0 = idx0 % 16;
        reset();
    }

    __device__ __forceinline__ void reset() {
        m_run = -INFINITY;
        l_run = 0.f;
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < E; ++e) acc[g][e] = 0.f;
    }

    // query slice of this lane from a [G][D] fp32 array (already scaled)
    __device__ __forceinline__ void load_q_smem(const float *qs) {
#pragma unroll
        for (int g = 0; g < G; ++g)
#pragma unroll
            for (int e = 0; e < E; ++e) qreg[g][e] = qs[g * D + c * E + e];
    }

    // query slice of this lane straight from global memory: q points at the
    // first of the G heads ([G][D], 16-byte aligned rows)
    __device__ __forceinline__ void load_q_global(const T *q, float scale_log2) {
        prefetch_q(q);
        take_q(scale_log2);
    }

    __device__ __forceinline__ void prefetch_q(const T *q) {
#pragma unroll
        for (int g = 0; g < G; ++g)
            qraw[g] = __ldg(reinterpret_cast<const uint4 *>(q + g * D + c * E));
    }

    __device__ __forceinline__ void take_q(float scale_log2) {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            float f[E];
            Elem<T>::to_f32(qraw[g], f);
#pragma unroll
            for (int e = 0; e < E; ++e) qreg[g][e] = f[e] * scale_log2;
        }
    }

    // After finish(): this warp's own result for its G heads (a unit no other
    // warp touched).  f(g, d, v0, v1, first, m, l) gets the normalised outputs
    // of head g at d, d+1; `first` marks one call per head, which also carries
    // the head's running maximum m (log2 units) and sum l.
    template <typename Fn>
    __device__ __forceinline__ void for_each_result(Fn &&f) const {
#pragma unroll
        for (int g = 0; g < G; ++g) {
            const float l = __shfl_sync(0xffffffffu, l_run, g * LPH);
            const float m = __shfl_sync(0xffffffffu, m_run, g * LPH);
            const float inv = l > 0.f ? 1.f / l : 0.f;
            if (r == 0) {
#pragma unroll
                for (int e = 0; e < E; e += 2)
                    f(g, c * E + e, acc[g][e] * inv, acc[g][e + 1] * inv, c == 0 && e == 0, m, l);
            }
        }
    }

    // One block: Kt, Vt are the tile's rows in shared memory; rows in 1..16.
    // Sc, Pb, Al: this warp's scratch ([16][G], [16][G], [G] floats).
    __device__ __forceinline__ void block(const unsigned char *Kt, const unsigned char *Vt,
                                          int rows, float *Sc, float *Pb, float *Al) {
        // -- scores: s[row][g] = sum_d q[g][d] * K[row][d]
#pragma unroll
        for (int sp = 0; sp < NSUB; ++sp) {
            float v[NV];
#pragma unroll
            for (int i = 0; i < SUB; ++i) {
                const int row = (sp * SUB + i) * RPW + r;
                const uint4 raw = *reinterpret_cast<const uint4 *>(Kt + row * ROWB + c * 16);
                float kf[E];
                Elem<T>::to_f32(raw, kf);
#pragma unroll
                for (int g = 0; g < G; ++g) {
                    float a = 0.f;
#pragma unroll
                    for (int e = 0; e < E; ++e) a = fmaf(qreg[g][e], kf[e], a);
                    v[i * G + g] = a;
                }
            }
            ReduceScatter<NV, NCH / 2>::run(v, c);
            if ((c & ((1 << LOWB) - 1)) == 0) {
                const int cidx = c >> LOWB;
#pragma unroll
                for (int f = 0; f < NVF; ++f) {
                    const int vi = cidx * NVF + f;
                    const int il = vi / G, g = vi % G;
                    const int row = (sp * SUB + il) * RPW + r;
                    Sc[row * G + g] = v[f];
                }
            }
        }
        __syncwarp();

        // -- online softmax
        {
            float sc[VPL];
            float mx = -INFINITY;
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                const int row = row0 + u;
                const float x = Sc[row * G + g_sm];
                sc[u] = row < rows ? x : -INFINITY;
                mx = fmaxf(mx, sc[u]);
            }
#pragma unroll
            for (int m = 1; m < LPH; m <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, m));
            const float m_new = fmaxf(m_run, mx);
            const float alpha = ex2(m_run - m_new);
            float psum = 0.f;
#pragma unroll
            for (int u = 0; u < VPL; ++u) {
                const float pv = ex2(sc[u] - m_new);
                Pb[(row0 + u) * G + g_sm] = pv;
                psum += pv;
            }
            l_run = l_run * alpha + psum;
            m_run = m_new;
            if ((lane % LPH) == 0) Al[g_sm] = alpha;
        }
        __syncwarp();

        // -- P.V
        {
            float al[G];
#pragma unroll
            for (int g = 0; g < G; ++g) al[g] = Al[g];
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < E; ++e) acc[g][e] *= al[g];
#pragma unroll
            for (int i = 0; i < STEPS; ++i) {
                const int row = i * RPW + r;
                if (row < rows) {
                    const uint4 raw = *reinterpret_cast<const uint4 *>(Vt + row * ROWB + c * 16);
                    float vf[E];
                    Elem<T>::to_f32(raw, vf);
                    float pr[G];
#pragma unroll
                    for (int g = 0; g < G; ++g) pr[g] = Pb[row * G + g];
#pragma unroll
                    for (int g = 0; g < G; ++g)
#pragma unroll
                        for (int e = 0; e < E; ++e) acc[g][e] = fmaf(pr[g], vf[e], acc[g][e]);
                }
            }
        }
    }

    // Sum the row groups' accumulators and the per-lane sums; afterwards the
    // lanes with r == 0 hold acc for chunk c, and every lane of head group
    // g_sm holds (m_run, l_run) of head g_sm.
    __device__ __forceinline__ void finish() {
#pragma unroll
        for (int m = NCH; m < 32; m <<= 1)
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < E; ++e) acc[g][e] += __shfl_xor_sync(0xffffffffu, acc[g][e], m);
#pragma unroll
        for (int m = 1; m < LPH; m <<= 1) l_run += __shfl_xor_sync(0xffffffffu, l_run, m);
    }

    // Write this warp's (m, l, acc) into a merge slot: Mw[G], Lw[G], Aw[G][D].
    __device__ __forceinline__ void store_partial(float *Mw, float *Lw, float *Aw) const {
        if ((lane % LPH) == 0) {
            Mw[g_sm] = m_run;
            Lw[g_sm] = l_run;
        }
        if (r == 0) {
#pragma unroll
            for (int g = 0; g < G; ++g)
#pragma unroll
                for (int e = 0; e < E; ++e) Aw[g * D + c * E + e] = acc[g][e];
        }
    }
};

// Store E fp32 values as one 16-byte chunk of T (round to nearest even).
template <typename T>
__device__ __forceinline__ void store_chunk(T *dst, const float *v);

template <>
__device__ __forceinline__ void store_chunk<float>(float *dst, const float *v) {
    *reinterpret_cast<float4 *>(dst) = make_float4(v[0], v[1], v[2], v[3]);
}

template <>
__device__ __forceinline__ void store_chunk<__nv_bfloat16>(__nv_bfloat16 *dst, const float *v) {
    uint4 o;
    __nv_bfloat162 h;
    h = __floats2bfloat162_rn(v[0], v[1]); o.x = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2bfloat162_rn(v[2], v[3]); o.y = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2bfloat162_rn(v[4], v[5]); o.z = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2bfloat162_rn(v[6], v[7]); o.w = *reinterpret_cast<uint32_t *>(&h);
    *reinterpret_cast<uint4 *>(dst) = o;
}

template <>
__device__ __forceinline__ void store_chunk<__half>(__half *dst, const float *v) {
    uint4 o;
    __half2 h;
    h = __floats2half2_rn(v[0], v[1]); o.x = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2half2_rn(v[2], v[3]); o.y = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2half2_rn(v[4], v[5]); o.z = *reinterpret_cast<uint32_t *>(&h);
    h = __floats2half2_rn(v[6], v[7]); o.w = *reinterpret_cast<uint32_t *>(&h);
    *reinterpret_cast<uint4 *>(dst) = o;
}

// Store two fp32 values as two consecutive elements of T.
template <typename T>
__device__ __forceinline__ void store_pair(T *dst, float a, float b);

template <>
__device__ __forceinline__ void store_pair<float>(float *dst, float a, float b) {
    *reinterpret_cast<float2 *>(dst) = make_float2(a, b);
}

template <>
__device__ __forceinline__ void store_pair<__nv_bfloat16>(__nv_bfloat16 *dst, float a, float b) {
    *reinterpret_cast<__nv_bfloat162 *>(dst) = __floats2bfloat162_rn(a, b);
}

template <>
__device__ __forceinline__ void store_pair<__half>(__half *dst, float a, float b) {
    *reinterpret_cast<__half2 *>(dst) = __floats2half2_rn(a, b);
}

}  // namespace pa
