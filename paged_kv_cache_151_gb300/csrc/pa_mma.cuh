// pa_mma.cuh -- per-warp decode arithmetic on the tensor cores for 16-bit
// caches (bf16, f16), over one 16-token block whose K and V tiles were
// placed in shared memory by tensor-map bulk copies with the 128-byte
// swizzle.
//
// With G query heads sharing a KV head, one block's scores are the product
// S^T[heads x 16 tokens] = Q[heads x d] . K^T[d x 16 tokens] and its value
// update is O[heads x d] += P[heads x 16 tokens] . V[16 tokens x d]: the
// grouped heads turn the step into two small dense contractions.  Each is a
// run of mma.sync.m16n8k16 (16-bit inputs, fp32 accumulation) with the heads
// on the M side (rows G..15 are zero), so:
//   - Q stays in registers as A fragments for the whole unit;
//   - K^T and V arrive as B fragments through ldmatrix (V transposed), which
//     reads the swizzled tiles without bank conflicts;
//   - the fp32 score fragment of the first product has exactly the layout of
//     the A fragment of the second, so P never leaves registers (it is
//     rounded to the input type, as the tensor cores require);
//   - the online-softmax statistics of head g live in the four lanes that
//     hold row g, so a block needs two shuffles for its maximum.
// Everything else follows WarpAttn in pa_math.cuh: scores carry
// scale*log2(e), the softmax uses exp2, and the running sum is accumulated
// from the same rounded P that multiplies V, so the weights applied to V are
// exactly normalised.
#pragma once

#include "pa_common.cuh"
#include "pa_math.cuh"

namespace pa {

#ifndef PA_QK_SPLIT
#define PA_QK_SPLIT 0
#endif

// Lazy rescaling of the online softmax: the reference level m of a row moves
// only when a block's maximum exceeds it by more than RESCALE_LOG2 (log2
// units), so the accumulators are rescaled on few blocks instead of nearly
// every one; probabilities exp2(s - m) then stay below 2^RESCALE_LOG2, well
// inside bf16 / f16 range.  The true maximum is tracked alongside and the
// state is brought to it once, when the unit ends, so (m, l, acc) keep their
// exact meaning: l = sum exp2(s - max s), acc = sum exp2(s - max s) v.
constexpr float RESCALE_LOG2 = 8.f;

// smem byte offset of 16-byte chunk `chunk` (0..D/8-1) of row `row` (0..15)
// in a tile stored as D/64 boxes of [16 rows][128 bytes], each box swizzled
// with the 128-byte pattern (chunk position XOR row mod 8).
__device__ __forceinline__ uint32_t swz_offset(int row, int chunk) {
    const int h = chunk >> 3, cc = chunk & 7;
    return (uint32_t)(h * 2048 + row * 128 + ((cc ^ (row & 7)) << 4));
}

__device__ __forceinline__ void ldsm_x4(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                        uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

__device__ __forceinline__ void ldsm_x4_t(uint32_t addr, uint32_t &r0, uint32_t &r1, uint32_t &r2,
                                          uint32_t &r3) {
    asm volatile("ldmatrix.sync.aligned.m8n8.x4.trans.shared.b16 {%0, %1, %2, %3}, [%4];"
                 : "=r"(r0), "=r"(r1), "=r"(r2), "=r"(r3) : "r"(addr));
}

template <typename T> struct Mma;

template <> struct Mma<__nv_bfloat16> {
    // d = a . b + d with all 16 rows of a
    __device__ __forceinline__ static void run4(float *d, uint32_t a0, uint32_t a1, uint32_t a2,
                                                uint32_t a3, uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    // d = a . b + d, a: rows 0-7 only (a1 = a3 = 0)
    __device__ __forceinline__ static void run(float *d, uint32_t a0, uint32_t a2, uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.bf16.bf16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static void unpack(uint32_t w, float &lo, float &hi) {
        lo = __uint_as_float(w << 16);
        hi = __uint_as_float(w & 0xffff0000u);
    }
};

template <> struct Mma<__half> {
    __device__ __forceinline__ static void run4(float *d, uint32_t a0, uint32_t a1, uint32_t a2,
                                                uint32_t a3, uint32_t b0, uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(a1), "r"(a2), "r"(a3), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static void run(float *d, uint32_t a0, uint32_t a2, uint32_t b0,
                                               uint32_t b1) {
        asm volatile(
            "mma.sync.aligned.m16n8k16.row.col.f32.f16.f16.f32 "
            "{%0, %1, %2, %3}, {%4, %5, %6, %7}, {%8, %9}, {%0, %1, %2, %3};"
            : "+f"(d[0]), "+f"(d[1]), "+f"(d[2]), "+f"(d[3])
            : "r"(a0), "r"(0u), "r"(a2), "r"(0u), "r"(b0), "r"(b1));
    }
    __device__ __forceinline__ static uint32_t pack(float lo, float hi) {
        __half2 h = __floats2half2_rn(lo, hi);
        return *reinterpret_cast<uint32_t *>(&h);
    }
    __device__ __forceinline__ static void unpack(uint32_t w, float &lo, float &hi) {
        __half2 h = *reinterpret_cast<__half2 *>(&w);
        const float2 f = __half22float2(h);
        lo = f.x;
        hi = f.y;
    }
};

template <typename T, int D, int G>
struct WarpAttnTC {
    static_assert(sizeof(T) == 2, "tensor-core path is for 16-bit caches");
    static_assert(G >= 1 && G <= 8, "group size");
    static constexpr int KS = D / 16;     // k-steps of the score product
    static constexpr int NT = D / 8;      // n-tiles of the value product
    static constexpr int TILE_BYTES = 16 * D * 2;

    int lane, g, t;
    bool head_ok;                          // this lane's row g is a real head
    uint32_t qa0[KS], qa2[KS];             // A fragments of Q (rows 0..7)
    uint32_t qn0[KS], qn2[KS];             // the next unit's, loaded ahead
    float acc[NT][4];                      // O fragments ([2],[3]: rows 8..15, unused)
    float m_run, l_run;                    // reference level and sum of head g
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
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    }

    // q points at the first of the G heads ([G][D] of T); rows >= G are zero
    __device__ __forceinline__ void load_q_global(const T *q) {
        prefetch_q(q);
        take_q();
    }

    // start loading the next unit's query fragments (used by take_q)
    __device__ __forceinline__ void prefetch_q(const T *q) {
        const uint32_t *qw = reinterpret_cast<const uint32_t *>(q + (head_ok ? g : 0) * D);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qn0[ks] = head_ok ? __ldg(qw + (16 * ks + 2 * t) / 2) : 0u;
            qn2[ks] = head_ok ? __ldg(qw + (16 * ks + 2 * t + 8) / 2) : 0u;
        }
    }

    __device__ __forceinline__ void take_q() {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qa0[ks] = qn0[ks];
            qa2[ks] = qn2[ks];
        }
    }

    // After finish(): this warp's own result for its G heads (a unit no other
    // warp touched).  f(g, d, v0, v1, first, m, l) gets the normalised outputs
    // of head g at d, d+1; `first` marks one call per head, which also carries
    // the head's running maximum m (log2 units) and sum l.
    template <typename Fn>
    __device__ __forceinline__ void for_each_result(Fn &&f) const {
        if (!head_ok) return;
        const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
#pragma unroll
        for (int j = 0; j < NT; ++j)
            f(g, 8 * j + 2 * t, acc[j][0] * inv, acc[j][1] * inv, t == 0 && j == 0, m_run, l_run);
    }

    // One block: kt, vt are shared-memory addresses of the swizzled tiles.
    // rows in 1..16; rows past `rows` may hold anything and are ignored (their
    // scores are masked, their values dropped from the fragments).
    __device__ __forceinline__ void block(uint32_t kt, uint32_t vt, int rows, float scale_log2) {
        // -- scores S^T[g][tok] for tok in {2t, 2t+1} (s0) and {8+2t, 9+2t} (s1)
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        const int rr = lane & 7, mi = lane >> 3;
#if PA_QK_SPLIT
        // even and odd k-steps accumulate separately: two shorter MMA chains
        float s2[4] = {0.f, 0.f, 0.f, 0.f}, s3[4] = {0.f, 0.f, 0.f, 0.f};
#endif
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            // matrices: (tok 0-7, chunk 2ks), (tok 0-7, 2ks+1), (tok 8-15, 2ks), (tok 8-15, 2ks+1)
            const int tok = (mi >> 1) * 8 + rr, chunk = 2 * ks + (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kt + swz_offset(tok, chunk), b0, b1, b2, b3);
#if PA_QK_SPLIT
            if (ks & 1) {
                Mma<T>::run(s2, qa0[ks], qa2[ks], b0, b1);
                Mma<T>::run(s3, qa0[ks], qa2[ks], b2, b3);
                continue;
            }
#endif
            Mma<T>::run(s0, qa0[ks], qa2[ks], b0, b1);
            Mma<T>::run(s1, qa0[ks], qa2[ks], b2, b3);
        }
#if PA_QK_SPLIT
        s0[0] += s2[0]; s0[1] += s2[1];
        s1[0] += s3[0]; s1[1] += s3[1];
#endif
        float sc[4] = {s0[0] * scale_log2, s0[1] * scale_log2, s1[0] * scale_log2,
                       s1[1] * scale_log2};
        const int tk[4] = {2 * t, 2 * t + 1, 8 + 2 * t, 9 + 2 * t};
#pragma unroll
        for (int e = 0; e < 4; ++e) sc[e] = tk[e] < rows ? sc[e] : -INFINITY;

        // -- online softmax for head g (the four lanes g*4 .. g*4+3)
        float mx = fmaxf(fmaxf(sc[0], sc[1]), fmaxf(sc[2], sc[3]));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 1));
        mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 2));
        m_max = fmaxf(m_max, mx);
        const float m_new = mx > m_run + RESCALE_LOG2 ? mx : m_run;
        const float ms = m_new == -INFINITY ? 0.f : m_new;
        const float alpha = ex2(m_run - ms);
        const uint32_t pa0 = Mma<T>::pack(ex2(sc[0] - ms), ex2(sc[1] - ms));
        const uint32_t pa2 = Mma<T>::pack(ex2(sc[2] - ms), ex2(sc[3] - ms));
        float p0, p1, p2, p3;
        Mma<T>::unpack(pa0, p0, p1);
        Mma<T>::unpack(pa2, p2, p3);
        l_run = l_run * alpha + ((p0 + p1) + (p2 + p3));
        m_run = m_new;
        if (__any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                acc[j][0] *= alpha;
                acc[j][1] *= alpha;
            }
        }

        // -- P.V: for each pair of 8-wide d tiles, V^T fragments via ldmatrix.trans.
        // A lane's B fragments hold tokens {2t, 2t+1} (b0, b2) and {8+2t, 9+2t}
        // (b1, b3), the tokens of its P fragment; V rows past `rows` may hold
        // anything (NaN included), so their halves are cleared here and 0 * NaN
        // never reaches the accumulators.
        const uint32_t vm0 = (tk[0] < rows ? 0x0000ffffu : 0u) | (tk[1] < rows ? 0xffff0000u : 0u);
        const uint32_t vm1 = (tk[2] < rows ? 0x0000ffffu : 0u) | (tk[3] < rows ? 0xffff0000u : 0u);
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
            // matrices: (tok 0-7, chunk j), (tok 8-15, j), (tok 0-7, j+1), (tok 8-15, j+1)
            const int tok = (mi & 1) * 8 + rr, chunk = j + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vt + swz_offset(tok, chunk), b0, b1, b2, b3);
            b0 &= vm0;
            b1 &= vm1;
            b2 &= vm0;
            b3 &= vm1;
            Mma<T>::run(acc[j], pa0, pa2, b0, b1);
            Mma<T>::run(acc[j + 1], pa0, pa2, b2, b3);
        }
    }

    // Zero V rows [rows, 16) of a tile (all chunks); call before block() on a
    // partial block whose tail rows hold data of other tokens.
    __device__ __forceinline__ static void zero_rows(unsigned char *vt, int rows, int lane) {
        const int n = (16 - rows) * (D / 8);
        for (int i = lane; i < n; i += 32) {
            const int row = rows + i / (D / 8), chunk = i % (D / 8);
            *reinterpret_cast<uint4 *>(vt + swz_offset(row, chunk)) = make_uint4(0, 0, 0, 0);
        }
    }

    // Bring the state to the true maximum and sum the per-lane partial sums of
    // each head (the four lanes of row g).
    __device__ __forceinline__ void finish() {
        const float f = m_max == -INFINITY ? 1.f : ex2((m_run == -INFINITY ? m_max : m_run) - m_max);
        if (__any_sync(0xffffffffu, f != 1.f)) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                acc[j][0] *= f;
                acc[j][1] *= f;
            }
        }
        l_run *= f;
        m_run = m_max;
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 1);
        l_run += __shfl_xor_sync(0xffffffffu, l_run, 2);
    }

    // Write this warp's (m, l, acc) into a merge slot: Mw[G], Lw[G], Aw[G][D].
    __device__ __forceinline__ void store_partial(float *Mw, float *Lw, float *Aw) const {
        if (!head_ok) return;
        if (t == 0) {
            Mw[g] = m_run;
            Lw[g] = l_run;
        }
#pragma unroll
        for (int j = 0; j < NT; ++j)
            *reinterpret_cast<float2 *>(Aw + g * D + 8 * j + 2 * t) = make_float2(acc[j][0], acc[j][1]);
    }
};

// Sixteen query rows at once: the (query token, head) pairs of a multi-token
// query (a prefill chunk or the k+1 positions of a speculative step) that
// share one KV head.  Lane (g, t) holds rows g ("lo") and g + 8 ("hi"); each
// row has its own causal limit, the last position it may see.  The layout
// of scores, probabilities and accumulators is that of WarpAttnTC with the
// upper eight rows in use.
template <typename T, int D>
struct WarpAttnTC16 {
    static_assert(sizeof(T) == 2, "tensor-core path is for 16-bit caches");
    static constexpr int KS = D / 16;
    static constexpr int NT = D / 8;

    int lane, g, t;
    int lim_lo, lim_hi;                    // last visible position per row (-1: no row)
    uint32_t qa[KS][4];                    // A fragments (lo k-lo, hi k-lo, lo k-hi, hi k-hi)
    float acc[NT][4];                      // [0],[1]: row lo; [2],[3]: row hi
    float m_lo, m_hi, l_lo, l_hi;          // reference levels and sums of the two rows
    float x_lo, x_hi;                      // their largest scores so far

    __device__ __forceinline__ void init(int lane_) {
        lane = lane_;
        g = lane >> 2;
        t = lane & 3;
        lim_lo = lim_hi = -1;
        reset();
    }

    __device__ __forceinline__ void reset() {
        m_lo = m_hi = x_lo = x_hi = -INFINITY;
        l_lo = l_hi = 0.f;
#pragma unroll
        for (int j = 0; j < NT; ++j)
#pragma unroll
            for (int e = 0; e < 4; ++e) acc[j][e] = 0.f;
    }

    // query rows (nullptr: no such row) and their causal limits
    __device__ __forceinline__ void load_q(const T *q_lo, const T *q_hi, int lo_lim, int hi_lim) {
        lim_lo = q_lo ? lo_lim : -1;
        lim_hi = q_hi ? hi_lim : -1;
        const uint32_t *wl = reinterpret_cast<const uint32_t *>(q_lo);
        const uint32_t *wh = reinterpret_cast<const uint32_t *>(q_hi);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            qa[ks][0] = q_lo ? __ldg(wl + 8 * ks + t) : 0u;
            qa[ks][1] = q_hi ? __ldg(wh + 8 * ks + t) : 0u;
            qa[ks][2] = q_lo ? __ldg(wl + 8 * ks + t + 4) : 0u;
            qa[ks][3] = q_hi ? __ldg(wh + 8 * ks + t + 4) : 0u;
        }
    }

    // One block whose row 0 is at sequence position pos0.  With vrows < 16 the
    // V rows from vrows on (past the sequence's end: other tokens' data, or
    // anything) are dropped from this lane's fragments, so they need not be
    // cleared in shared memory.
    __device__ __forceinline__ void block(uint32_t kt, uint32_t vt, int pos0, float scale_log2,
                                          int vrows = 16) {
        float s0[4] = {0.f, 0.f, 0.f, 0.f}, s1[4] = {0.f, 0.f, 0.f, 0.f};
        const int rr = lane & 7, mi = lane >> 3;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
            const int tok = (mi >> 1) * 8 + rr, chunk = 2 * ks + (mi & 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4(kt + swz_offset(tok, chunk), b0, b1, b2, b3);
            Mma<T>::run4(s0, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b0, b1);
            Mma<T>::run4(s1, qa[ks][0], qa[ks][1], qa[ks][2], qa[ks][3], b2, b3);
        }
        // s0: (lo, 2t) (lo, 2t+1) (hi, 2t) (hi, 2t+1); s1: the same at 8 + 2t
        const int p0 = pos0 + 2 * t, p1 = p0 + 1, p2 = p0 + 8, p3 = p0 + 9;
        float lo[4] = {p0 <= lim_lo ? s0[0] * scale_log2 : -INFINITY,
                       p1 <= lim_lo ? s0[1] * scale_log2 : -INFINITY,
                       p2 <= lim_lo ? s1[0] * scale_log2 : -INFINITY,
                       p3 <= lim_lo ? s1[1] * scale_log2 : -INFINITY};
        float hi[4] = {p0 <= lim_hi ? s0[2] * scale_log2 : -INFINITY,
                       p1 <= lim_hi ? s0[3] * scale_log2 : -INFINITY,
                       p2 <= lim_hi ? s1[2] * scale_log2 : -INFINITY,
                       p3 <= lim_hi ? s1[3] * scale_log2 : -INFINITY};
        float mxl = fmaxf(fmaxf(lo[0], lo[1]), fmaxf(lo[2], lo[3]));
        float mxh = fmaxf(fmaxf(hi[0], hi[1]), fmaxf(hi[2], hi[3]));
        mxl = fmaxf(mxl, __shfl_xor_sync(0xffffffffu, mxl, 1));
        mxh = fmaxf(mxh, __shfl_xor_sync(0xffffffffu, mxh, 1));
        mxl = fmaxf(mxl, __shfl_xor_sync(0xffffffffu, mxl, 2));
        mxh = fmaxf(mxh, __shfl_xor_sync(0xffffffffu, mxh, 2));
        x_lo = fmaxf(x_lo, mxl);
        x_hi = fmaxf(x_hi, mxh);
        // a row may see nothing yet (all -inf): keep its state at zero weight
        const float nl = mxl > m_lo + RESCALE_LOG2 ? mxl : m_lo;
        const float nh = mxh > m_hi + RESCALE_LOG2 ? mxh : m_hi;
        const float sl = nl == -INFINITY ? 0.f : nl, sh = nh == -INFINITY ? 0.f : nh;
        const float al = ex2(m_lo - sl), ah = ex2(m_hi - sh);
        const uint32_t pa0 = Mma<T>::pack(ex2(lo[0] - sl), ex2(lo[1] - sl));
        const uint32_t pa2 = Mma<T>::pack(ex2(lo[2] - sl), ex2(lo[3] - sl));
        const uint32_t pa1 = Mma<T>::pack(ex2(hi[0] - sh), ex2(hi[1] - sh));
        const uint32_t pa3 = Mma<T>::pack(ex2(hi[2] - sh), ex2(hi[3] - sh));
        float x0, x1, x2, x3;
        Mma<T>::unpack(pa0, x0, x1);
        Mma<T>::unpack(pa2, x2, x3);
        l_lo = l_lo * al + ((x0 + x1) + (x2 + x3));
        Mma<T>::unpack(pa1, x0, x1);
        Mma<T>::unpack(pa3, x2, x3);
        l_hi = l_hi * ah + ((x0 + x1) + (x2 + x3));
        m_lo = nl;
        m_hi = nh;
        if (__any_sync(0xffffffffu, al != 1.f || ah != 1.f)) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                acc[j][0] *= al;
                acc[j][1] *= al;
                acc[j][2] *= ah;
                acc[j][3] *= ah;
            }
        }
        // after the transposing load a lane holds tokens 2t, 2t+1 (b0, b2) and
        // 2t+8, 2t+9 (b1, b3) of its d column
        const bool tail = vrows < 16;
        const uint32_t keep0 = (2 * t < vrows ? 0xffffu : 0u) | (2 * t + 1 < vrows ? 0xffff0000u : 0u);
        const uint32_t keep1 = (2 * t + 8 < vrows ? 0xffffu : 0u) | (2 * t + 9 < vrows ? 0xffff0000u : 0u);
#pragma unroll
        for (int j = 0; j < NT; j += 2) {
            const int tok = (mi & 1) * 8 + rr, chunk = j + (mi >> 1);
            uint32_t b0, b1, b2, b3;
            ldsm_x4_t(vt + swz_offset(tok, chunk), b0, b1, b2, b3);
            if (tail) {
                b0 &= keep0; b2 &= keep0;
                b1 &= keep1; b3 &= keep1;
            }
            Mma<T>::run4(acc[j], pa0, pa1, pa2, pa3, b0, b1);
            Mma<T>::run4(acc[j + 1], pa0, pa1, pa2, pa3, b2, b3);
        }
    }

    __device__ __forceinline__ void finish() {
        const float fl = x_lo == -INFINITY ? 1.f : ex2((m_lo == -INFINITY ? x_lo : m_lo) - x_lo);
        const float fh = x_hi == -INFINITY ? 1.f : ex2((m_hi == -INFINITY ? x_hi : m_hi) - x_hi);
        if (__any_sync(0xffffffffu, fl != 1.f || fh != 1.f)) {
#pragma unroll
            for (int j = 0; j < NT; ++j) {
                acc[j][0] *= fl;
                acc[j][1] *= fl;
                acc[j][2] *= fh;
                acc[j][3] *= fh;
            }
        }
        l_lo *= fl;
        l_hi *= fh;
        m_lo = x_lo;
        m_hi = x_hi;
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 1);
        l_lo += __shfl_xor_sync(0xffffffffu, l_lo, 2);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 1);
        l_hi += __shfl_xor_sync(0xffffffffu, l_hi, 2);
    }

    // merge slot: Mw[16], Lw[16], Aw[16][D]
    __device__ __forceinline__ void store_partial(float *Mw, float *Lw, float *Aw) const {
        if (t == 0) {
            Mw[g] = m_lo; Lw[g] = l_lo;
            Mw[g + 8] = m_hi; Lw[g + 8] = l_hi;
        }
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            *reinterpret_cast<float2 *>(Aw + g * D + 8 * j + 2 * t) = make_float2(acc[j][0], acc[j][1]);
            *reinterpret_cast<float2 *>(Aw + (g + 8) * D + 8 * j + 2 * t) =
                make_float2(acc[j][2], acc[j][3]);
        }
    }

    // f(row, d, v0, v1, first, m, l) for the rows that exist
    template <typename Fn>
    __device__ __forceinline__ void for_each_result(Fn &&f) const {
        const float il = l_lo > 0.f ? 1.f / l_lo : 0.f, ih = l_hi > 0.f ? 1.f / l_hi : 0.f;
#pragma unroll
        for (int j = 0; j < NT; ++j) {
            if (lim_lo >= 0) f(g, 8 * j + 2 * t, acc[j][0] * il, acc[j][1] * il, t == 0 && j == 0, m_lo, l_lo);
            if (lim_hi >= 0) f(g + 8, 8 * j + 2 * t, acc[j][2] * ih, acc[j][3] * ih, t == 0 && j == 0, m_hi, l_hi);
        }
    }
};

}  // namespace pa
