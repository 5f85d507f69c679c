/*
 * pa_ref.c -- fp64 CPU oracle for paged decode attention.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline leg load this library; the product path never
 * does.  It shares no code, header, table or helper with the CUDA library.
 *
 * What it computes, and where the pages define it:
 *
 *  - Cache write ("vLLM: Architecture, PagedAttention & Internals", *The
 *    forward step in detail*): every new token t with slot s_t >= 0 has its
 *    key and value rows copied, byte for byte, into row (s_t mod block_size)
 *    of physical block floor(s_t / block_size).  Nothing else changes.
 *
 *  - Decode attention (same page, *PagedAttention in one paragraph*: "the
 *    arithmetic of attention is unchanged -- only the addressing is
 *    indirected"; "vLLM: High-Throughput Serving with PagedAttention" (lesson 13.15), *PagedAttention, the core idea*,
 *    step 4): for sequence s and query head h, gather K and V of tokens
 *    0..L_s-1 through the block table into contiguous fp64 arrays, then run
 *    textbook softmax attention:
 *        z_t  = scale * sum_d q[d] * K[t][d]
 *        w_t  = exp(z_t - max_t z_t) / sum_u exp(z_u - max_t z_t)
 *        out  = sum_t w_t * V[t]
 *    Query head h reads KV head h / G with G = H_q / H_kv (grouped-query
 *    attention with consecutive query heads sharing a KV head, the layer's
 *    `Attention(num_heads, head_size, scale, num_kv_heads)` contract in
 *    "vLLM: Architecture, PagedAttention & Internals", *Custom model
 *    registration*).  L_s == 0 gives out = 0.
 *
 *  - Multi-token queries (the prefill chunk or the k+1 positions a
 *    speculative step verifies, "vLLM: Architecture, PagedAttention &
 *    Internals", *Chunked prefill* and *Speculative decoding*, over the same
 *    paged cache): sequence s has n_s new query tokens, already written to
 *    the cache, at positions L_s - n_s .. L_s - 1; query token i attends to
 *    positions 0 .. L_s - n_s + i (causal among the new tokens) with the same
 *    textbook softmax.
 *
 *  - Split-KV partition statistics and their log-sum-exp merge: the token
 *    range is cut into fixed partitions; partition p reports
 *        m_p = max z_t,  l_p = sum exp(z_t - m_p),
 *        o_p = sum exp(z_t - m_p) V[t] / l_p          (t in partition p)
 *    and the merge is  M = max m_p,  c_p = l_p exp(m_p - M),
 *        out = sum_p c_p o_p / sum_p c_p,
 *    which equals the unpartitioned softmax exactly in real arithmetic.
 *
 *  - Block copies for copy-on-write ("vLLM: Architecture, PagedAttention &
 *    Internals", *Copy-on-write for shared blocks*; "vLLM: High-Throughput
 *    Serving with PagedAttention", *PagedAttention, the core idea*): when a
 *    writer must not clobber a shared block, a fresh block receives a copy
 *    of the shared block's contents.  For every (src, dst) pair of the
 *    mapping and every cache (K and V of every layer), the bytes of block
 *    src are copied to block dst; pairs with an id outside the pool are
 *    skipped and counted.
 *
 *  - FP8 KV cache (named, without a format, as the way to enlarge the pool in
 *    "vLLM: Architecture, PagedAttention & Internals", *The knobs that
 *    actually matter*, item 5, and "vLLM: High-Throughput Serving with
 *    PagedAttention", *The benefits of vLLM*).  Reading taken here: the OCP
 *    FP8 E4M3 format with one float scale per KV head for K and one for V.
 *    The cache write stores code = E4M3(x / scale_j), the quotient rounded
 *    once to binary32 and then to E4M3 (round to nearest, ties to even;
 *    finite values beyond the largest code, and infinities, saturate to
 *    +-448; NaN becomes the NaN code 0x7F).  Attention reads
 *    value(code) * scale_j and is otherwise unchanged.
 *
 * Storage formats read here: f32, bf16 (the upper 16 bits of an IEEE binary32)
 * and f16 (IEEE binary16), each widened exactly to double, and E4M3 codes in
 * FP8 caches.
 */
#include <math.h>
#include <pthread.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

enum { REF_F32 = 0, REF_BF16 = 1, REF_F16 = 2, REF_E4M3 = 3 };

/* ---- element access ---------------------------------------------------- */

static double f16_bits_to_double(uint16_t h) {
    /* IEEE 754 binary16: 1 sign bit, 5 exponent bits (bias 15), 10 fraction bits */
    int sign = (h >> 15) & 1;
    int e = (h >> 10) & 0x1f;
    int f = h & 0x3ff;
    double v;
    if (e == 0) {
        v = ldexp((double)f, -24);              /* subnormal: f * 2^-14 * 2^-10 */
    } else if (e == 31) {
        v = f ? NAN : INFINITY;
    } else {
        v = ldexp((double)(f + 1024), e - 25);  /* (1 + f/1024) * 2^(e-15) */
    }
    return sign ? -v : v;
}

/* OCP FP8 E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 fraction bits; no
 * infinities; exponent 15 with fraction 7 is NaN, so the largest finite
 * magnitude is 1.75 * 2^8 = 448; exponent 0 holds the subnormals f * 2^-9. */
double pa_ref_e4m3_to_double(int32_t code) {
    int sign = (code >> 7) & 1;
    int e = (code >> 3) & 0xf;
    int f = code & 7;
    double v;
    if (e == 15 && f == 7) return NAN;
    if (e == 0) v = ldexp((double)f, -9);
    else v = ldexp((double)(8 + f), e - 10);    /* (1 + f/8) * 2^(e-7) */
    return sign ? -v : v;
}

/* Round a binary32 value to E4M3: to nearest, ties to even; magnitudes above
 * 448 (after rounding) and infinities saturate to 448; NaN gives 0x7F. */
int32_t pa_ref_e4m3_from_float(float x) {
    if (isnan(x)) return 0x7f;
    const int sign = signbit(x) ? 0x80 : 0;
    const double a = fabs((double)x);
    if (a > 448.0) return sign | 0x7e;
    /* the spacing of E4M3 values around a: 2^(E-3) for a in [2^E, 2^(E+1)),
     * E >= -6; the subnormal range [0, 2^-6) has spacing 2^-9 */
    int E = -6;
    if (a >= ldexp(1.0, -6)) {
        int e2;
        frexp(a, &e2);                 /* a = f * 2^e2, f in [0.5, 1) */
        E = e2 - 1;
    }
    const double step = ldexp(1.0, E - 3);
    const double n = a / step;         /* exact: a power-of-two divisor */
    double r = floor(n);
    const double rem = n - r;
    if (rem > 0.5 || (rem == 0.5 && fmod(r, 2.0) != 0.0)) r += 1.0;
    const double v = r * step;         /* the rounded magnitude */
    if (v > 448.0) return sign | 0x7e;
    if (v < ldexp(1.0, -6)) return sign | (int)(v / ldexp(1.0, -9));
    int ev;
    frexp(v, &ev);
    const int Ev = ev - 1;             /* v in [2^Ev, 2^(Ev+1)) */
    const int f = (int)(v / ldexp(1.0, Ev - 3)) - 8;
    return sign | ((Ev + 7) << 3) | f;
}

static double load_elem(const void *base, int64_t idx, int dtype) {
    if (dtype == REF_E4M3) {
        return pa_ref_e4m3_to_double(((const uint8_t *)base)[idx]);
    } else if (dtype == REF_F32) {
        return (double)((const float *)base)[idx];
    } else if (dtype == REF_BF16) {
        uint32_t bits = (uint32_t)((const uint16_t *)base)[idx] << 16;
        float f;
        memcpy(&f, &bits, sizeof f);
        return (double)f;
    } else {
        return f16_bits_to_double(((const uint16_t *)base)[idx]);
    }
}

static int elem_bytes(int dtype) { return dtype == REF_F32 ? 4 : (dtype == REF_E4M3 ? 1 : 2); }

/* ---- sizes ("vLLM: High-Throughput Serving with PagedAttention" (lesson 13.15), *The problem: the KV cache eats GPU
 * memory*; "vLLM: Architecture, PagedAttention & Internals", *How many blocks
 * exist?*) --------------------------------------------------------------- */

/* KV bytes one token occupies across all layers: 2 (K and V) * L * H_kv * d * b */
int64_t pa_ref_kv_bytes_per_token(int64_t num_layers, int64_t num_kv_heads,
                                  int64_t head_dim, int64_t dtype_bytes) {
    return 2 * num_layers * num_kv_heads * head_dim * dtype_bytes;
}

/* bytes of one block = block_size tokens */
int64_t pa_ref_bytes_per_block(int64_t block_size, int64_t num_layers,
                               int64_t num_kv_heads, int64_t head_dim,
                               int64_t dtype_bytes) {
    return block_size * pa_ref_kv_bytes_per_token(num_layers, num_kv_heads,
                                                  head_dim, dtype_bytes);
}

/* blocks a sequence of n tokens holds: ceil(n / block_size) */
int64_t pa_ref_blocks_for_tokens(int64_t n_tokens, int64_t block_size) {
    return (n_tokens + block_size - 1) / block_size;
}

/* ---- cache write --------------------------------------------------------- */

/* k, v: [T, H_kv, D] rows with token stride (elements) k_tok_stride /
 * v_tok_stride, heads contiguous; caches: [num_blocks, H_kv, block_size, D].
 * Returns the number of tokens skipped because their slot was out of range
 * (negative slots are padding and are skipped silently). */
int64_t pa_ref_reshape_and_cache(const void *k, const void *v, void *k_cache,
                                 void *v_cache, const int64_t *slot_mapping,
                                 int64_t num_tokens, int32_t num_kv_heads,
                                 int32_t head_dim, int64_t k_tok_stride,
                                 int64_t v_tok_stride, int32_t block_size,
                                 int64_t num_blocks, int32_t dtype) {
    const int eb = elem_bytes(dtype);
    const size_t row_bytes = (size_t)head_dim * eb;
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) { ++bad; continue; }
        int64_t blk = slot / block_size;
        int64_t row = slot % block_size;
        for (int32_t j = 0; j < num_kv_heads; ++j) {
            int64_t dst = ((blk * num_kv_heads + j) * block_size + row) * head_dim;
            memcpy((char *)k_cache + dst * eb,
                   (const char *)k + (t * k_tok_stride + (int64_t)j * head_dim) * eb,
                   row_bytes);
            memcpy((char *)v_cache + dst * eb,
                   (const char *)v + (t * v_tok_stride + (int64_t)j * head_dim) * eb,
                   row_bytes);
        }
    }
    return bad;
}

/* FP8 cache write: k, v as above in `src_dtype` (f32, bf16 or f16); caches
 * hold E4M3 codes; element d of KV head j becomes E4M3(x / scale_j) with the
 * quotient taken in binary32.  Returns the number of out-of-range slots. */
int64_t pa_ref_reshape_and_cache_fp8(const void *k, const void *v, uint8_t *k_cache,
                                     uint8_t *v_cache, const int64_t *slot_mapping,
                                     int64_t num_tokens, int32_t num_kv_heads,
                                     int32_t head_dim, int64_t k_tok_stride,
                                     int64_t v_tok_stride, int32_t block_size,
                                     int64_t num_blocks, int32_t src_dtype,
                                     const float *k_scale, const float *v_scale) {
    int64_t bad = 0;
    for (int64_t t = 0; t < num_tokens; ++t) {
        int64_t slot = slot_mapping[t];
        if (slot < 0) continue;
        if (slot >= num_blocks * (int64_t)block_size) { ++bad; continue; }
        int64_t blk = slot / block_size;
        int64_t row = slot % block_size;
        for (int32_t j = 0; j < num_kv_heads; ++j) {
            int64_t dst = ((blk * num_kv_heads + j) * block_size + row) * head_dim;
            for (int32_t d = 0; d < head_dim; ++d) {
                float xk = (float)load_elem(k, t * k_tok_stride + (int64_t)j * head_dim + d, src_dtype);
                float xv = (float)load_elem(v, t * v_tok_stride + (int64_t)j * head_dim + d, src_dtype);
                k_cache[dst + d] = (uint8_t)pa_ref_e4m3_from_float(xk / k_scale[j]);
                v_cache[dst + d] = (uint8_t)pa_ref_e4m3_from_float(xv / v_scale[j]);
            }
        }
    }
    return bad;
}

/* ---- block copies (copy-on-write) ---------------------------------------- */

/* caches[c] holds num_blocks blocks of block_bytes bytes; mapping is
 * [num_pairs][2] (src, dst).  Pairs are applied in order.  Returns the number
 * of pairs skipped because src or dst is outside [0, num_blocks). */
int64_t pa_ref_copy_blocks(void *const *caches, int32_t num_caches, const int64_t *mapping,
                           int64_t num_pairs, int64_t num_blocks, int64_t block_bytes) {
    int64_t bad = 0;
    for (int64_t i = 0; i < num_pairs; ++i) {
        const int64_t src = mapping[2 * i], dst = mapping[2 * i + 1];
        if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) { ++bad; continue; }
        for (int32_t c = 0; c < num_caches; ++c) {
            char *base = (char *)caches[c];
            memmove(base + dst * block_bytes, base + src * block_bytes, (size_t)block_bytes);
        }
    }
    return bad;
}

/* ---- decode attention ---------------------------------------------------- */

typedef struct {
    const void *q;            /* [B, H_q, D] with q_seq_stride / q_head_stride */
    const void *k_cache;      /* [N, H_kv, bs, D] */
    const void *v_cache;
    const int32_t *block_tables;  /* [B, max_blocks] */
    const int32_t *seq_lens;      /* [B] */
    int64_t num_seqs;
    int32_t num_heads, num_kv_heads, head_dim, block_size;
    int64_t num_blocks, max_blocks;
    int64_t q_seq_stride, q_head_stride;
    double scale;
    int32_t dtype;            /* q (and, unless kv_dtype says otherwise, the caches) */
    int32_t kv_dtype;         /* storage of k_cache / v_cache */
    const float *k_scale;     /* E4M3 caches: [H_kv] dequantisation scales */
    const float *v_scale;
} ref_args;

/* Gather the L tokens of (sequence s, KV head j) through the block table into
 * contiguous K[L][D], V[L][D].  Returns -1 on a block id outside the pool. */
static int gather_kv(const ref_args *a, int64_t s, int32_t j, int64_t L,
                     double *K, double *V) {
    const int64_t D = a->head_dim, bs = a->block_size;
    for (int64_t t = 0; t < L; ++t) {
        int64_t lb = t / bs;
        int64_t pb = a->block_tables[s * a->max_blocks + lb];
        if (pb < 0 || pb >= a->num_blocks) return -1;
        int64_t base = ((pb * a->num_kv_heads + j) * bs + t % bs) * D;
        const double ks = a->k_scale ? (double)a->k_scale[j] : 1.0;
        const double vs = a->v_scale ? (double)a->v_scale[j] : 1.0;
        for (int64_t d = 0; d < D; ++d) {
            K[t * D + d] = load_elem(a->k_cache, base + d, a->kv_dtype) * ks;
            V[t * D + d] = load_elem(a->v_cache, base + d, a->kv_dtype) * vs;
        }
    }
    return 0;
}

/* scores z_t = scale * q . K[t] for query head h of sequence s */
static void scores(const ref_args *a, int64_t s, int32_t h, int64_t L,
                   const double *K, double *z) {
    const int64_t D = a->head_dim;
    const int64_t qoff = s * a->q_seq_stride + (int64_t)h * a->q_head_stride;
    for (int64_t t = 0; t < L; ++t) {
        double acc = 0.0;
        for (int64_t d = 0; d < D; ++d)
            acc += load_elem(a->q, qoff + d, a->dtype) * K[t * D + d];
        z[t] = a->scale * acc;
    }
}

static int32_t check_len(const ref_args *a, int64_t s, int64_t *L) {
    *L = a->seq_lens[s];
    if (*L < 0 || *L > a->max_blocks * (int64_t)a->block_size) return -1;
    return 0;
}

/* One (sequence, query head): out[D] (fp64).  Returns 0, or -1 on bad input. */
static int decode_one(const ref_args *a, int64_t s, int32_t h, double *out,
                      double *weights /* optional [L] */) {
    const int64_t D = a->head_dim;
    const int32_t G = a->num_heads / a->num_kv_heads;
    const int32_t j = h / G;
    int64_t L;
    if (check_len(a, s, &L)) return -1;
    for (int64_t d = 0; d < D; ++d) out[d] = 0.0;
    if (L == 0) return 0;
    double *K = malloc(sizeof(double) * L * D);
    double *V = malloc(sizeof(double) * L * D);
    double *z = malloc(sizeof(double) * L);
    int rc = -1;
    if (!K || !V || !z) goto done;
    if (gather_kv(a, s, j, L, K, V)) goto done;
    scores(a, s, h, L, K, z);
    double M = -INFINITY;
    for (int64_t t = 0; t < L; ++t) M = z[t] > M ? z[t] : M;
    double S = 0.0;
    for (int64_t t = 0; t < L; ++t) { z[t] = exp(z[t] - M); S += z[t]; }
    for (int64_t t = 0; t < L; ++t) {
        double w = z[t] / S;
        if (weights) weights[t] = w;
        for (int64_t d = 0; d < D; ++d) out[d] += w * V[t * D + d];
    }
    rc = 0;
done:
    free(K); free(V); free(z);
    return rc;
}

typedef struct {
    const ref_args *a;
    double *out;
    int64_t begin, end;   /* flattened (s, h) pairs */
    int rc;
} ref_job;

static void *decode_range(void *p) {
    ref_job *job = (ref_job *)p;
    const ref_args *a = job->a;
    job->rc = 0;
    for (int64_t i = job->begin; i < job->end; ++i) {
        int64_t s = i / a->num_heads;
        int32_t h = (int32_t)(i % a->num_heads);
        if (decode_one(a, s, h, job->out + i * a->head_dim, NULL)) job->rc = -1;
    }
    return NULL;
}

static int make_args(ref_args *a, const void *q, const void *k_cache,
                     const void *v_cache, const int32_t *block_tables,
                     const int32_t *seq_lens, int64_t num_seqs,
                     int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                     int32_t block_size, int64_t num_blocks, int64_t max_blocks,
                     int64_t q_seq_stride, int64_t q_head_stride, float scale,
                     int32_t dtype) {
    if (num_kv_heads <= 0 || num_heads % num_kv_heads) return -1;
    a->q = q; a->k_cache = k_cache; a->v_cache = v_cache;
    a->block_tables = block_tables; a->seq_lens = seq_lens;
    a->num_seqs = num_seqs; a->num_heads = num_heads;
    a->num_kv_heads = num_kv_heads; a->head_dim = head_dim;
    a->block_size = block_size; a->num_blocks = num_blocks;
    a->max_blocks = max_blocks; a->q_seq_stride = q_seq_stride;
    a->q_head_stride = q_head_stride; a->scale = (double)scale;
    a->dtype = dtype;
    a->kv_dtype = dtype;
    a->k_scale = NULL;
    a->v_scale = NULL;
    return 0;
}

/* Full decode: out[B][H_q][D] (fp64).  The (s, h) pairs are split over
 * `nthreads` threads; each pair is computed independently, so the result does
 * not depend on the thread count. */
static int run_decode(const ref_args *a, double *out, int32_t nthreads) {
    int64_t n = a->num_seqs * a->num_heads;
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if (n < nthreads) nthreads = (int32_t)(n > 0 ? n : 1);
    pthread_t th[256];
    ref_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].a = a; jobs[i].out = out;
        jobs[i].begin = n * i / nthreads; jobs[i].end = n * (i + 1) / nthreads;
        jobs[i].rc = 0;
    }
    int rc = 0;
    if (nthreads == 1) {
        decode_range(&jobs[0]);
        rc = jobs[0].rc;
    } else {
        for (int i = 0; i < nthreads; ++i)
            pthread_create(&th[i], NULL, decode_range, &jobs[i]);
        for (int i = 0; i < nthreads; ++i) {
            pthread_join(th[i], NULL);
            if (jobs[i].rc) rc = -1;
        }
    }
    return rc;
}

int pa_ref_decode(double *out, const void *q, const void *k_cache,
                  const void *v_cache, const int32_t *block_tables,
                  const int32_t *seq_lens, int64_t num_seqs, int32_t num_heads,
                  int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                  int64_t num_blocks, int64_t max_blocks, int64_t q_seq_stride,
                  int64_t q_head_stride, float scale, int32_t dtype,
                  int32_t nthreads) {
    ref_args a;
    if (make_args(&a, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                  num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks, q_seq_stride, q_head_stride, scale, dtype))
        return -1;
    return run_decode(&a, out, nthreads);
}

/* Decode over E4M3 caches: `dtype` is the type of q; K and V of KV head j
 * read value(code) * k_scale[j] and value(code) * v_scale[j]. */
int pa_ref_decode_fp8(double *out, const void *q, const void *k_cache,
                      const void *v_cache, const int32_t *block_tables,
                      const int32_t *seq_lens, int64_t num_seqs, int32_t num_heads,
                      int32_t num_kv_heads, int32_t head_dim, int32_t block_size,
                      int64_t num_blocks, int64_t max_blocks, int64_t q_seq_stride,
                      int64_t q_head_stride, float scale, int32_t dtype,
                      const float *k_scale, const float *v_scale, int32_t nthreads) {
    ref_args a;
    if (make_args(&a, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                  num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks, q_seq_stride, q_head_stride, scale, dtype))
        return -1;
    if (!k_scale || !v_scale) return -1;
    a.kv_dtype = REF_E4M3;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return run_decode(&a, out, nthreads);
}

/* One (sequence, query head) over E4M3 caches (see pa_ref_decode_fp8). */
int pa_ref_decode_one_fp8(double *out, double *weights, int64_t s, int32_t h,
                          const void *q, const void *k_cache, const void *v_cache,
                          const int32_t *block_tables, const int32_t *seq_lens,
                          int64_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                          int32_t head_dim, int32_t block_size, int64_t num_blocks,
                          int64_t max_blocks, int64_t q_seq_stride,
                          int64_t q_head_stride, float scale, int32_t dtype,
                          const float *k_scale, const float *v_scale) {
    ref_args a;
    if (make_args(&a, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                  num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks, q_seq_stride, q_head_stride, scale, dtype))
        return -1;
    if (!k_scale || !v_scale) return -1;
    if (s < 0 || s >= num_seqs || h < 0 || h >= num_heads) return -1;
    a.kv_dtype = REF_E4M3;
    a.k_scale = k_scale;
    a.v_scale = v_scale;
    return decode_one(&a, s, h, out, weights);
}

/* One (sequence, query head): out[D], and the normalised softmax weights
 * w[L_s] when `weights` is not NULL. */
int pa_ref_decode_one(double *out, double *weights, int64_t s, int32_t h,
                      const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, const int32_t *seq_lens,
                      int64_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                      int32_t head_dim, int32_t block_size, int64_t num_blocks,
                      int64_t max_blocks, int64_t q_seq_stride,
                      int64_t q_head_stride, float scale, int32_t dtype) {
    ref_args a;
    if (make_args(&a, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                  num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks, q_seq_stride, q_head_stride, scale, dtype))
        return -1;
    if (s < 0 || s >= num_seqs || h < 0 || h >= num_heads) return -1;
    return decode_one(&a, s, h, out, weights);
}

/* ---- multi-token queries ------------------------------------------------- */

/* out[T][H_q][D] (fp64) for q[T][H_q][D] (token stride q_tok_stride, head
 * stride D); query_start[B+1] gives each sequence's tokens.  Query token i of
 * sequence s sees the first L_s - n_s + i + 1 tokens of the sequence.
 * Returns 0, or -1 on bad input. */
int pa_ref_decode_multi(double *out, const void *q, const void *k_cache,
                        const void *v_cache, const int32_t *block_tables,
                        const int32_t *seq_lens, const int32_t *query_start,
                        int64_t num_seqs, int32_t num_heads,
                        int32_t num_kv_heads, int32_t head_dim,
                        int32_t block_size, int64_t num_blocks,
                        int64_t max_blocks, int64_t q_tok_stride, float scale,
                        int32_t dtype) {
    ref_args a;
    if (make_args(&a, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                  num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks, q_tok_stride, head_dim, scale, dtype))
        return -1;
    const int64_t D = head_dim;
    const int32_t G = num_heads / num_kv_heads;
    int rc = 0;
    for (int64_t s = 0; s < num_seqs; ++s) {
        int64_t L;
        if (check_len(&a, s, &L)) return -1;
        const int64_t t0 = query_start[s], n = query_start[s + 1] - query_start[s];
        if (n < 0 || n > L) return -1;
        double *K = malloc(sizeof(double) * (L > 0 ? L : 1) * D);
        double *V = malloc(sizeof(double) * (L > 0 ? L : 1) * D);
        double *z = malloc(sizeof(double) * (L > 0 ? L : 1));
        if (!K || !V || !z) { free(K); free(V); free(z); return -1; }
        for (int32_t j = 0; j < num_kv_heads && rc == 0; ++j) {
            if (L > 0 && gather_kv(&a, s, j, L, K, V)) { rc = -1; break; }
            for (int32_t g = 0; g < G; ++g) {
                const int32_t h = j * G + g;
                for (int64_t i = 0; i < n; ++i) {
                    const int64_t tok = t0 + i;
                    const int64_t seen = L - n + i + 1;     /* causal prefix */
                    double *o = out + (tok * num_heads + h) * D;
                    const int64_t qoff = tok * q_tok_stride + (int64_t)h * D;
                    for (int64_t t = 0; t < seen; ++t) {
                        double acc = 0.0;
                        for (int64_t d = 0; d < D; ++d)
                            acc += load_elem(q, qoff + d, dtype) * K[t * D + d];
                        z[t] = a.scale * acc;
                    }
                    double M = -INFINITY;
                    for (int64_t t = 0; t < seen; ++t) M = z[t] > M ? z[t] : M;
                    double S = 0.0;
                    for (int64_t t = 0; t < seen; ++t) { z[t] = exp(z[t] - M); S += z[t]; }
                    for (int64_t d = 0; d < D; ++d) o[d] = 0.0;
                    for (int64_t t = 0; t < seen; ++t) {
                        const double w = z[t] / S;
                        for (int64_t d = 0; d < D; ++d) o[d] += w * V[t * D + d];
                    }
                }
            }
        }
        free(K); free(V); free(z);
        if (rc) return rc;
    }
    return 0;
}

/* ---- split-KV partitions ------------------------------------------------- */

/* Statistics of each partition of (sequence s, query head h):
 * m[p], l[p], o[p][D] for p < ceil(L_s / partition_size).  Returns the number
 * of partitions, or -1 on bad input. */
int64_t pa_ref_partition_stats(double *m, double *l, double *o, int64_t s,
                               int32_t h, int32_t partition_size,
                               const void *q, const void *k_cache,
                               const void *v_cache, const int32_t *block_tables,
                               const int32_t *seq_lens, int64_t num_seqs,
                               int32_t num_heads, int32_t num_kv_heads,
                               int32_t head_dim, int32_t block_size,
                               int64_t num_blocks, int64_t max_blocks,
                               int64_t q_seq_stride, int64_t q_head_stride,
                               float scale, int32_t dtype) {
    ref_args a;
    if (partition_size <= 0) return -1;
    if (make_args(&a, q, k_cache, v_cache, block_tables, seq_lens, num_seqs,
                  num_heads, num_kv_heads, head_dim, block_size, num_blocks,
                  max_blocks, q_seq_stride, q_head_stride, scale, dtype))
        return -1;
    int64_t L;
    if (s < 0 || s >= num_seqs || check_len(&a, s, &L)) return -1;
    const int64_t D = head_dim;
    const int32_t j = h / (num_heads / num_kv_heads);
    int64_t n_parts = (L + partition_size - 1) / partition_size;
    if (L == 0) return 0;
    double *K = malloc(sizeof(double) * L * D);
    double *V = malloc(sizeof(double) * L * D);
    double *z = malloc(sizeof(double) * L);
    int64_t rc = -1;
    if (!K || !V || !z) goto done;
    if (gather_kv(&a, s, j, L, K, V)) goto done;
    scores(&a, s, h, L, K, z);
    for (int64_t p = 0; p < n_parts; ++p) {
        int64_t t0 = p * partition_size;
        int64_t t1 = t0 + partition_size < L ? t0 + partition_size : L;
        double mp = -INFINITY;
        for (int64_t t = t0; t < t1; ++t) mp = z[t] > mp ? z[t] : mp;
        double lp = 0.0;
        for (int64_t d = 0; d < D; ++d) o[p * D + d] = 0.0;
        for (int64_t t = t0; t < t1; ++t) {
            double e = exp(z[t] - mp);
            lp += e;
            for (int64_t d = 0; d < D; ++d) o[p * D + d] += e * V[t * D + d];
        }
        for (int64_t d = 0; d < D; ++d) o[p * D + d] /= lp;
        m[p] = mp;
        l[p] = lp;
    }
    rc = n_parts;
done:
    free(K); free(V); free(z);
    return rc;
}

/* Log-sum-exp merge of n_parts partition results into out[D]. */
void pa_ref_lse_merge(double *out, const double *m, const double *l,
                      const double *o, int64_t n_parts, int32_t head_dim) {
    double M = -INFINITY;
    for (int64_t p = 0; p < n_parts; ++p) M = m[p] > M ? m[p] : M;
    double S = 0.0;
    for (int32_t d = 0; d < head_dim; ++d) out[d] = 0.0;
    if (n_parts == 0) return;
    for (int64_t p = 0; p < n_parts; ++p) {
        double c = l[p] * exp(m[p] - M);
        S += c;
        for (int32_t d = 0; d < head_dim; ++d) out[d] += c * o[p * head_dim + d];
    }
    for (int32_t d = 0; d < head_dim; ++d) out[d] /= S;
}
