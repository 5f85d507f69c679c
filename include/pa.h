/*
 * pa.h -- C ABI of the GB300 (sm_103a) PagedAttention decode library.
 *
 * The library implements the data-parallel hot path of a paged KV cache as
 * described in "vLLM: Architecture, PagedAttention & Internals" (LLM stack
 * book 7.3) and "vLLM: High-Throughput Serving with PagedAttention" (lesson 13.15):
 *
 *   pa_reshape_and_cache   scatter each step's new K/V rows into their slots
 *   pa_decode              one query token per sequence attends over its
 *                          paged context, walking the block table
 *   pa_decode_partitioned  the same attention split into fixed token
 *                          partitions whose results are merged by
 *                          log-sum-exp (for long contexts)
 *   pa_decode_multi        several new query tokens per sequence (a
 *                          prompt chunk or speculative positions), causal
 *                          among themselves, over the same paged cache
 *   pa_decode_cascade      decode of a batch sharing a prompt prefix: the
 *                          shared blocks read once per KV head
 *   pa_copy_blocks         block copies of copy-on-write, all layers at once
 *   *_fp8                  the cache write, decode and split-KV decode
 *                          over an FP8 (E4M3) cache with per-KV-head scales
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 * Memory.  Every pointer argument except `workspace_bytes`-style sizes is a
 * DEVICE pointer on the current CUDA device.  The caller owns all memory,
 * including the workspace of pa_decode_partitioned; the library allocates
 * nothing and frees nothing.
 *
 * Layouts (elements, row-major):
 *   k_cache, v_cache : [num_blocks, num_kv_heads, block_size, head_dim],
 *                      contiguous; a (physical block, KV head) tile is one
 *                      contiguous run of block_size * head_dim elements.
 *   q                : [num_seqs, num_heads, head_dim]; heads contiguous,
 *                      sequence stride q_seq_stride (>= num_heads*head_dim).
 *   out              : [num_seqs, num_heads, head_dim], contiguous.
 *   k, v (new rows)  : [num_tokens, num_kv_heads, head_dim]; heads
 *                      contiguous, token stride k_token_stride /
 *                      v_token_stride.
 *   block_tables     : int32 [num_seqs, max_blocks_per_seq]; entry
 *                      [s][i] is the physical block holding tokens
 *                      16*i .. 16*i+15 of sequence s.  Entries at and past
 *                      ceil(seq_lens[s] / block_size) are never read.
 *   seq_lens         : int32 [num_seqs], tokens each sequence attends over.
 *   slot_mapping     : int64 [num_tokens]; slot = block * block_size + row;
 *                      a negative slot marks a padding token (skipped).
 *
 * Query head h reads KV head h / (num_heads / num_kv_heads) (grouped-query
 * attention with consecutive query heads sharing a KV head).  A sequence
 * with seq_len 0 produces zeros.
 *
 * dtype (pa_dtype) is the storage type of q, out, k, v and both caches (all
 * the same).  Arithmetic is fp32; out is rounded to nearest-even.
 *
 * Streams.  `stream` is a cudaStream_t (NULL = the legacy default stream).
 * Every call only enqueues kernels on it and never synchronises, except
 * pa_device_error, which reads device memory synchronously.  The decode
 * kernels are launched with programmatic stream serialization: when the
 * kernel before them in the stream is a cache write of this library
 * (pa_reshape_and_cache, pa_reshape_and_cache_fp8), they start while it
 * finishes and read seq_lens, block_tables and query_start meanwhile -- the
 * cache writes never touch those -- and touch the caches, q and out only
 * after it has completed.  After any other kernel they start as usual.
 *
 * Errors.  Calls return PA_OK (0) or a negative pa_status; nothing is
 * launched when the host-side checks fail.  Contents of device arrays are not
 * inspected on the host.  Instead the kernels range-check every block id,
 * slot and sequence length they read, skip the offending access and set a bit
 * in a sticky device-side error word (PA_DEVERR_*), read and cleared with
 * pa_device_error.  No input can make a kernel read or write outside the
 * buffers described by the arguments.
 *
 * Thread safety.  Calls may be made from any host thread; the only shared
 * state is the device error word.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum {
    PA_F32 = 0,
    PA_BF16 = 1,
    PA_F16 = 2,
    PA_E4M3 = 3      /* FP8 E4M3 cache storage (the *_fp8 entry points only) */
} pa_dtype;

typedef enum {
    PA_OK = 0,
    PA_ERR_INVALID_ARG = -1,   /* NULL pointer, bad size, misaligned pointer */
    PA_ERR_UNSUPPORTED = -2,   /* head_dim, GQA group, block_size or dtype not built */
    PA_ERR_WORKSPACE = -3,     /* workspace missing or too small */
    PA_ERR_CUDA = -4           /* a CUDA runtime call or launch failed */
} pa_status;

/* bits of the device error word */
#define PA_DEVERR_BLOCK_ID   0x1u  /* a block-table entry outside [0, num_blocks) was skipped */
#define PA_DEVERR_SEQ_LEN    0x2u  /* a seq_len < 0 or > max_blocks_per_seq*block_size (or past
                                      max_seq_len in the partitioned call) was clamped, or
                                      a query row range of pa_decode_multi was invalid */
#define PA_DEVERR_SLOT       0x4u  /* a slot >= num_blocks*block_size was skipped */
#define PA_DEVERR_TIMEOUT    0x8u  /* a wait on an asynchronous copy exceeded its limit */

/*
 * pa_reshape_and_cache -- write the step's new keys and values into the cache.
 *
 * Defined in "vLLM: Architecture, PagedAttention & Internals", *The forward
 * step in detail*: the runner computes, for each token being written, the
 * physical slot (block * block_size + offset) and the attention layer first
 * scatters the fresh K and V there.  For every token t with slot_mapping[t]
 * >= 0, the rows k[t][j][:] and v[t][j][:] of every KV head j are copied bit
 * for bit to k_cache[slot/bs][j][slot%bs][:] and v_cache[...]; nothing else
 * in the caches changes.  Two tokens with the same slot race (last writer
 * wins, per element).
 *
 * Requirements: num_tokens >= 0 (0 launches nothing); block_size == 16;
 * head_dim * element size a multiple of 16 bytes; the token strides >=
 * num_kv_heads*head_dim.
 */
int pa_reshape_and_cache(const void *k, const void *v, void *k_cache,
                         void *v_cache, const int64_t *slot_mapping,
                         int64_t num_tokens, int32_t num_kv_heads,
                         int32_t head_dim, int64_t k_token_stride,
                         int64_t v_token_stride, int64_t num_blocks,
                         int32_t block_size, int32_t dtype, void *stream);

/*
 * pa_decode -- decode-step paged attention.
 *
 * Defined in "vLLM: Architecture, PagedAttention & Internals", *PagedAttention
 * in one paragraph* (the kernel gathers K and V block by block through the
 * block table; the arithmetic of attention is unchanged) and "vLLM:
 * High-Throughput Serving with PagedAttention", *PagedAttention, the core
 * idea* (step 4, attend through the table).
 * For every sequence s and query head h:
 *     out[s][h] = sum_t softmax_t(scale * q[s][h] . K_s[t]) * V_s[t],
 *     t = 0 .. seq_lens[s]-1, K_s[t] = k_cache[bt[s][t/16]][h/G][t%16].
 * The softmax is evaluated online (running maximum and sum in fp32), which is
 * exact up to rounding.
 *
 * Requirements: block_size == 16; head_dim in {64, 128}; num_heads a
 * multiple of num_kv_heads with G = num_heads/num_kv_heads in {1, 2, 4, 8};
 * num_seqs <= 65535 (batches larger than one thread block orders in shared
 * memory -- 4096 sequences at head_dim 128 -- run as consecutive slices);
 * num_kv_heads <= 65535; k_cache and v_cache 16-byte
 * aligned.  num_seqs == 0 launches nothing.
 */
int pa_decode(void *out, const void *q, const void *k_cache,
              const void *v_cache, const int32_t *block_tables,
              const int32_t *seq_lens, int32_t num_seqs, int32_t num_heads,
              int32_t num_kv_heads, int32_t head_dim, int64_t num_blocks,
              int32_t block_size, int32_t max_blocks_per_seq,
              int64_t q_seq_stride, float scale, int32_t dtype, void *stream);

/*
 * pa_decode_split -- pa_decode with an explicit work split: each (sequence,
 * KV head) is processed by a cluster of `splits` thread blocks (1, 2, 4 or 8)
 * whose partial results are merged on chip.  splits == 0 picks the split from
 * the problem shape (what pa_decode does).  The result does not depend on the
 * thread count within a block, but its rounding may differ between split
 * counts.
 */
int pa_decode_split(void *out, const void *q, const void *k_cache,
                    const void *v_cache, const int32_t *block_tables,
                    const int32_t *seq_lens, int32_t num_seqs,
                    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int64_t num_blocks, int32_t block_size,
                    int32_t max_blocks_per_seq, int64_t q_seq_stride,
                    float scale, int32_t dtype, int32_t splits, void *stream);

/*
 * pa_decode_partitioned_workspace_size -- bytes of workspace that
 * pa_decode_partitioned needs for these sizes.  Returns 0 on invalid sizes.
 *
 * Workspace layout (fp32, documented so that callers and tests can read the
 * per-partition results; P = ceil(max_seq_len / partition_size)):
 *   o_part [num_seqs][num_heads][P][head_dim]   normalised partial outputs
 *   m_part [num_seqs][num_heads][P]             max of scale*q.k in the
 *                                               partition (natural units)
 *   l_part [num_seqs][num_heads][P]             sum of exp(scale*q.k - m)
 * each array starting on a 256-byte boundary in that order.  Entries of
 * partitions past a sequence's last one are not written.
 */
size_t pa_decode_partitioned_workspace_size(int32_t num_seqs,
                                            int32_t num_heads,
                                            int32_t head_dim,
                                            int32_t max_seq_len,
                                            int32_t partition_size);

/*
 * pa_decode_partitioned -- split-KV decode for long contexts.
 *
 * Same result as pa_decode.  The tokens of each sequence are cut into
 * partitions of partition_size tokens (a multiple of 16); one thread block
 * per (sequence, KV head, partition) writes that partition's softmax
 * statistics (m_p, l_p) and normalised output o_p to the workspace, and a
 * second kernel merges them:  M = max_p m_p,  c_p = l_p exp(m_p - M),
 * out = sum_p c_p o_p / sum_p c_p.  The streaming softmax this rests on is
 * named in "vLLM" (stanleyjacob.dev), Part IV, *Stage 6: The forward pass*
 * (the kernel streams through a sequence it never holds in one piece).
 *
 * max_seq_len bounds seq_lens (it sizes the grid and the workspace); a
 * larger seq_len is clamped and flagged PA_DEVERR_SEQ_LEN.
 * Requirements as pa_decode, plus partition_size a positive multiple of 16
 * and workspace_bytes >= pa_decode_partitioned_workspace_size(...); the
 * workspace must be 256-byte aligned.
 *
 * If pa_device_error reports PA_DEVERR_TIMEOUT after a call, that call's
 * output is undefined: a partition whose bounded wait ran out is not written,
 * and the merge then reads whatever the workspace held before the call.
 */
int pa_decode_partitioned(void *out, const void *q, const void *k_cache,
                          const void *v_cache, const int32_t *block_tables,
                          const int32_t *seq_lens, int32_t num_seqs,
                          int32_t num_heads, int32_t num_kv_heads,
                          int32_t head_dim, int64_t num_blocks,
                          int32_t block_size, int32_t max_blocks_per_seq,
                          int64_t q_seq_stride, float scale, int32_t dtype,
                          int32_t partition_size, int32_t max_seq_len,
                          void *workspace, size_t workspace_bytes,
                          void *stream);

/*
 * pa_decode_multi -- paged attention for several new query tokens per
 * sequence: a chunk of a long prompt (chunked prefill) or the k+1 positions
 * a target model verifies in one pass of speculative decoding.
 *
 * Defined in "vLLM: Architecture, PagedAttention & Internals", *Prefill,
 * decode, and chunked prefill* (one forward pass mixes a slice of a prompt's
 * tokens with one-token decodes, each attending over its sequence's cache)
 * and *Speculative decoding* (the target model scores the k drafted tokens
 * and the one after them in a single pass).  The new tokens' keys and values
 * are in the cache already (pa_reshape_and_cache of the same step), and new
 * token i of a sequence sees the cache up to and including itself.
 *
 * Sequence s owns query rows r = query_start[s] .. query_start[s+1]-1
 * (n_s = query_start[s+1] - query_start[s] of them, 0 <= n_s <= seq_lens[s]);
 * row r = query_start[s] + i is the token at position seq_lens[s] - n_s + i.
 * For every such row and query head h:
 *     out[r][h] = sum_t softmax_t(scale * q[r][h] . K_s[t]) * V_s[t],
 *     t = 0 .. seq_lens[s] - n_s + i,
 * with K_s, V_s and the GQA mapping as in pa_decode.  A sequence with n_s = 0
 * (a request that runs no token this step) has no rows.
 *
 * Layouts: q is [num_q_rows][num_heads][head_dim] with row stride
 * q_row_stride (>= num_heads*head_dim, a multiple of 8 elements); out is
 * [num_q_rows][num_heads][head_dim], contiguous; query_start is int32
 * [num_seqs + 1], non-decreasing, query_start[num_seqs] <= num_q_rows.
 *
 * Requirements: as pa_decode, and dtype PA_BF16 or PA_F16 (PA_F32 gives
 * PA_ERR_UNSUPPORTED); max_query_len >= every n_s (it sizes the launch);
 * q, out 16-byte aligned.  A sequence whose row range is out of bounds,
 * decreasing, longer than max_query_len or longer than seq_lens[s] sets
 * PA_DEVERR_SEQ_LEN and its rows are not written.  num_seqs == 0 or
 * num_q_rows == 0 launches nothing.
 */
int pa_decode_multi(void *out, const void *q, const void *k_cache,
                    const void *v_cache, const int32_t *block_tables,
                    const int32_t *seq_lens, const int32_t *query_start,
                    int32_t num_seqs, int32_t num_q_rows, int32_t max_query_len,
                    int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                    int64_t num_blocks, int32_t block_size,
                    int32_t max_blocks_per_seq, int64_t q_row_stride,
                    float scale, int32_t dtype, void *stream);

/*
 * pa_copy_blocks -- the GPU half of copy-on-write.
 *
 * Defined in "vLLM: Architecture, PagedAttention & Internals", *Copy-on-write
 * for shared blocks* (a writer about to append into a block whose refcount is
 * above one gets a fresh block holding a copy of the shared one; the
 * scheduler emits the copy) and "vLLM: High-Throughput Serving with
 * PagedAttention", *PagedAttention, the core idea* (parallel sampling, beam
 * search and prefix caching share blocks until one writer diverges).
 * For every pair i and every cache c, bytes
 * [src_i * block_bytes, (src_i + 1) * block_bytes) of caches[c] are copied to
 * the same range at dst_i.  One launch covers K and V of every layer.
 *
 * caches        HOST array of num_caches (0..256) DEVICE pointers, each the
 *               base of a cache of num_blocks blocks of block_bytes bytes
 *               (any storage type: K, V, of any layer, 16-bit or E4M3), each
 *               16-byte aligned.
 * block_mapping DEVICE int64 [num_pairs][2]: (src, dst) block ids.
 * block_bytes   bytes of one block of one cache, a positive multiple of 16
 *               (num_kv_heads * block_size * head_dim * element size).
 * Pairs run in parallel: no dst may appear twice or also be a src (what
 * copy-on-write produces: fresh destinations, shared sources, possibly one
 * source copied several times).  A pair with src or dst outside
 * [0, num_blocks) is skipped and sets PA_DEVERR_BLOCK_ID.  num_pairs == 0 or
 * num_caches == 0 launches nothing.
 */
int pa_copy_blocks(void *const *caches, int32_t num_caches,
                   const int64_t *block_mapping, int64_t num_pairs,
                   int64_t num_blocks, int64_t block_bytes, void *stream);

/*
 * FP8 KV cache.
 *
 * Defined in "vLLM: Architecture, PagedAttention & Internals", *The knobs
 * that actually matter*, item 5 (an FP8 KV cache enlarges the effective pool)
 * and "vLLM: High-Throughput Serving with PagedAttention", *The benefits of
 * vLLM* (quantized KV cache); the pages fix no format.  This library stores
 * OCP FP8 E4M3 codes (1 sign, 4 exponent bits with bias 7, 3 fraction bits;
 * largest finite 448; S.1111.111 is NaN) in the same layout
 * [num_blocks, num_kv_heads, 16, head_dim] (one byte per element), with one
 * float scale per KV head for K and one for V: code c of KV head j stands for
 * value(c) * k_scale[j] (or v_scale[j]).  Scales are device arrays float32
 * [num_kv_heads] owned by the caller; a per-tensor scale is the case where
 * all entries are equal.  Scales must be positive and finite (others are
 * not checked; they make the results meaningless, never unsafe).
 *
 * pa_reshape_and_cache_fp8 -- the cache write of pa_reshape_and_cache, with
 * each element x of KV head j stored as E4M3(x / scale_j): the quotient is
 * rounded to binary32 (IEEE division), then to E4M3 with round to nearest,
 * ties to even; finite magnitudes above 448 and infinities saturate to
 * +-448, NaN stays NaN.  k and v are in `dtype` (PA_F32, PA_BF16, PA_F16),
 * 16-byte aligned with token strides whose byte size is a multiple of 16;
 * head_dim a multiple of 16; k_cache and v_cache 16-byte aligned.
 */
int pa_reshape_and_cache_fp8(const void *k, const void *v, void *k_cache,
                             void *v_cache, const float *k_scale,
                             const float *v_scale, const int64_t *slot_mapping,
                             int64_t num_tokens, int32_t num_kv_heads,
                             int32_t head_dim, int64_t k_token_stride,
                             int64_t v_token_stride, int64_t num_blocks,
                             int32_t block_size, int32_t dtype, void *stream);

/*
 * pa_decode_fp8 / pa_decode_partitioned_fp8 -- pa_decode and
 * pa_decode_partitioned over E4M3 caches: K_s[t] = value(code) * k_scale[j]
 * and V_s[t] = value(code) * v_scale[j] for KV head j, the attention itself
 * unchanged.  `dtype` is the type of q and out: PA_BF16 or PA_F16 (q is
 * rounded to f16 for the tensor cores, so its entries must lie within the
 * f16 range, |q| < 65504).  The partitioned form takes the workspace of
 * pa_decode_partitioned_workspace_size and writes the same statistics.
 * Other requirements as pa_decode, plus q and out 16-byte aligned with a q
 * stride whose byte size is a multiple of 16.
 */
int pa_decode_fp8(void *out, const void *q, const void *k_cache,
                  const void *v_cache, const float *k_scale, const float *v_scale,
                  const int32_t *block_tables, const int32_t *seq_lens,
                  int32_t num_seqs, int32_t num_heads, int32_t num_kv_heads,
                  int32_t head_dim, int64_t num_blocks, int32_t block_size,
                  int32_t max_blocks_per_seq, int64_t q_seq_stride, float scale,
                  int32_t dtype, void *stream);

int pa_decode_partitioned_fp8(void *out, const void *q, const void *k_cache,
                              const void *v_cache, const float *k_scale,
                              const float *v_scale, const int32_t *block_tables,
                              const int32_t *seq_lens, int32_t num_seqs,
                              int32_t num_heads, int32_t num_kv_heads,
                              int32_t head_dim, int64_t num_blocks,
                              int32_t block_size, int32_t max_blocks_per_seq,
                              int64_t q_seq_stride, float scale, int32_t dtype,
                              int32_t partition_size, int32_t max_seq_len,
                              void *workspace, size_t workspace_bytes,
                              void *stream);

/*
 * pa_decode_cascade_workspace_size -- bytes of workspace pa_decode_cascade
 * needs for these sizes (fp32 partial results in the layout documented at
 * pa_decode_partitioned_workspace_size, with one partition per prefix chunk
 * followed by 512-token partitions of each sequence's own blocks).  Returns
 * 0 on invalid sizes (num_prefix_blocks must be positive).
 */
size_t pa_decode_cascade_workspace_size(int32_t num_seqs, int32_t num_heads,
                                        int32_t head_dim,
                                        int32_t num_prefix_blocks,
                                        int32_t max_blocks_per_seq);

/*
 * pa_decode_cascade -- decode for a batch whose sequences all begin with
 * the same physical blocks (a shared prompt: "vLLM: High-Throughput Serving
 * with PagedAttention", *How PagedAttention shares memory*; "vLLM:
 * Architecture, PagedAttention & Internals", *Prefix caching: reuse KV
 * across requests*), reading the shared blocks once per KV head instead of
 * once per sequence.
 *
 * Sequence s attends over 16 * num_prefix_blocks prefix tokens, held in the
 * physical blocks prefix_blocks[0 .. num_prefix_blocks) (int32, device),
 * followed by seq_lens[s] tokens of its own, held in block_tables[s][0 ..].
 * The result equals pa_decode over the concatenated table
 * (prefix_blocks ++ block_tables[s]) with seq_len 16 * num_prefix_blocks +
 * seq_lens[s].  The caller states the sharing (the block manager knows which
 * leading blocks a batch shares); nothing here compares tables.
 *
 * Work: the prefix is cut into chunks; per (chunk, KV head) the query heads
 * of all sequences, 128 (sequence, head) rows at a time, are multiplied
 * against the chunk's keys and values on the tensor cores (tcgen05); each
 * sequence's own blocks are decoded as 512-token split-KV partitions; a last
 * kernel merges every (sequence, head)'s partials by log-sum-exp.  Three
 * launches on `stream`.
 *
 * Requirements as pa_decode, plus: dtype PA_BF16 or PA_F16 (PA_F32:
 * PA_ERR_UNSUPPORTED when num_prefix_blocks > 0), q rows and out 16-byte
 * aligned, workspace_bytes >= pa_decode_cascade_workspace_size(...) with a
 * 256-byte aligned workspace.  num_prefix_blocks == 0 is pa_decode (no
 * workspace needed).  A prefix block id outside the pool is skipped and
 * flagged PA_DEVERR_BLOCK_ID; a seq_len past max_blocks_per_seq * 16 is
 * clamped and flagged PA_DEVERR_SEQ_LEN.
 */
int pa_decode_cascade(void *out, const void *q, const void *k_cache,
                      const void *v_cache, const int32_t *prefix_blocks,
                      int32_t num_prefix_blocks, const int32_t *block_tables,
                      const int32_t *seq_lens, int32_t num_seqs,
                      int32_t num_heads, int32_t num_kv_heads, int32_t head_dim,
                      int64_t num_blocks, int32_t block_size,
                      int32_t max_blocks_per_seq, int64_t q_seq_stride,
                      float scale, int32_t dtype, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * pa_decode_partitioned_noalloc -- pa_decode_partitioned without a caller
 * workspace, for callers that cannot allocate device memory where they
 * decode (for example while another stream is being captured into a CUDA
 * graph, under an allocator that forbids allocation after start-up, or in a
 * plug-in whose host program owns all device memory).  It is an addition of
 * this library with no counterpart on the reference pages.
 *
 * Same arguments, result and requirements as pa_decode_partitioned, minus
 * `workspace` and `workspace_bytes`: the partition workspace is a fixed
 * array of PA_NOALLOC_SCRATCH_BYTES compiled into the library, which every
 * GPU that loads the library holds until the process exits.  Problems whose
 * pa_decode_partitioned_workspace_size(...) exceeds that size are rejected
 * with PA_ERR_WORKSPACE before anything is launched.  Nothing is allocated
 * or freed (no cudaMalloc, cudaFree or allocating library routine).
 *
 * The arguments are checked in the same order, and bad ones refused with
 * the same status, as by pa_decode_partitioned.
 *
 * The first call on a device looks up the array's device address (with that
 * device current) and caches it; make that first call before any stream
 * capture.  The cached address belongs to the CUDA context it was looked up
 * in: after cudaDeviceReset (or anything else that destroys the device's
 * primary context) it is stale, and this entry point must not be called
 * again on that device in the same process.  All calls on a device share the
 * one array, which keeps whatever the last call left in it.  Every entry a
 * call reads is first written by the same call, so nothing needs clearing --
 * except after PA_DEVERR_TIMEOUT, when the output is undefined and may mix in
 * an earlier call's partials (see pa_decode_partitioned).  Calls whose
 * kernels may overlap on the GPU -- on different streams, or from several
 * host threads -- race on the array and must be serialised by the caller.
 */
#define PA_NOALLOC_SCRATCH_BYTES (32u << 20)

int pa_decode_partitioned_noalloc(void *out, const void *q, const void *k_cache,
                                  const void *v_cache, const int32_t *block_tables,
                                  const int32_t *seq_lens, int32_t num_seqs,
                                  int32_t num_heads, int32_t num_kv_heads,
                                  int32_t head_dim, int64_t num_blocks,
                                  int32_t block_size, int32_t max_blocks_per_seq,
                                  int64_t q_seq_stride, float scale, int32_t dtype,
                                  int32_t partition_size, int32_t max_seq_len,
                                  void *stream);

/* Human-readable text of a pa_status (static storage). */
const char *pa_status_string(int status);

/*
 * pa_device_error -- read the sticky device error word of the current device
 * into *flags (PA_DEVERR_* bits) and clear it when `clear` is non-zero.
 * Synchronises the device first.  Returns PA_OK or PA_ERR_CUDA.
 */
int pa_device_error(uint32_t *flags, int clear);

/*
 * pa_test_stall_next_decode -- test hook for the kernels' bounded waits.  The
 * next decode call (any pa_decode* entry point, from any host thread) makes
 * the first copy of every warp of its persistent kernel expect 16 bytes more
 * than it delivers, so the wait for that copy runs out at its 1 s limit: the
 * kernel sets PA_DEVERR_TIMEOUT, waits (bounded) for its copies in flight and
 * returns, leaving that call's output incomplete (the call takes ~2 s).  The
 * context stays usable.  For tests of the error path only.  Returns PA_OK.
 */
int pa_test_stall_next_decode(void);

/* ABI version of this header (increments on any signature change or addition). */
int pa_abi_version(void);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
