/*
 * pa_blocks.h -- C ABI of the host-side block manager and serving loop that
 * feed the paged-attention kernels of pa.h (block tables, slot mappings,
 * copy-on-write copies), one step at a time.
 *
 * Defined in "vLLM: Architecture, PagedAttention & Internals":
 *   *The free list and the block table* -- a free list of physical block
 *     ids, per-block reference counts, allocation of ceil(n / block_size)
 *     blocks for a prompt, append_slot taking a new block only when the next
 *     token starts one, release when the last owner frees a block;
 *   *Copy-on-write for shared blocks* -- a write into a shared, partly
 *     filled block first moves the writer to a fresh block and emits a
 *     (src, dst) copy (executed on the GPU by pa_copy_blocks);
 *   *Prefix caching: reuse KV across requests* -- a full block is known by
 *     everything before it plus its own tokens and an extra key (adapter id,
 *     cache salt); a new request reuses its leading cached blocks and
 *     allocates the rest; unreferenced cached blocks stay until evicted.
 * and "vLLM: High-Throughput Serving with PagedAttention" (lesson 13.15),
 *   *Practice: try it yourself* -- the serving loop of pa_loop_*.
 *
 * Readings where the pages leave a choice:
 *   - the free list is popped from its end; freed blocks are put at its
 *     front, the blocks of one sequence in reverse order, so never-used
 *     blocks go first, then the least recently freed, and a sequence's leaf
 *     blocks before its root blocks;
 *   - a prompt's full blocks become matchable when the request is added, a
 *     decoded block when its last slot is written; if the same identity is
 *     already cached the block stays private;
 *   - a block's identity is a 128-bit chained hash of (extra key, all tokens
 *     up to the block's end), checked together with the block's own tokens
 *     and extra key on every match.
 *
 * Everything here is host memory and host code; nothing launches a kernel.
 * Calls on one handle must not run concurrently; distinct handles are
 * independent.  Sequence and request ids are caller-chosen int64 values.
 *
 * Status: PA_OK (0), PA_BM_FULL (1: not enough free blocks; nothing changed),
 * or a negative pa_status of pa.h (PA_ERR_INVALID_ARG for unknown or
 * duplicate ids, bad sizes or NULL pointers).
 */
#ifndef PA_BLOCKS_H_
#define PA_BLOCKS_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define PA_BM_FULL 1

typedef struct pa_bm pa_bm;

/*
 * A manager of num_blocks blocks of block_size tokens.  free_order (NULL:
 * 0, 1, ..., num_blocks-1) is the initial free list, a permutation of the
 * block ids; its LAST entry is handed out first.  prefix_caching != 0
 * enables matching of full blocks across sequences.  Returns NULL on bad
 * arguments or allocation failure.  The handle owns its memory; free it with
 * pa_bm_destroy.
 */
pa_bm *pa_bm_create(int32_t num_blocks, int32_t block_size, const int32_t *free_order,
                    int32_t prefix_caching);
void pa_bm_destroy(pa_bm *bm);

/* Blocks on the free list (never used, or released and possibly cached). */
int32_t pa_bm_num_free(const pa_bm *bm);

/* 1 if a prompt of num_tokens tokens fits without any cache hit, else 0. */
int32_t pa_bm_can_allocate(const pa_bm *bm, int64_t num_tokens);

/*
 * Add sequence seq_id holding tokens[0 .. n) (n >= 0; tokens may be NULL,
 * meaning all zeros) with the given extra key.  With prefix caching its
 * leading full blocks are matched first; *num_cached (may be NULL) receives
 * the number of tokens in matched blocks.  PA_BM_FULL if the remaining
 * blocks do not fit.
 */
int pa_bm_add_sequence(pa_bm *bm, int64_t seq_id, const int32_t *tokens, int64_t n,
                       int64_t extra, int64_t *num_cached);

/* child shares every block of parent (reference counts + 1), same tokens. */
int pa_bm_fork(pa_bm *bm, int64_t parent, int64_t child);

/*
 * Room for the next token of seq_id (at position seq_len): *slot receives
 * block * block_size + position % block_size.  A new block is taken when the
 * position starts one; if the last block is shared and partly filled, the
 * sequence moves to a fresh block first and (*copy_src, *copy_dst) receive
 * the copy to execute before the write, else both are -1.  PA_BM_FULL if a
 * block is needed and none is free.
 */
int pa_bm_append(pa_bm *bm, int64_t seq_id, int32_t token, int64_t *slot,
                 int32_t *copy_src, int32_t *copy_dst);

/* Release seq_id's blocks (and forget the sequence). */
int pa_bm_free(pa_bm *bm, int64_t seq_id);

/* Length of seq_id's block table (written to out[0 .. min(len, cap))),
 * or -1 for an unknown id. */
int32_t pa_bm_table(const pa_bm *bm, int64_t seq_id, int32_t *out, int32_t cap);

/* Tokens held by seq_id, or -1 for an unknown id. */
int64_t pa_bm_seq_len(const pa_bm *bm, int64_t seq_id);

/* Reference count of a block (0 when free), or -1 for a bad id. */
int32_t pa_bm_refcount(const pa_bm *bm, int32_t block);

/*
 * The decode inputs of a batch: row i of tables ([n][width], row-major)
 * receives seq_ids[i]'s block table padded with `pad`, seq_lens[i] its
 * length.  PA_ERR_INVALID_ARG if an id is unknown or a table is wider than
 * width.
 */
int pa_bm_batch(const pa_bm *bm, const int64_t *seq_ids, int32_t n, int32_t *tables,
                int32_t width, int32_t pad, int32_t *seq_lens);

/*
 * Leading blocks every sequence of seq_ids[0 .. n) shares: the largest P such
 * that all their tables hold the same physical block at each of positions
 * 0 .. P-1 and every one of them holds at least block_size * P tokens (the
 * prefix a cascade decode, pa_decode_cascade, reads once).  0 for n == 0 or when
 * nothing is shared; PA_ERR_INVALID_ARG for an unknown id.
 */
int32_t pa_bm_common_prefix(const pa_bm *bm, const int64_t *seq_ids, int32_t n);

/* ---- serving loop ----------------------------------------------------------
 *
 * The pages' toy serving loop over a block manager (which it does not own;
 * use one without prefix caching): requests wait in a FIFO queue; each
 * iteration admits queued requests in order while the first one's blocks
 * fit, then advances the step and lets every running request, in admission
 * order, write one token (taking a block when the token starts one); when a
 * request needs a block and none is free, the most recently admitted running
 * request is preempted: its blocks are released and it returns to the front
 * of the queue holding the tokens it had, to be prefilled again.  A request
 * finishes when it has written its output tokens and releases its blocks.
 */

typedef struct pa_loop pa_loop;

enum { PA_EV_ADMIT = 0, PA_EV_PREEMPT = 1, PA_EV_FINISH = 2 };

pa_loop *pa_loop_create(pa_bm *bm);
void pa_loop_destroy(pa_loop *loop);

/* Queue request id holding `tokens` tokens with max_new tokens to write. */
int pa_loop_submit(pa_loop *loop, int64_t id, int64_t tokens, int64_t max_new);

/*
 * One iteration.  events ([cap][5] int64: step, PA_EV_*, id, tokens, free
 * blocks after the event) receive this iteration's events in order;
 * written ([cap][2] int64: id, slot) the requests that wrote a token this
 * step with the slot of that token, in order.  Returns 1 if requests remain,
 * 0 when all are finished, or PA_ERR_INVALID_ARG if a buffer is too small
 * (sized num_requests * 3 events and num_requests written rows, this never
 * happens), if a queued request cannot fit even into an empty pool, or if a
 * submitted id is already running.  *step receives the step reached.
 */
int pa_loop_step(pa_loop *loop, int64_t *events, int32_t events_cap, int32_t *num_events,
                 int64_t *written, int32_t written_cap, int32_t *num_written, int64_t *step);

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCKS_H_ */
