/*
 * pa_block_manager.h -- host-side block manager of libpa.so: the bookkeeping
 * that produces the metadata the kernels of pa.h consume (block tables,
 * sequence lengths, slot mappings, copy-on-write block pairs).
 *
 * The method ("03 - Engines Papers", section 2 PagedAttention (vLLM): Key
 * trick and What to extract; "The LLM inference engine playbook", Theme 3):
 *  - the KV cache is a pool of fixed-size physical blocks; each sequence owns
 *    a block table mapping its logical block j to a physical block id;
 *  - physical blocks can be shared between sequences (fork for parallel
 *    sampling / beam search, or reuse of a cached prompt prefix); each block
 *    carries a refcount, and a write into a block whose refcount is above one
 *    first copies it to a private block (copy on write);
 *  - prefix reuse, hash flavour ("03 - Engines Papers", section 4 SGLang
 *    (RadixAttention): What to extract, automatic prefix caching; playbook
 *    Theme 3): every full block is keyed by a hash chained over its parent
 *    block's key and its own token ids, so a new request whose prompt starts
 *    with the same full blocks reuses them instead of recomputing; blocks no
 *    sequence references stay cached and are evicted least recently released
 *    first (the cache is a cache, not a database: LRU eviction).
 *
 * Policy (deterministic, so that results can be compared exactly):
 *  - free blocks form a FIFO queue that starts as 0, 1, ..., num_blocks-1;
 *    a released block that holds no cached prefix goes to its tail when
 *    the step ends;
 *  - allocation takes the head of the free queue; when it is empty, it
 *    evicts the least recently released cached block (refcount 0) and takes
 *    that; when there is none, the call fails with PA_ERR_NO_BLOCKS and
 *    changes nothing;
 *  - a sequence's blocks are released last block first, so its tail blocks
 *    are evicted before its head blocks;
 *  - a block is registered in the prefix cache when it becomes full (at
 *    admission for the prompt's full blocks, or when an appended token fills
 *    it), unless an identical chain already holds a registered block;
 *  - admission reuses the longest run of registered full blocks that matches
 *    the prompt from its start, keeping at least the prompt's last token to
 *    compute (at most floor((n - 1) / block_size) blocks are reused).
 *    Matches compare the token ids and the parent block, not the hash alone.
 *
 * Steps.  The calls between two pa_bm_end_step calls build one step's
 * metadata; the caller then runs, in stream order, pa_copy_blocks on the
 * step's copy pairs, the scatter of the step's new tokens (the slots handed
 * out), and the attention.  pa_copy_blocks runs its pairs concurrently and
 * before the scatter, so within one step:
 *  - a block released to refcount 0 is parked until the step ends (it can be
 *    neither reallocated nor evicted, so no pending copy reads or writes a
 *    block that is handed out again, and no slot is handed out twice); a
 *    parked block that holds a cached prefix can still be reused by a match;
 *  - a copy on write of a block that already got a slot in this step is
 *    refused with PA_ERR_BM_STEP (its copy would miss that token): end the
 *    step first.
 * A block registered at admission is filled by the same step's scatter,
 * which the stream orders before any reader.
 *
 * Every function is host-only and touches no GPU.  A manager is not thread
 * safe: one thread (the scheduler) drives it.  Status codes are those of
 * pa.h plus PA_ERR_NO_BLOCKS and PA_ERR_BM_STEP.
 */
#ifndef PA_BLOCK_MANAGER_H_
#define PA_BLOCK_MANAGER_H_

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* The pool has no free block and no evictable cached block. */
#define PA_ERR_NO_BLOCKS (-6)
/* The call needs the current step to end first (see Steps above). */
#define PA_ERR_BM_STEP (-7)

typedef struct pa_block_manager pa_block_manager;

/* A manager of `num_blocks` physical blocks of `block_size` token slots
 * (block_size >= 1; the kernels of pa.h need 16).  prefix_caching != 0
 * enables the prefix cache.  Returns NULL on bad arguments or when memory
 * for the bookkeeping cannot be had. */
pa_block_manager *pa_bm_create(int64_t num_blocks, int block_size, int prefix_caching);
void pa_bm_destroy(pa_block_manager *bm);

/* Admit sequence `seq_id` (not live yet) with prompt tokens[0..n) (n >= 1).
 * Reuses cached prefix blocks, allocates the rest, and writes slots[0..n):
 * -1 for the *num_cached reused tokens (their KV is already in the pool),
 * else the slot each token's K/V is to be scattered to.  On
 * PA_ERR_NO_BLOCKS nothing changes. */
int pa_bm_add_sequence(pa_block_manager *bm, int64_t seq_id, const int32_t *tokens, int n,
                       int64_t *slots, int *num_cached);

/* Append one token to a live sequence and write the slot its K/V goes to.
 * A new block is allocated when the last one is full; a shared last block
 * (refcount > 1) is first copied to a private block, recorded as a copy pair
 * of the step (see pa_bm_end_step); PA_ERR_BM_STEP if that block already got
 * a slot in this step.  On an error nothing changes. */
int pa_bm_append_token(pa_block_manager *bm, int64_t seq_id, int32_t token, int64_t *slot);

/* One decode step's appends in one call: tokens[i] to seq_ids[i] for i in
 * [0, n), in order, writing slots[i], exactly as n calls of
 * pa_bm_append_token.  Stops at the first failing append and returns the
 * number done (n when all succeed); *status gets PA_OK or the failing
 * append's status, and the appends before it stay done. */
int pa_bm_append_tokens(pa_block_manager *bm, const int64_t *seq_ids, const int32_t *tokens,
                        int n, int64_t *slots, int *status);

/* New sequence `child_id` sharing every block of live sequence `parent_id`
 * (refcounts + 1): parallel sampling / beam search. */
int pa_bm_fork(pa_block_manager *bm, int64_t parent_id, int64_t child_id);

/* End a sequence and release its blocks (last block first; a block whose
 * refcount reaches 0 is parked until the step ends). */
int pa_bm_free_sequence(pa_block_manager *bm, int64_t seq_id);

/* Copy pairs of the current step so far. */
int64_t pa_bm_num_step_copies(const pa_block_manager *bm);

/* End the current step: write its copy-on-write pairs (src, dst block ids,
 * in the order they arose) to pairs[0 .. 2 * count) and return count (>= 0);
 * then the parked blocks become reusable (cached ones join the eviction
 * order, released in the order they were parked; the rest join the free
 * queue).  The pairs are the input of pa_copy_blocks for this step.
 * PA_ERR_INVALID, with nothing changed, if max_pairs is below the count. */
int pa_bm_end_step(pa_block_manager *bm, int64_t *pairs, int max_pairs);

/* Metadata of a batch: for seq_ids[0..n), block table rows
 * tables[n * max_blocks] (entries past a sequence's blocks are -1) and
 * seq_lens[n].  PA_ERR_INVALID if an id is not live or a sequence has more
 * than max_blocks blocks. */
int pa_bm_build_tables(const pa_block_manager *bm, const int64_t *seq_ids, int n,
                       int32_t *tables, int max_blocks, int32_t *seq_lens);

/* Introspection. */
int64_t pa_bm_num_free_blocks(const pa_block_manager *bm);   /* free queue length */
int64_t pa_bm_num_parked_blocks(const pa_block_manager *bm); /* released in this step */
int64_t pa_bm_num_cached_blocks(const pa_block_manager *bm); /* registered blocks, in use or not */
int64_t pa_bm_num_evictable_blocks(const pa_block_manager *bm); /* registered, refcount 0 */
int pa_bm_refcount(const pa_block_manager *bm, int64_t block);   /* -1 if out of range */
int64_t pa_bm_seq_len(const pa_block_manager *bm, int64_t seq_id); /* -1 if not live */

#ifdef __cplusplus
}
#endif

#endif /* PA_BLOCK_MANAGER_H_ */
