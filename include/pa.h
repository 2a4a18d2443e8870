/*
 * pa.h -- C ABI of libpa.so: paged attention over a block-table-addressed
 * KV cache on GB300 (sm_103a).
 *
 * The method: keys and values live in fixed-size physical blocks of 16
 * tokens; a per-sequence block table maps logical positions to physical
 * blocks, like virtual memory; blocks may be shared between sequences with
 * refcounts and copied on write ("03 - Engines Papers", section 2, Efficient
 * Memory Management for LLM Serving with PagedAttention (vLLM): Key trick and
 * What to extract; "The LLM inference engine playbook: tricks in vLLM and
 * SGLang", Theme 3).  The attention kernel gathers K/V from those
 * non-contiguous blocks (same section), tiles them through on-chip memory with
 * an online softmax (FlashAttention and Milakov & Gimelshein, "References"
 * page), splits long contexts over KV partitions and reduces the partial
 * softmaxes by log-sum-exp ("The LLM inference engine playbook", Theme 4;
 * "03 - Engines Papers", section 12 Cascade Inference), and serves the
 * prefill chunks of a Sarathi hybrid batch next to the decodes
 * ("03 - Engines Papers", section 3 Sarathi / Sarathi-Serve).
 *
 * Common conventions
 *  - Every pointer argument named *device* below is a CUDA device pointer the
 *    caller owns; the library never frees, retains or allocates memory.
 *    Every call is asynchronous on `stream` (a cudaStream_t passed as void*;
 *    NULL = the legacy default stream).
 *  - bf16 tensors are row-major and contiguous unless a stride is given:
 *      q        [num_q_tokens, num_q_heads, head_dim]
 *      out      [num_q_tokens, num_q_heads, head_dim]
 *      k_cache, v_cache [num_blocks, block_size, num_kv_heads, head_dim]
 *      block_tables int32 [num_seqs, max_blocks_per_seq]
 *      seq_lens     int32 [num_seqs]
 *      slot_mapping int64 [num_tokens], slot = block * block_size + offset
 *  - GQA: query head h reads kv head h / (num_q_heads / num_kv_heads).
 *  - block_size must be 16 and head_dim 64 or 128; num_q_heads /
 *    num_kv_heads must be an integer in [1, 8] (PA_ERR_UNSUPPORTED otherwise).
 *  - Scores are scale * <q, k>; lse outputs are natural-log log-sum-exp of
 *    the scaled scores, fp32.  A sequence with seq_len == 0 yields out = 0 and
 *    lse = -inf.
 *  - Arguments are checked on the host before anything is launched; a
 *    failing check returns PA_ERR_INVALID / PA_ERR_UNSUPPORTED /
 *    PA_ERR_WORKSPACE and touches nothing.  A launch failure returns
 *    PA_ERR_CUDA.  Device-side checks (block id or slot out of range, a
 *    length beyond the table) never fault: the offending access is skipped or
 *    clamped and a bit is set in the device error word (pa_device_error_flags).
 *    No call aborts, exits or traps.
 */
#ifndef PA_H_
#define PA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef enum pa_status {
  PA_OK = 0,
  PA_ERR_INVALID = -1,     /* bad pointer, size or metadata */
  PA_ERR_UNSUPPORTED = -2, /* valid but not implemented (head_dim, group, block_size) */
  PA_ERR_CUDA = -3,        /* a CUDA runtime call or launch failed */
  PA_ERR_WORKSPACE = -4,   /* workspace missing, too small or misaligned */
  PA_ERR_SCRATCH_LIMIT = -5 /* pa_decode_noalloc: needs more than its static scratch */
} pa_status;

/* Bits of the device error word. */
#define PA_DEVERR_BLOCK_ID 1u  /* block-table entry outside [0, num_blocks) */
#define PA_DEVERR_SEQ_LEN 2u   /* seq_len < 0 or > max_blocks_per_seq * block_size */
#define PA_DEVERR_SLOT 4u      /* slot >= num_blocks * block_size (skipped) */
#define PA_DEVERR_TIMEOUT 8u   /* a pipeline wait ran past its iteration limit */
#define PA_DEVERR_CHUNK 16u    /* prefill chunk metadata inconsistent (skipped) */
#define PA_DEVERR_GROUP 32u    /* cascade group / shared-block metadata out of range (clamped) */

/* Human-readable name of a pa_status value.  Never NULL. */
const char *pa_status_string(int status);

/* ABI version, (major << 16) | minor. */
int pa_version(void);

/*
 * Slot scatter ("reshape and cache"): for every new token t with
 * slot_mapping[t] >= 0,
 *   k_cache[slot / block_size][slot % block_size][h][:] = key[t][h][:]
 *   v_cache[...same...]                                 = value[t][h][:]
 * for all kv heads h -- a bit-exact copy.  A negative slot is padding and is
 * skipped.  The paged layout it writes is the one the block table addresses
 * ("03 - Engines Papers", section 2, Key trick).
 *   key, value        device, bf16, row t at key + t * key_token_stride
 *                     (strides in elements, multiples of 8; head h at + h*head_dim)
 *   k_cache, v_cache  device, bf16 [num_blocks, block_size, num_kv_heads, head_dim]
 *   slot_mapping      device, int64 [num_tokens]
 * Duplicate non-negative slots are invalid input (the surviving value is
 * unspecified); pa_validate_metadata detects them.
 */
int pa_reshape_and_cache(const void *key, const void *value, int64_t key_token_stride,
                         int64_t value_token_stride, void *k_cache, void *v_cache,
                         const int64_t *slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int64_t num_blocks, void *stream);

/*
 * Copy-on-write support: copy whole physical blocks of both pools,
 * k_cache[dst] = k_cache[src], v_cache[dst] = v_cache[src], bit-exact, for
 * every pair (src, dst) in block_pairs (device, int64 [num_pairs, 2]).  A
 * sequence about to write into a block whose refcount is above one is given
 * a private copy first ("03 - Engines Papers", section 2, copy-on-write with
 * refcounts).  Destinations must be distinct and must not be sources.
 */
int pa_copy_blocks(void *k_cache, void *v_cache, const int64_t *block_pairs, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                   void *stream);

/*
 * Bytes of workspace pa_decode needs for these sizes and partition_tokens,
 * on the current device.  0 when no workspace is needed.  Returns 0 and sets
 * nothing on invalid sizes (pa_decode then reports the error).
 */
size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int max_blocks_per_seq, int block_size, int partition_tokens);

/*
 * Paged decode attention: one query per sequence, attending over positions
 * [0, seq_lens[s]) of its paged KV (this step's new token included, so the
 * scatter runs first):
 *   out[s][h] = sum_j softmax_j(scale * <q[s][h], K_s[j]>) V_s[j],
 *   K_s[j] = k_cache[block_tables[s][j / 16]][j % 16][h / group]
 * ("03 - Engines Papers", section 2, the PagedAttention kernel gathering K/V
 * from non-contiguous blocks; online softmax per "References", Milakov &
 * Gimelshein).
 *   out        device bf16 [num_seqs, num_q_heads, head_dim]
 *   q          device bf16 [num_seqs, num_q_heads, head_dim]
 *   out_lse    device fp32 [num_seqs, num_q_heads] or NULL
 * partition_tokens selects how the KV is split across the GPU:
 *   < 0  single pass: each (sequence, kv head) is one work item; no workspace.
 *   = 0  balanced: the total KV is cut into equal contiguous ranges, one per
 *        persistent CTA; pieces of a sequence that straddle ranges are merged
 *        by log-sum-exp inside the same launch.  Needs workspace, which must
 *        be zero-filled before its first use (the kernel leaves it zeroed).
 *   > 0  split-KV with fixed partitions of partition_tokens tokens (a multiple
 *        of block_size): partition p covers [p * P, (p + 1) * P) and writes a
 *        partial (o_p, lse_p) to the workspace, laid out exactly as
 *        pa_merge_partials reads it; a merge kernel then combines them
 *        (partial buffers first: part_out [S, Hq, P_max, D] fp32, then part_lse
 *        [S, Hq, P_max] fp32, P_max = ceil(max_blocks_per_seq * 16 / P)).
 * A workspace may not be shared by two calls in flight at the same time.
 */
int pa_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
              const int32_t *block_tables, int max_blocks_per_seq, const int32_t *seq_lens,
              int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
              int64_t num_blocks, float scale, int partition_tokens, float *out_lse,
              void *workspace, size_t workspace_bytes, void *stream);

/*
 * Cascade decode: decode of pa_decode for batches whose sequences share
 * prompt prefixes ("03 - Engines Papers", section 12 Cascade Inference /
 * Multi-Query Cascade Attention): the attention over a group's shared prefix
 * is computed once for all the group's queries, batched, and combined with
 * each sequence's private-suffix attention by log-sum-exp.  The result is the
 * same as pa_decode's (same formula, same outputs).
 *
 * Groups: the sequences are ordered by group; group g holds sequences
 * [group_offsets[g], group_offsets[g + 1]) (device, int32 [num_groups + 1],
 * group_offsets[0] = 0, group_offsets[num_groups] = num_seqs, each group at
 * most max_group_size sequences, max_group_size * (num_q_heads /
 * num_kv_heads) <= 32).  A sequence with nothing shared forms its own group
 * or has shared_blocks = 0.
 *   prefix_tables  device, int32 [num_groups, max_prefix_blocks]: the
 *                  physical blocks of group g's shared prefix, in order
 *   shared_blocks  device, int32 [num_seqs]: sequence s's first
 *                  shared_blocks[s] table entries are prefix_tables[g][0 ..
 *                  shared_blocks[s]) (the caller guarantees it); its tokens
 *                  [0, min(len, 16 * shared_blocks[s])) are attended in the
 *                  group's prefix pass, the rest [16 * shared_blocks[s], len)
 *                  through its own table in the suffix pass
 * Other arguments, modes and outputs as pa_decode (head_dim 128).  The
 * workspace (pa_cascade_workspace_size, 256-byte aligned) holds the prefix
 * pass's fp32 partials followed by pa_decode's workspace, which must be
 * zero-filled before its first use as for pa_decode.  Out-of-range group or
 * shared-block metadata sets PA_DEVERR_GROUP and is clamped, never faults.
 */
size_t pa_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size, int partition_tokens);
int pa_cascade_decode(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *seq_lens, int num_seqs, const int32_t *group_offsets,
                      int num_groups, int max_group_size, const int32_t *prefix_tables,
                      int max_prefix_blocks, const int32_t *shared_blocks, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                      float scale, int partition_tokens, float *out_lse, void *workspace,
                      size_t workspace_bytes, void *stream);

/*
 * FP8 (E4M3) KV cache: the pools hold one byte per element, with one
 * dequantization scale per kv head for K and one for V (pass the same value
 * for every head to get a per-tensor scale).  Both engines of the pages ship
 * an FP8 KV cache with per-tensor or per-head scales, and quantizing the
 * cache is the "shrink the cache" lever ("The LLM inference engine playbook",
 * Theme 3); decode reads half the bytes of a bf16 pool.
 *
 * E4M3: 1 sign bit, 4 exponent bits (bias 7), 3 mantissa bits; no infinity;
 * the largest finite magnitude is 448; 0x7F / 0xFF are NaN.
 *
 * pa_reshape_and_cache_fp8 -- quantizing slot scatter: for every new token t
 * with slot_mapping[t] >= 0 and every element x of key[t][h] (likewise V):
 *   code = E4M3(x / k_scales[h])
 * where the division is IEEE fp32 (correctly rounded) and E4M3() rounds to
 * nearest, ties to even, saturating finite values beyond +-448 to +-448.
 * Arguments as pa_reshape_and_cache, except
 *   k_cache, v_cache  device, uint8 [num_blocks, block_size, num_kv_heads, head_dim]
 *   k_scales, v_scales device, fp32 [num_kv_heads], positive and finite
 */
int pa_reshape_and_cache_fp8(const void *key, const void *value, int64_t key_token_stride,
                             int64_t value_token_stride, void *k_cache, void *v_cache,
                             const int64_t *slot_mapping, const float *k_scales,
                             const float *v_scales, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int64_t num_blocks, void *stream);

/* pa_copy_blocks for E4M3 pools (bytes; head_dim a multiple of 16). */
int pa_copy_blocks_fp8(void *k_cache, void *v_cache, const int64_t *block_pairs, int num_pairs,
                       int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                       void *stream);

/*
 * pa_decode over E4M3 pools: the attention of pa_decode with
 *   K_s[j] = e4m3_value(k_cache[...]) * k_scales[h / group]
 *   V_s[j] = e4m3_value(v_cache[...]) * v_scales[h / group]
 * (the dequantized cache).  head_dim must be 128.  Same arguments, modes,
 * workspace (sized by pa_decode_workspace_size) and outputs as pa_decode,
 * plus the two scale arrays (device, fp32 [num_kv_heads]).  The contraction
 * runs on f16 copies of the E4M3 values (exact) with the queries scaled by a
 * power of two per sequence and kv head, fp32 accumulation.
 */
int pa_decode_fp8(void *out, const void *q, const void *k_cache, const void *v_cache,
                  const float *k_scales, const float *v_scales, const int32_t *block_tables,
                  int max_blocks_per_seq, const int32_t *seq_lens, int num_seqs,
                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int64_t num_blocks, float scale, int partition_tokens, float *out_lse,
                  void *workspace, size_t workspace_bytes, void *stream);

/*
 * Log-sum-exp merge of partial attentions ("03 - Engines Papers", section 12
 * Cascade Inference, merged via LSE; split-K softmax reduction, "The LLM
 * inference engine playbook", Theme 4):
 *   L = max_p lse_p,  w_p = exp(lse_p - L),
 *   out = sum_p w_p o_p / sum_p w_p,  lse = L + ln sum_p w_p
 * over p < num_parts[s].  Parts with lse = -inf have weight 0; if every part
 * is -inf the output is 0 and lse -inf.
 *   part_out  device fp32 [num_seqs, num_q_heads, max_parts, head_dim]
 *   part_lse  device fp32 [num_seqs, num_q_heads, max_parts]
 *   num_parts device int32 [num_seqs], each in [0, max_parts]
 *   out       device bf16 [num_seqs, num_q_heads, head_dim]; out_lse fp32 or NULL
 */
int pa_merge_partials(void *out, float *out_lse, const float *part_out, const float *part_lse,
                      const int32_t *num_parts, int num_seqs, int num_q_heads, int head_dim,
                      int max_parts, void *stream);

/*
 * Causal prefill chunks of a hybrid batch ("03 - Engines Papers", section 3
 * Sarathi / Sarathi-Serve: long prefills split into chunks co-scheduled with
 * decodes; a chunk's queries see the K/V of earlier positions and of the chunk
 * itself, not of later chunks).  Chunk c owns query rows
 * [cu_q_lens[c], cu_q_lens[c + 1]); row i sits at absolute position
 * q_start_pos[c] + i and attends over keys 0 .. that position of sequence c
 * (block table row c), which holds seq_lens[c] >= q_start_pos[c] + q_len
 * tokens (the chunk's own K/V already scattered).  Runs on tcgen05 tensor
 * cores with fp32 accumulation in tensor memory.
 *   q, out     device bf16 [total_q_tokens, num_q_heads, head_dim]
 *   cu_q_lens  device int32 [num_chunks + 1]; q_start_pos, seq_lens int32 [num_chunks]
 *   max_q_len  host int, an upper bound of every chunk's query count
 *   out_lse    device fp32 [total_q_tokens, num_q_heads] or NULL
 * head_dim must be 128 for this call.  A chunk whose metadata is inconsistent
 * (rows outside [0, total_q_tokens), q_start_pos + q_len > seq_len, or
 * seq_len beyond its table row) is skipped, its rows left unwritten, and
 * sets PA_DEVERR_CHUNK.
 */
int pa_prefill_chunk(void *out, const void *q, const void *k_cache, const void *v_cache,
                     const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *cu_q_lens, const int32_t *q_start_pos,
                     const int32_t *seq_lens, int num_chunks, int total_q_tokens, int max_q_len,
                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                     int64_t num_blocks, float scale, float *out_lse, void *stream);

/*
 * Bytes of workspace pa_hybrid_attention needs (a balanced decode's workspace
 * plus 256 reserved bytes); 0 on invalid sizes.
 */
size_t pa_hybrid_workspace_size(int num_decode_seqs, int num_q_heads, int num_kv_heads,
                                int head_dim, int max_blocks_per_seq, int block_size);

/*
 * One Sarathi hybrid batch ("03 - Engines Papers", section 3 Sarathi /
 * Sarathi-Serve: a step carries prefill chunks next to decodes under one
 * token budget) in one call, after pa_reshape_and_cache of all the step's
 * new tokens: the prefill chunks of pa_prefill_chunk (chunk arguments, same
 * meaning and layouts) and the balanced decode of pa_decode with
 * partition_tokens = 0 (decode arguments).  Both read the same pools.
 *
 * One kernel launch: its first CTAs (num_sms - chunk_sms, rounded down to
 * an even count) run the balanced decode, one per SM, and the rest run the
 * chunk's query tiles as tensor-core CTA pairs, which start at once on the SMs
 * the decode leaves free, so the chunk's tensor-core work runs under the
 * decode's HBM streaming instead of after it.  chunk_sms = 0 picks about a
 * seventh of the SMs (22 of 152); values are clamped to [1, num_sms - 2].  The chunk reads
 * nothing the decode writes; work queued after the call on the stream sees
 * both results.  With no chunk (or no decode) the call is pa_decode (or
 * pa_prefill_chunk) alone.  The decode of this call needs head_dim 128
 * (PA_ERR_UNSUPPORTED otherwise), as the chunk does.
 *   workspace  device, pa_hybrid_workspace_size bytes, 256-byte aligned,
 *              zero-filled before its first use (calls leave it zeroed);
 *              one call in flight per workspace.
 * Errors as pa_decode and pa_prefill_chunk; every argument is checked before
 * anything is launched, except device errors, which surface at the caller's
 * synchronization (pa_device_error_flags).
 */
int pa_hybrid_attention(void *out_chunk, const void *q_chunk, const int32_t *chunk_block_tables,
                        int chunk_max_blocks, const int32_t *cu_q_lens,
                        const int32_t *q_start_pos, const int32_t *chunk_seq_lens,
                        int num_chunks, int total_q_tokens, int max_q_len, float *chunk_lse,
                        void *out_decode, const void *q_decode,
                        const int32_t *decode_block_tables, int decode_max_blocks,
                        const int32_t *decode_seq_lens, int num_decode_seqs, float *decode_lse,
                        const void *k_cache, const void *v_cache, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                        float scale, int chunk_sms, void *workspace, size_t workspace_bytes,
                        void *stream);

/*
 * pa_hybrid_attention_append -- one Sarathi hybrid step with the step's slot
 * scatter fused in ("03 - Engines Papers", section 3 Sarathi / Sarathi-Serve:
 * a step carries a prefill chunk and decodes; section 2 PagedAttention: the
 * step's new K/V go into their slots before attention reads them).  The
 * result is that of pa_reshape_and_cache of every new row, then
 * pa_hybrid_attention with the same arguments, in one kernel launch:
 *   key_chunk / value_chunk  device bf16 [total_q_tokens, *, Hkv, D], row i
 *              the K / V of query row i of the chunk inputs; chunk c's row
 *              q0 + t (q0 = cu_q_lens[c]) goes into the slot of position
 *              q_start_pos[c] + t of chunk c's block table;
 *   key_decode / value_decode  device bf16 [num_decode_seqs, *, Hkv, D], row
 *              s the new token of decode s, which goes into the slot of
 *              position decode_seq_lens[s] - 1 (as pa_decode_append);
 *   key_token_stride / value_token_stride  elements between consecutive rows
 *              of both the chunk's and the decodes' arrays (>= Hkv * D, a
 *              multiple of 8); pointers 16-byte aligned.
 * The chunk's keys at its own positions are read from key_chunk / value_chunk,
 * not from the pool the same launch is writing, so every chunk must start a
 * block: q_start_pos[c] a multiple of 16 (chunks of a multiple of 16 tokens
 * after whole cached blocks are).  A chunk that does not is skipped and
 * flagged (PA_DEVERR_CHUNK); use pa_reshape_and_cache + pa_hybrid_attention
 * for it.  Slots receiving new rows must be owned by their sequence alone
 * (copy-on-write done before).  Every other argument, the workspace and the
 * errors as pa_hybrid_attention; with no decodes the launch runs the chunk
 * alone (workspace unused), with no chunk it is pa_decode_append.
 */
int pa_hybrid_attention_append(
    void *out_chunk, const void *q_chunk, const void *key_chunk, const void *value_chunk,
    const int32_t *chunk_block_tables, int chunk_max_blocks, const int32_t *cu_q_lens,
    const int32_t *q_start_pos, const int32_t *chunk_seq_lens, int num_chunks,
    int total_q_tokens, int max_q_len, float *chunk_lse, void *out_decode, const void *q_decode,
    const void *key_decode, const void *value_decode, const int32_t *decode_block_tables,
    int decode_max_blocks, const int32_t *decode_seq_lens, int num_decode_seqs, float *decode_lse,
    int64_t key_token_stride, int64_t value_token_stride, void *k_cache, void *v_cache,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
    float scale, int chunk_sms, void *workspace, size_t workspace_bytes, void *stream);

/*
 * pa_decode_append -- one decode step with the slot scatter fused in:
 * sequence s's new token (row s of key / value, [num_seqs, *, Hkv, D] bf16
 * with token strides in elements) is written into the slot of position
 * seq_len[s] - 1 named by its block table, and sequence s's query attends
 * over [0, seq_len[s]) with that token in place.  The result is that of
 * pa_reshape_and_cache with slot_mapping[s] = block_tables[s][(seq_len[s] -
 * 1) / 16] * 16 + (seq_len[s] - 1) % 16, then pa_decode, in one launch
 * ("03 - Engines Papers", section 2 PagedAttention: the step's new K/V go
 * into their slots, then the kernel gathers K/V from the blocks; reading of
 * the pages: seq_len counts the new token).  A sequence with seq_len 0 has
 * no token to write.  bf16 pools only; every other argument, mode,
 * workspace and error as pa_decode.  The last block of every sequence must be
 * its own (copy-on-write done before, as for pa_reshape_and_cache).
 */
int pa_decode_append(void *out, const void *q, const void *key, const void *value,
                     int64_t key_token_stride, int64_t value_token_stride, void *k_cache,
                     void *v_cache, const int32_t *block_tables, int max_blocks_per_seq,
                     const int32_t *seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int64_t num_blocks, float scale,
                     int partition_tokens, float *out_lse, void *workspace,
                     size_t workspace_bytes, void *stream);

/*
 * Size of the static device scratch behind pa_decode_noalloc (8 MiB).
 */
#define PA_NOALLOC_SCRATCH_BYTES (8u << 20)

/*
 * pa_decode_noalloc -- the balanced decode of pa_decode (partition_tokens = 0)
 * for callers that cannot allocate device memory.  The paper has no
 * counterpart: this is a deployment variant of the same computation.
 *
 * Who needs it: a serving loop that must not call cudaMalloc on its hot path
 * (an allocation can synchronize the device and stall every other stream),
 * an engine whose device memory is reserved up front for the KV pool under a
 * fixed budget, and plain-C callers with no framework allocator to carve a
 * workspace from.  This entry point allocates nothing and calls no
 * allocating routine; the caller still passes every input and output,
 * exactly as for pa_decode (same arguments, layouts and results).
 *
 * Its scratch (the merge tickets and partial results of the balanced split)
 * is one file-scope device array of PA_NOALLOC_SCRATCH_BYTES inside libpa.so;
 * every GPU that loads the library holds it until the process exits.  The
 * first call on a device looks up that array's device address (once per
 * device, with that device current); make that first call before any stream
 * capture.  Every call shares the one array and clears its tickets at the
 * start, so calls that overlap on the GPU (two streams, or two threads) race
 * and give wrong results: serialize them.  A shape whose scratch need
 * exceeds the array (more than 32 q heads at head_dim 128 on a 152-SM GB300)
 * is rejected with PA_ERR_SCRATCH_LIMIT before anything is launched.
 */
int pa_decode_noalloc(void *out, const void *q, const void *k_cache, const void *v_cache,
                      const int32_t *block_tables, int max_blocks_per_seq,
                      const int32_t *seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                      int head_dim, int block_size, int64_t num_blocks, float scale,
                      float *out_lse, void *stream);

/*
 * Host-side metadata check (host pointers; any of block_tables / slot_mapping
 * / refcount may be NULL to skip that part).  Returns PA_OK or PA_ERR_INVALID:
 * table entries of every used block in [0, num_blocks); 0 <= seq_len <=
 * max_blocks_per_seq * block_size; slots in range and pairwise distinct; with
 * a refcount array, no slot targets a block whose refcount is above one (the
 * copy-on-write rule).
 */
int pa_validate_metadata(const int32_t *block_tables, int max_blocks_per_seq,
                         const int32_t *seq_lens, int num_seqs, const int64_t *slot_mapping,
                         int num_slots, const int32_t *refcount, int64_t num_blocks,
                         int block_size);

/*
 * Read (and with reset != 0, clear) the device error word of the current
 * device into *flags (PA_DEVERR_* bits).  Synchronizes with the device.
 */
int pa_device_error_flags(unsigned int *flags, int reset);

/*
 * Test entry points of the failure path (no product call needs them).  Each
 * makes one launch of the kernel its name gives, with the same arguments as
 * pa_decode (workspace and mode included; no lse) / pa_prefill_chunk (no
 * lse), in which the producer / loader warps issue no load at all and every
 * mbarrier wait is bounded by wait_limit_us (1 .. 2,000,000 us) instead of
 * the default two seconds.  Every wait therefore runs out with no copy in
 * flight: the kernel sets PA_DEVERR_TIMEOUT, skips the rest of its waits,
 * frees its tensor memory and returns; the outputs are unspecified.  The
 * call itself returns PA_OK once launched (PA_ERR_INVALID for a limit out of
 * range, or any status the plain call would return).  A decode's balanced-
 * split tickets are left at zero, so the same workspace serves the next
 * call.  The pages have no counterpart: these exist to exercise the kernels'
 * bounded waits on a GPU without faulting or hanging it.
 */
int pa_test_decode_stalled(void *out, const void *q, const void *k_cache, const void *v_cache,
                           const int32_t *block_tables, int max_blocks_per_seq,
                           const int32_t *seq_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           float scale, int partition_tokens, void *workspace,
                           size_t workspace_bytes, unsigned int wait_limit_us, void *stream);
int pa_test_prefill_stalled(void *out, const void *q, const void *k_cache, const void *v_cache,
                            const int32_t *block_tables, int max_blocks_per_seq,
                            const int32_t *cu_q_lens, const int32_t *q_start_pos,
                            const int32_t *seq_lens, int num_chunks, int total_q_tokens,
                            int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, float scale,
                            unsigned int wait_limit_us, void *stream);

#ifdef __cplusplus
}
#endif

#endif /* PA_H_ */
