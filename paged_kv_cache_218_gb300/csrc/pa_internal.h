// pa_internal.h -- launch parameters shared between the C-ABI front end
// (pa_api.cu) and the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

namespace pa {

constexpr int kBlockSize = 16;
constexpr int kMaxGroup = 8;            // q heads per kv head handled by one MMA column tile
constexpr int kMaxSeqsBalanced = 16000; // per-CTA prefix of block counts lives in shared memory
constexpr int kMaxCluster = 2;          // prefill: most query tiles per cluster (a CTA pair)

enum DecodeMode : int {
  kModeSinglePass = 0,  // one work item per (sequence, kv head)
  kModeFixedSplit = 1,  // fixed partitions of part_blocks blocks, partials + merge kernel
  kModeBalanced = 2,    // equal contiguous block ranges per CTA, merged in-kernel
};

struct DecodeArgs {
  __nv_bfloat16* out;           // [S, Hq, D]
  const __nv_bfloat16* q;       // [S, Hq, D]
  const int32_t* block_tables;  // [S, max_blocks]
  const int32_t* seq_lens;      // [S]
  float* out_lse;               // [S, Hq] or null
  float* part_o;                // fixed: [S, Hq, P_max, D]; balanced: slots
  float* part_lse;              // fixed: [S, Hq, P_max]
  int* counters;                // balanced: [grid] merge tickets (self-resetting)
  unsigned int* err;            // device error word
  int64_t num_blocks;
  int max_blocks;
  int num_seqs;
  int num_q_heads;
  int num_kv_heads;
  int group;
  float scale_log2;  // scale * log2(e)
  int mode;
  int part_blocks;   // fixed split / single pass: blocks per partition
  int max_parts;     // fixed split: P_max
  int slot_floats;   // balanced: floats per partial slot
  int warps_per_head;  // set by the launcher
  int stages;          // set by the launcher
  int piece_cost;      // balanced: a sequence's fixed cost in blocks (set by the launcher)
  int kv_fp8;          // pools hold E4M3 bytes (head_dim 128) with per-kv-head scales
  const float* k_scales;  // E4M3: [Hkv] dequantization scales of K and V
  const float* v_scales;
  // cascade suffix pass (all null otherwise): sequence s attends over its own
  // blocks [start_blocks[s], ceil(len/16)) only, starting from the prefix
  // pass's normalized o [S, Hq, D] and lse [S, Hq] (natural log)
  const int32_t* start_blocks;
  const float* init_o;
  const float* init_lse;
  uint64_t wait_ns;  // limit of every mbarrier wait (normally kWaitLimitNs)
  int stall_loads;   // test launch: the producer issues no load, every wait runs out
  // append (pa_decode_append; null otherwise): sequence s's new token, row s
  // of new_k / new_v (strides in elements), is written into the slot of
  // position seq_len-1 of the pools and attended there
  const __nv_bfloat16* new_k;
  const __nv_bfloat16* new_v;
  long long new_k_stride;
  long long new_v_stride;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
};

struct MergeArgs {
  __nv_bfloat16* out;
  float* out_lse;
  const float* part_o;
  const float* part_lse;
  const int32_t* num_parts;  // explicit counts, or null to derive from seq_lens
  const int32_t* seq_lens;   // with part_blocks: parts = max(1, ceil(ceil(len/16)/part_blocks))
  int part_blocks;
  int max_blocks;
  int skip_single;           // parts == 1 were written final by the decode kernel
  const int32_t* start_blocks;  // cascade suffix pass: parts cover blocks [start, ceil(len/16))
  int num_seqs;
  int num_q_heads;
  int head_dim;
  int max_parts;
};

struct PrefillArgs {
  __nv_bfloat16* out;
  const int32_t* block_tables;
  const int32_t* cu_q_lens;
  const int32_t* q_start_pos;
  const int32_t* seq_lens;
  float* out_lse;
  unsigned int* err;
  int64_t num_blocks;
  int max_blocks;
  int num_chunks;
  int total_q;               // rows of q and out; cu_q_lens must stay within
  int num_q_heads;
  int num_kv_heads;
  int group;
  int tiles_per_chunk;  // M tiles of 128 rows per (chunk, kv head)
  float scale_log2;
  uint64_t wait_ns;          // limit of every mbarrier wait (normally kWaitLimitNs)
  int stall_loads;           // test launch: the loaders issue no load, every wait runs out
  // append (pa_hybrid_attention_append; null / 0 otherwise): row i of new_k /
  // new_v (token strides in elements) is the K / V of the chunk's query row i;
  // the chunk's keys at positions >= q_start_pos are read from there, and its
  // rows are written into their pool slots by the CTA of their query tile
  const __nv_bfloat16* new_k;
  const __nv_bfloat16* new_v;
  long long new_k_stride;
  long long new_v_stride;
  __nv_bfloat16* k_pool;
  __nv_bfloat16* v_pool;
};

struct CascadeArgs {
  const __nv_bfloat16* q;        // [S, Hq, 128]
  const int32_t* seq_lens;       // [S]
  const int32_t* group_offsets;  // [num_groups + 1]
  const int32_t* prefix_tables;  // [num_groups, max_prefix_blocks]
  const int32_t* shared_blocks;  // [S]
  float* pre_o;                  // [S, Hq, 128] normalized prefix attention
  float* pre_lse;                // [S, Hq] natural log, -inf without a prefix
  unsigned int* err;
  int64_t num_blocks;
  int num_seqs;
  int max_prefix_blocks;
  int num_groups;
  int max_group;
  int num_q_heads;
  int num_kv_heads;
  int group;
  int kv_per_cta;   // kv heads per CTA
  int warps_per_kv; // consumer warps per kv head (16 query rows each)
  int stages;       // K/V ring depth
  int parts;        // CTAs that split one (group, kv-head subset)'s prefix blocks
  float* part_o;    // parts > 1: partials of parts 1.. [parts - 1][S, Hq, 128]
  float* part_lse;  // parts > 1: [parts - 1][S, Hq]
  int* tickets;     // parts > 1: [num_groups * subsets] (self-resetting)
  float scale_log2;
};

constexpr int kMaxPrefixParts = 4;  // cascade: most CTAs per (group, kv-head subset)

// Balanced-mode workspace layout (shared by the size query and the launch):
// per-CTA merge tickets, then two partial slots per CTA of Hq*(D+1) floats.
size_t balanced_slot_floats(int num_q_heads, int head_dim);
size_t balanced_workspace_bytes(int grid, int num_q_heads, int head_dim);

// Kernel launchers (return cudaError_t of the launch).
cudaError_t launch_decode(DecodeArgs a, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                          int head_dim, int grid, cudaStream_t stream);
int decode_grid(int num_sms, int mode, int group, bool kv_fp8);  // CTAs of a decode launch
bool decode_supported(int head_dim, int num_kv_heads, int num_q_heads, int mode, int num_seqs,
                      bool kv_fp8, bool append = false);
cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream);
cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                           const CUtensorMap* tm_v, int grid_tiles, cudaStream_t stream);
size_t prefill_smem_bytes();
bool cascade_shape(int num_kv_heads, int group, int max_group, int* kv_per_cta, int* warps_per_kv,
                   int* stages);
cudaError_t launch_cascade_prefix(const CascadeArgs& a, const CUtensorMap* tm_k,
                                  const CUtensorMap* tm_v, cudaStream_t stream);
// One launch for a hybrid batch: the balanced decode (bf16, head_dim 128) on
// its first decode_ctas CTAs and the prefill's CTA pairs on the rest.
// append: the decode role writes its sequences' new tokens (d.new_k) and the
// prefill role its chunks' (p.new_k), reading the chunks' new keys through
// nk / nv (maps of p.new_k / p.new_v); otherwise nk / nv are unused.
cudaError_t launch_hybrid(DecodeArgs d, const CUtensorMap* dk, const CUtensorMap* dv,
                          const PrefillArgs& p, const CUtensorMap* pq, const CUtensorMap* pk,
                          const CUtensorMap* pv, const CUtensorMap* nk, const CUtensorMap* nv,
                          int decode_ctas, int prefill_ctas, cudaStream_t stream);
// Shared-memory layout and warp split of a decode launch (pa_decode.cu).
size_t decode_smem_bytes(DecodeArgs& a, int head_dim);

}  // namespace pa
