// pa_prefill_body.cuh -- causal paged prefill chunks on tcgen05 tensor cores
// (sm_103a): one CTA's work (prefill_cta) and its shared-memory plan, included
// by the prefill launcher (pa_prefill.cu) and by the fused hybrid launch
// (pa_hybrid.cu).
//
// A Sarathi hybrid batch carries prefill chunks next to decodes ("03 -
// Engines Papers", section 3 Sarathi / Sarathi-Serve); a chunk's query at
// absolute position p attends over keys 0..p of its own paged KV, the K/V of
// later chunks not being there yet.  This is the one dense contraction of the
// path, so it runs on the 5th-generation tensor cores, FlashAttention-style
// (tiles through on-chip memory with an online softmax: FlashAttention and
// Milakov & Gimelshein, "References" page):
//
//  * One CTA per (128-row query tile, chunk, kv head).  GQA packs the group's
//    q heads into the rows: row r = token (r / G), head (r % G), so each K/V
//    tile serves all G heads (128 / G tokens per tile).
//  * CTA pairs (pa_prefill_chunk).  Two consecutive query tiles of the same
//    kv head run on the two SMs of a tcgen05 pair (a cluster of two): the
//    even CTA issues M = 256 products (cta_group::2) whose rows and score /
//    output accumulators stay in each CTA's own tensor memory, while each
//    CTA takes in only half of every K/V tile -- keys 64r .. 64r+63 of a K
//    tile and head-dim columns 64r .. 64r+63 of a V tile for CTA r -- and
//    the tensor cores of the pair exchange the halves.  Every SM thus
//    receives half the K/V bytes per product that a lone CTA does: a K/V
//    tile's intake, not the tensor pipe, set the pace of a lone CTA.  Each
//    CTA loads its own halves with plain TMA tensor loads (no load is shared
//    between SMs); the odd CTA's loads complete on the even CTA's barriers,
//    except the V tile holding a sequence's partly filled last block, which
//    lands on the odd CTA's own barrier, has its rows past seq_len zeroed and
//    is then reported to the even CTA.
//  * In a hybrid batch (pa_hybrid_attention) the same pairs run in the launch
//    of the decodes, on the SMs the decode's CTAs leave free.
//  * Warp roles.  Warp 9 loads Q once, then the K tiles; warp 10 the V
//    tiles (128 keys each, assembled from 16-token paged blocks by TMA
//    boxes, 128-byte swizzle) in rings of three, and
//    reports each landed V tile to the MMA issuer after zeroing the slots of
//    a sequence's last block that lie past its length.  A K slot is free
//    once the scores of its tile are done, a V slot once its PV product is.
//    Each loader reads its block ids 32 tiles at a time into shared memory.
//    A K box is a whole block of one head (both 64-column halves, 4 KB: a
//    4-D view of the pool that splits the block's 16 tokens into two groups
//    of 8 around the half), a V box the CTA's 64-column half of a block (2
//    KB, a 2-D view): 4 + 8 boxes per tile and CTA of a pair.
//    Warp 8 issues the score products from one thread (of the even CTA of a
//    pair): S = Q K^T into one of three tensor-memory score buffers
//    (tcgen05.mma, N = 128, K = 16, bf16 in, fp32 accumulate); warp 11 the
//    products O += P V into a fourth region.  Warps 0-7 run the softmax:
//    two warps per tensor-memory lane quadrant, each owning 64 of a row's
//    128 score columns.
//  * Three score buffers.  Scores of a tile can be computed as soon as its K
//    tile lands (while the softmax still works on the two before it), so a K
//    tile leaves its ring slot soon after it arrives.
//  * Pipelining.  Loaders and MMA issuers poll their barriers and issue
//    whatever is ready, so scores of the next tiles are computed while the
//    softmax works on tile j and PV of tile j-1 runs meanwhile.
//  * Softmax per row: tcgen05.ld of its scores, causal mask, row maximum
//    shared by the two half-row owners, p = 2^(x - m) rounded to bf16 and
//    stored back into tensor memory (tcgen05.st) over the first half of the
//    score columns it came from, where the PV product reads it as its A
//    operand; a score buffer takes new scores once that PV product is
//    complete.
//    The running maximum only moves (and O in tensor memory is only
//    rescaled) when the row maximum grows by more than 2^8, which keeps every
//    p below 256 and the fp32 accumulators far from overflow; the final
//    division uses the same reference maximum, so the result is exact up to
//    rounding.
//  * Epilogue: tcgen05.ld of O, divide by the row sum, bf16 store; lse.
// Every mbarrier wait is bounded; after a timeout the roles skip their
// remaining waits, still meet their barriers, and PA_DEVERR_TIMEOUT is set.
#pragma once

#include <math.h>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace pre {
namespace {


static_assert(kMaxCluster == 2, "tile counts are bounded with kMaxCluster");
constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = 8;     // issues the score products S = Q K^T
constexpr int kLoadKWarp = 9;   // Q and K tiles
constexpr int kLoadVWarp = 10;  // V tiles, and their reports to the MMA issuer
constexpr int kPvWarp = 11;     // issues the PV products O += P V
constexpr int kThreads = 12 * 32;
constexpr int kTileKeys = 128;
constexpr int kHalf = 128 * 128;  // a 64-column half of a 128-row operand: 128 rows x 128 B
constexpr int kBlockBytes = kBlockSize * 128;  // one paged block's 64-column half: 16 rows x 128 B
// K slot layout: block b of the slot at 4 KB * b, as [8-token group g][64-column
// half h][8 tokens][128 B]: key 8 * (2b + g) + r of half h at 2 KB * (2b + g) +
// 1 KB * h + 128 B * r, so a half's 8-key groups are 2 KB apart throughout
constexpr int kKGroupStride = 2048;
constexpr int kKHalfOffset = 1024;
constexpr int kIdBatch = 32;      // tiles whose block ids the loader reads at once
constexpr int kIdRing = 2 * kIdBatch;  // tiles whose block ids are kept in shared memory
constexpr int kMaxRing = 4;       // barrier slots per K / V ring

// Shared-memory plan of one CTA.  kPair 1: whole K / V tiles (128 keys x 128
// columns); kPair 2: this CTA's half of each (64 keys x 128 columns of K,
// 128 keys x 64 columns of V).
template <int kPair>
struct Plan {
  // four K and four V tiles in flight for pairs (about 1 % faster than
  // three, whose slots the score-full / PV-done barriers free)
  static constexpr int kNK = kPair == 2 ? 4 : 2;  // K tiles in flight
  static constexpr int kNV = kPair == 2 ? 4 : 2;  // V tiles in flight
  static constexpr int kKSlot = 2 * kHalf / kPair;
  static constexpr int kVSlot = 2 * kHalf / kPair;
  static constexpr int kQOff = 0;
  static constexpr int kKOff = kQOff + 2 * kHalf;
  static constexpr int kVOff = kKOff + kNK * kKSlot;
  static constexpr int kIdsOff = kVOff + kNV * kVSlot;  // block ids: one ring per loader warp
  static constexpr int kRedOff = kIdsOff + 2 * kIdRing * 8 * 4;  // row max exchange
  static constexpr int kRedOff2 = kRedOff + 2 * 2 * 128 * 4; // row-sum exchange
  static constexpr int kBarOff = kRedOff2 + 2 * 128 * 4;
  static constexpr int kSmemBytes = kBarOff + 320;
  static_assert(kNK <= kMaxRing && kNV <= kMaxRing, "barrier slots");
};

constexpr int kNS = 3;  // score buffers

// With as many K (V) slots as score buffers, K slot j % 3 is free once S(j)
// is done and V slot j % 3 once PV(j) is: the loaders then wait on the
// score-full / PV-done barriers themselves and the issuer makes two commits
// per tile fewer (the issuing thread's time per tile set the pace).  Tile
// j + 3 cannot complete its S (PV) before its own K (V) is loaded, so a
// loader never sees those barriers run two phases ahead.
template <int kPair>
constexpr bool kFreeByS = Plan<kPair>::kNK == kNS;
template <int kPair>
constexpr bool kFreeByPV = Plan<kPair>::kNV == kNS;

// S0 [0,128), S1 [128,256), S2 [256,384), O [384,512); P of a tile (bf16
// pairs) over its scores: keys 64h .. 64h+63 at columns 64h .. 64h+31
constexpr uint32_t kTmemCols = 512;
constexpr uint32_t kTmemO = 384;
constexpr float kRescaleThreshold = 8.0f;  // log2 units
constexpr float kLn2 = 0.6931471805599453f;

// tcgen05 shared-memory matrix descriptor, 128-byte swizzle.
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((addr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;  // descriptor version of the sm_100 family
  d |= static_cast<uint64_t>(2) << 61;  // SWIZZLE_128B
  return d;
}

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, N = 128 and M =
// 128 per CTA (256 for a pair); A K-major; B K-major (b_mn = 0) or MN-major
// (b_mn = 1).
__host__ __device__ constexpr uint32_t instr_desc(uint32_t b_mn, uint32_t m) {
  return (1u << 4)              // D format: f32
         | (1u << 7)            // A format: bf16
         | (1u << 10)           // B format: bf16
         | (b_mn << 16)         // B major-ness
         | ((128u >> 3) << 17)  // N / 8
         | ((m >> 4) << 24);    // M / 16
}

// 64 consecutive fp32 columns of this thread's tensor-memory lane (32x32b
// shape) together with their maximum, which the load itself reduces
// (tcgen05.ld.red, sm_103a), waited.
__device__ __forceinline__ void tmem_ld64_max(uint32_t taddr, uint32_t (&r)[64], float& mx) {
  asm volatile(
      "tcgen05.ld.red.sync.aligned.32x32b.x64.max.f32 {%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31, %32, %33, %34, %35, %36, %37, %38, %39, %40, %41, %42, %43, %44, %45, %46, %47, %48, %49, %50, %51, %52, %53, %54, %55, %56, %57, %58, %59, %60, %61, %62, %63}, %64, [%65];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]),
        "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]),
        "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]),
        "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]),
        "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63]),
        "=f"(mx)
      : "r"(taddr)
      : "memory");
}

// One arrival on an mbarrier of the other CTA of the pair that also expects
// `bytes` more transaction bytes (the bytes of this CTA's loads that complete
// on that barrier).
__device__ __forceinline__ void mbar_arrive_expect_tx_remote(uint32_t cluster_addr,
                                                             uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cluster.b64 _, [%0], %1;" ::"r"(cluster_addr),
               "r"(bytes)
               : "memory");
}

// Barrier waits.  A pair's barriers also receive the other CTA's arrivals,
// TMA completions and the even CTA's MMA commits; the data they report is
// tensor-core or TMA work, ordered by the barrier itself and the tcgen05
// fences, so the polls keep the cheap CTA-scope form (a cluster-scope
// acquire on every poll measured several hundred ns per loader step).
template <int kPair>
__device__ __forceinline__ bool bar_wait(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  return mbar_wait(bar, parity, limit_ns);
}

template <int kPair>
__device__ __forceinline__ bool bar_test(uint32_t bar, uint32_t parity) {
  return mbar_test_wait(bar, parity);
}

// Bounded wait that gives up at once after an earlier timeout anywhere in
// the CTA (so every role still reaches its barriers).
template <int kPair>
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort,
                                              const PrefillArgs& a) {
  if (*abort) return false;
  if (bar_wait<kPair>(bar, parity, a.wait_ns)) return true;
  *abort = 1;
  atomicOr(a.err, PA_DEVERR_TIMEOUT);
  return false;
}

// wait_or_abort for a whole warp that goes on to warp-synchronous tensor-
// memory loads and stores: the lanes reconverge and agree on the result.
template <int kPair>
__device__ __forceinline__ bool wait_or_abort_warp(uint32_t bar, uint32_t parity,
                                                   volatile int* abort, const PrefillArgs& a) {
  bool ok = !warp_flag(abort);
  if (ok) {
    ok = bar_wait<kPair>(bar, parity, a.wait_ns);
    __syncwarp();
    ok = __all_sync(0xffffffffu, ok);
  }
  if (!ok && !*abort) {
    *abort = 1;
    if ((threadIdx.x & 31) == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
  }
  return ok;
}

// One CTA of the prefill: tile CTA `cta` (a prefill launch's block index,
// or the prefill role's share of a fused hybrid launch, which starts on an
// even block so that a cluster's CTAs are a pair).  kPair 2: the two CTAs of
// a cluster run consecutive query tiles as one tcgen05 pair; kPair 1: one CTA
// per tile, no cluster.  Uses kThreads threads and the dynamic shared memory.
// tm_nk / tm_nv map the chunk's new K / V rows (a.new_k / a.new_v) when
// a.new_k is set (append), and are not read otherwise.
template <int kPair>
__device__ __forceinline__ void prefill_cta(const CUtensorMap& tm_q, const CUtensorMap& tm_k,
                                            const CUtensorMap& tm_v, const CUtensorMap& tm_nk,
                                            const CUtensorMap& tm_nv, const PrefillArgs& a,
                                            const int cta) {
  using P = Plan<kPair>;
  constexpr int kNK = P::kNK, kNV = P::kNV;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_q = sbase + P::kBarOff;
  const uint32_t bar_k_full = bar_q + 8;                  // [kMaxRing]
  const uint32_t bar_k_empty = bar_k_full + 8 * kMaxRing;  // [kMaxRing]
  const uint32_t bar_v_full = bar_k_empty + 8 * kMaxRing;  // [kMaxRing]: this CTA's V landed
  const uint32_t bar_v_ready = bar_v_full + 8 * kMaxRing;  // [kMaxRing]: V of the pair ready
  const uint32_t bar_v_empty = bar_v_ready + 8 * kMaxRing; // [kMaxRing]
  const uint32_t bar_s_full = bar_v_empty + 8 * kMaxRing;  // [3]: scores of tile j in buffer j % 3
  const uint32_t bar_p_full = bar_s_full + 8 * kNS;        // [3]: softmax of tile j done
  const uint32_t bar_o_done = bar_p_full + 8 * kNS;        // [3]: PV of tile j done
  static_assert(8 + 5 * 8 * kMaxRing + 3 * 8 * kNS <= 256, "barrier area");
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + P::kBarOff + 256);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + P::kBarOff + 260);
  // [kIdRing tiles][8 blocks], the K loader's ring, then the V loader's
  int* ids_smem = reinterpret_cast<int*>(smem + P::kIdsOff) +
                  ((threadIdx.x >> 5) == kLoadVWarp ? kIdRing * 8 : 0);
  float* red_max = reinterpret_cast<float*>(smem + P::kRedOff);   // [2 parity][2 half][128]
  float* red_sum = reinterpret_cast<float*>(smem + P::kRedOff2);  // [2 half][128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = a.num_kv_heads, G = a.group;
  const int tpt = kTileKeys / G;  // query tokens per tile
  const int rank = cta % kPair;  // rank in the pair
  const int rest = cta / kPair;
  const int kvh = rest % Hkv;
  const int t3 = rest / Hkv;
  const int c = t3 % a.num_chunks;
  const int mg = t3 / a.num_chunks;  // pair index along the chunk
  const int m = mg * kPair + rank;
  const bool issuer = rank == 0;     // issues the (pair's) tensor-core work

  // Barriers and tensor memory are set up before the grid-dependency wait,
  // while the previous kernel on the stream may still run: none of it
  // touches global memory.
  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int k = 0; k < kNK; ++k) {
      mbar_init(bar_k_full + 8 * k, 1);
      mbar_init(bar_k_empty + 8 * k, 1);
    }
    for (int k = 0; k < kNV; ++k) {
      mbar_init(bar_v_full + 8 * k, 1);
      mbar_init(bar_v_ready + 8 * k, kPair);  // one report per CTA of the pair
      mbar_init(bar_v_empty + 8 * k, 1);
    }
    for (int k = 0; k < kNS; ++k) {
      mbar_init(bar_s_full + 8 * k, 1);
      mbar_init(bar_p_full + 8 * k, kSoftmaxWarps * kPair);
      mbar_init(bar_o_done + 8 * k, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc<kPair>(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish<kPair>();
  }
  tc_fence_before();
  if constexpr (kPair == 2)
    cluster_sync();  // both CTAs' barriers exist before either reports to the other
  else
    __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  // launched as a programmatic dependent of the previous kernel (the scatter
  // of this step's K/V): nothing before this line touches global memory
  griddep_wait();
  // the next kernel on the stream may start launching; it waits for this grid
  griddep_launch_dependents();

  // Each loader warp reads block ids kIdBatch tiles at a time (eight loads
  // in flight per lane) into its own shared-memory ring: read one tile at a
  // time, ahead of its loads, the table's latency set the pace of the whole
  // pipeline.  read_ids issues the loads of a batch (entries the table row
  // holds), put_ids stores them: blocks past the visible keys get id -1,
  // which TMA reads as zeros, and ids outside the pool are flagged and read
  // as -1 too.
  const long long id_row = static_cast<long long>(c) * a.max_blocks;
  auto read_ids = [&](int t_first, int lim, int (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int jb = t_first * 8 + lane + 32 * i;
      v[i] = jb < lim ? a.block_tables[id_row + jb] : -1;
    }
  };
  auto put_ids = [&](int t_first, int nb_vis, const int (&v)[8]) {
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const int jb = t_first * 8 + lane + 32 * i;
      int id = jb < nb_vis ? v[i] : -1;
      if (jb < nb_vis && (id < 0 || id >= a.num_blocks)) {
        atomicOr(a.err, PA_DEVERR_BLOCK_ID);
        id = -1;
      }
      ids_smem[jb % (kIdRing * 8)] = id;
    }
    __syncwarp();
  };
  // The loaders' first batch is requested together with the chunk's
  // metadata (the whole of the table row's first entries, which any chunk
  // may read), so the two round trips overlap.
  int ids0[8];
  if (warp == kLoadKWarp || warp == kLoadVWarp) read_ids(0, a.max_blocks, ids0);

  // ---- chunk metadata (uniform over the CTA, and over a pair)
  const int q0 = a.cu_q_lens[c], q1 = a.cu_q_lens[c + 1];
  const int p0 = a.q_start_pos[c], n = a.seq_lens[c];
  const int qlen = q1 - q0;
  if (q0 < 0 || q1 > a.total_q || qlen < 0 || p0 < 0 || p0 + qlen > n ||
      n > a.max_blocks * kBlockSize) {
    if (tid == 0 && m == 0 && kvh == 0) atomicOr(a.err, PA_DEVERR_CHUNK);
    if (warp == 0) tmem_dealloc<kPair>(tmem, kTmemCols);  // uniform over the pair
    return;
  }
  const int t0 = m * tpt;
  const int tc0 = mg * kPair * tpt;  // first query token of the pair
  if (tc0 >= qlen) {  // the whole pair is past the chunk
    if (warp == 0) tmem_dealloc<kPair>(tmem, kTmemCols);
    return;
  }
  // Append: the chunk's own keys (positions p0 .. p0+qlen-1) are read from
  // its new rows, not from the pool, which this launch is still filling with
  // them; that needs the chunk to start a block (chunks of a multiple of 16
  // tokens after full cached blocks do).  Blocks jb_new and later of the
  // sequence are new.
  const bool append = a.new_k != nullptr;
  if (append && (p0 & (kBlockSize - 1)) != 0) {
    if (tid == 0 && m == 0 && kvh == 0) atomicOr(a.err, PA_DEVERR_CHUNK);
    if (warp == 0) tmem_dealloc<kPair>(tmem, kTmemCols);
    return;
  }
  const int jb_new = append ? p0 / kBlockSize : 0x7fffffff;
  const int tv = qlen - t0 < tpt ? qlen - t0 : tpt;  // valid tokens here (<= 0: none)
  // keys [0, kmax) are visible to some row of the pair; both CTAs walk the
  // same tiles (their own rows mask what they may not see)
  const int kmax = p0 + min(qlen, tc0 + kPair * tpt);
  const int nkt = (kmax + kTileKeys - 1) / kTileKeys;
  const int nb_vis = (kmax + kBlockSize - 1) / kBlockSize;
  // the K/V tile holding the sequence's last block when that block is only
  // partly filled (its slots past seq_len are zeroed before PV), else -1
  const int tail_tile = ((n & (kBlockSize - 1)) != 0 && (n - 1) / kBlockSize < nb_vis)
                            ? (n - 1) / kBlockSize / 8
                            : -1;
  auto fetch_ids = [&](int t_first) {
    int v[8];
    read_ids(t_first, nb_vis, v);
    put_ids(t_first, nb_vis, v);
  };
  if (warp == kLoadKWarp || warp == kLoadVWarp) put_ids(0, nb_vis, ids0);


  if (warp == kLoadKWarp || warp == kLoadVWarp) {
    // ------------------------------------------------------------ loaders
    // Two warps, each blocked only by its own TMA issues: a TMA box of 16
    // rows of 128 bytes takes the unit about 50 ns, so one warp issuing K
    // and V in turn left the unit idle between them.
    // K/V tiles are re-read by every query tile of the chunk: keep them in L2
    const uint64_t pol = l2_policy_evict_last();
    int jf = kIdBatch;              // tiles whose ids are in this warp's ring: [0, jf)
    IdleClock clk(a.wait_ns);
    auto timed_out = [&](bool progressed) {
      if (progressed) {
        clk.progress();
        return false;
      }
      if (!clk.expired()) return false;
      if (lane == 0) {
        *abort_flag = 1;
        atomicOr(a.err, PA_DEVERR_TIMEOUT);
      }
      return true;
    };
    if (warp == kLoadKWarp) {
      // loads of this CTA completing on the issuer's barrier `bar`: Q (3-D
      // map) and K boxes of the 4-D pool map
      auto load_q = [&](uint32_t dst, int x, int y, int z, uint32_t bar) {
        if constexpr (kPair == 2) {
          if (!issuer) {
            tma_load_3d_pair(dst, &tm_q, x, y, z, mapa_shared(bar, 0), pol);
            return;
          }
        }
        tma_load_3d(dst, &tm_q, x, y, z, bar, pol);
      };
      auto load_k = [&](uint32_t dst, int chunk, int group8, uint32_t bar) {
        if constexpr (kPair == 2) {
          if (!issuer) {
            tma_load_4d_pair(dst, &tm_k, 0, 0, chunk, group8, mapa_shared(bar, 0), pol);
            return;
          }
        }
        tma_load_4d(dst, &tm_k, 0, 0, chunk, group8, bar, pol);
      };
      // 8 new rows (from row r) of head kvh's two 64-column halves: one
      // token group of a K block, [half][8 tokens][64 columns]
      auto load_nk = [&](uint32_t dst, int r, uint32_t bar) {
        if constexpr (kPair == 2) {
          if (!issuer) {
            tma_load_3d_pair(dst, &tm_nk, 0, r, 2 * kvh, mapa_shared(bar, 0), pol);
            return;
          }
        }
        tma_load_3d(dst, &tm_nk, 0, r, 2 * kvh, bar, pol);
      };
      // a stalled test launch issues no load: every wait runs out with no
      // copy in flight
      if (lane == 0 && !a.stall_loads) {
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_k);
        if (append) tma_prefetch_desc(&tm_nk);
        if (issuer) mbar_arrive_expect_tx(bar_q, kPair * 2 * kHalf);  // both Q tiles of a pair
        for (int h = 0; h < 2; ++h)
          load_q(sbase + P::kQOff + h * kHalf, h * 64, kvh * G, q0 + t0, bar_q);
      }
      // K tile j = paged blocks 8j .. 8j+7 (id -1 past the visible keys: a box
      // outside the pool, which reads zeros); CTA r of a pair takes keys
      // 64r .. 64r+63 (blocks 4r .. 4r+3); one box per lane: block `lane`,
      // both halves of head kvh (column chunks 2 kvh, 2 kvh + 1; token groups
      // 2 id, 2 id + 1).  The issuer's barrier counts the pair's whole tile.
      int jk = a.stall_loads ? nkt : 0;
      while (jk < nkt && !*abort_flag) {
        bool progressed = false;
        // the next batch of ids, half a batch ahead of the loads, into ring
        // slots whose tiles have all been loaded
        if (jf < nkt && jk + kIdBatch / 2 >= jf) {
          fetch_ids(jf);
          jf += kIdBatch;
          progressed = true;
        }
        const int slot = jk % kNK;
        bool free_slot = jk < kNK;
        if (!free_slot && lane == 0)
          free_slot = kFreeByS<kPair>
                          ? bar_test<kPair>(bar_s_full + 8 * slot, ((jk / kNK) - 1) & 1)
                          : bar_test<kPair>(bar_k_empty + 8 * slot, ((jk / kNK) - 1) & 1);
        if (jk < jf && __shfl_sync(0xffffffffu, free_slot ? 1 : 0, 0)) {
          const uint32_t bar = bar_k_full + 8 * slot;
          if (lane == 0 && issuer) mbar_arrive_expect_tx(bar, 2 * kHalf);
          __syncwarp();
          if (lane < 8 / kPair) {
            const int b = lane + (kPair == 2 ? 4 * rank : 0);  // block of the tile
            const int jb = jk * 8 + b;                         // block of the sequence
            const uint32_t dst = sbase + P::kKOff + slot * P::kKSlot + lane * 2 * kBlockBytes;
            if (jb >= jb_new && jb < nb_vis) {
              const int r = q0 + (jb - jb_new) * kBlockSize;
              load_nk(dst, r, bar);
              load_nk(dst + kBlockBytes, r + 8, bar);
            } else {
              load_k(dst, 2 * kvh, 2 * ids_smem[(jk % kIdRing) * 8 + b], bar);
            }
          }
          __syncwarp();
          ++jk;
          progressed = true;
        }
        if (timed_out(progressed)) break;
      }
      // the issuer's release of the last fill of each slot has reached this
      // CTA before it may exit
      if (lane == 0)
        for (int sl = 0; sl < kNK && sl < nkt; ++sl)
          wait_or_abort<kPair>((kFreeByS<kPair> ? bar_s_full : bar_k_empty) + 8 * sl,
                               ((nkt - 1 - sl) / kNK) & 1, abort_flag, a);
    } else {
      if (lane == 0) {
        tma_prefetch_desc(&tm_v);
        if (append) tma_prefetch_desc(&tm_nv);
      }
      // V tile j: this CTA's boxes complete on its own barrier; once landed
      // (and its slots past seq_len zeroed) the tile is reported to the issuer
      // V tile j: the boxes of both CTAs of a pair complete straight on the
      // issuer's ready barrier (each CTA one arrival that expects its own
      // bytes), as K's do -- except the tile holding the sequence's last block
      // when that block is only partly filled: it lands on this CTA's own
      // barrier first, its slots past seq_len are zeroed, and then it is
      // reported to the issuer
      int jv = a.stall_loads ? nkt : 0;  // next V tile to load
      int tail_slot = -1;                // the tail tile's slot while its report is pending
      while ((jv < nkt || tail_slot >= 0) && !*abort_flag) {
        bool progressed = false;
        if (jf < nkt && jv + kIdBatch / 2 >= jf) {
          fetch_ids(jf);
          jf += kIdBatch;
          progressed = true;
        }
        if (jv < nkt && jv < jf) {
          const int slot = jv % kNV;
          bool free_slot = jv < kNV;
          if (!free_slot && lane == 0)
            free_slot = kFreeByPV<kPair>
                            ? bar_test<kPair>(bar_o_done + 8 * slot, ((jv / kNV) - 1) & 1)
                            : bar_test<kPair>(bar_v_empty + 8 * slot, ((jv / kNV) - 1) & 1);
          if (__shfl_sync(0xffffffffu, free_slot ? 1 : 0, 0)) {
            const bool tail = tail_tile == jv;
            const bool remote = kPair == 2 && !issuer && !tail;
            const uint32_t bar = tail ? bar_v_full + 8 * slot
                                      : (remote ? mapa_shared(bar_v_ready + 8 * slot, 0)
                                                : bar_v_ready + 8 * slot);
            if (lane == 0) {
              if (remote)
                mbar_arrive_expect_tx_remote(bar, P::kVSlot);
              else
                mbar_arrive_expect_tx(bar, P::kVSlot);
            }
            __syncwarp();
            // CTA r of a pair takes columns 64r .. 64r+63 of every key; one
            // box per lane: (block lane & 7, half lane >> 3)
            if (lane < 16 / kPair) {
              const int b = lane & 7, hh = lane >> 3;
              const int jb = jv * 8 + b;
              const uint32_t dst = sbase + P::kVOff + slot * P::kVSlot + hh * kHalf + b * kBlockBytes;
              const bool fresh = jb >= jb_new && jb < nb_vis;
              const CUtensorMap* map = fresh ? &tm_nv : &tm_v;
              const int y = fresh ? q0 + (jb - jb_new) * kBlockSize
                                  : ids_smem[(jv % kIdRing) * 8 + b] * kBlockSize;
              if constexpr (kPair == 2) {
                if (remote) {
                  tma_load_2d_pair(dst, map, kvh * 128 + (hh + rank) * 64, y, bar, pol);
                } else {
                  tma_load_2d(dst, map, kvh * 128 + (hh + rank) * 64, y, bar, pol);
                }
              } else {
                tma_load_2d(dst, map, kvh * 128 + (hh + rank) * 64, y, bar, pol);
              }
            }
            __syncwarp();
            if (tail) tail_slot = slot;
            ++jv;
            progressed = true;
          }
        }
        if (tail_slot >= 0) {
          bool landed = false;
          if (lane == 0) landed = bar_test<kPair>(bar_v_full + 8 * tail_slot, 0);  // its one use
          if (__shfl_sync(0xffffffffu, landed ? 1 : 0, 0)) {
            // the sequence's last block ends inside this tile: its slots past
            // seq_len hold no token and must not reach the PV product
            const int jl = (n - 1) / kBlockSize;
            const uint32_t vt = sbase + P::kVOff + tail_slot * P::kVSlot;
            const int first = n - jl * kBlockSize;  // rows first..15 of block jl % 8
            const int per_row = 8 * (2 / kPair);    // 16-byte chunks of a key row here
            for (int e = lane; e < (kBlockSize - first) * per_row; e += 32) {
              const int row = first + e / per_row, hh = (e / 8) % (2 / kPair), ch = e & 7;
              st_shared_zero16(vt + hh * kHalf + ((jl & 7) * kBlockSize + row) * 128 + (ch << 4));
            }
            fence_proxy_async_smem();
            __syncwarp();
            if (lane == 0) {
              // the zeroed rows are generic stores the pair's MMA will read
              if (kPair == 2 && !issuer)
                mbar_arrive_remote_release(mapa_shared(bar_v_ready + 8 * tail_slot, 0));
              else
                mbar_arrive(bar_v_ready + 8 * tail_slot);
            }
            tail_slot = -1;
            progressed = true;
          }
        }
        if (timed_out(progressed)) break;
      }
      if (lane == 0)
        for (int sl = 0; sl < kNV && sl < nkt; ++sl)
          wait_or_abort<kPair>((kFreeByPV<kPair> ? bar_o_done : bar_v_empty) + 8 * sl,
                               ((nkt - 1 - sl) / kNV) & 1, abort_flag, a);
    }
    __syncwarp();
  } else if (warp == kMmaWarp || warp == kPvWarp) {
    // ------------------------------------------------------------ tensor-core issue
    // Two issuing threads of the even CTA, one per product: each blocks in
    // its own MMA issues and commits while the other's products keep the
    // tensor pipe fed (one thread issuing both left the pipe idle during its
    // commits and barrier polls, which set the pace of a tile).  A commit
    // tracks the products of the thread that makes it.
    if (lane == 0 && issuer) {
      // a completion reaches this CTA's barrier and, for a pair, the peer's
      auto commit = [&](uint32_t bar) {
        if constexpr (kPair == 2) tc_commit<kPair>(mapa_shared(bar, 1));  // the peer's first
        tc_commit<kPair>(bar);
      };
      IdleClock clk(a.wait_ns);
      auto give_up = [&]() {
        if (!*abort_flag) {
          *abort_flag = 1;
          atomicOr(a.err, PA_DEVERR_TIMEOUT);
        }
      };
      if (warp == kMmaWarp) {
        const uint32_t idesc_s = instr_desc(0, 128 * kPair);
        bool ok = wait_or_abort<kPair>(bar_q, 0, abort_flag, a);
        // Descriptors of the operands' first k-step: a k-step's descriptor
        // is the base's plus its byte offset / 16 (the start-address field,
        // whose sum stays below 2^14 in a 227 KB shared memory), so the
        // issue loop adds a constant per product instead of building each.
        const uint64_t dq = smem_desc(sbase + P::kQOff, 16, 1024);
        const uint64_t dk0 = smem_desc(sbase + P::kKOff, 16, kKGroupStride);
        // ring positions of js, kept as counters (no division per tile);
        // s_round = js / kNS
        int js = 0, s_buf = 0, s_round = 0, s_kslot = 0, s_kphase = 0;
        while (ok && js < nkt) {
          // S(js) = Q K_js^T into score buffer js % 3 once K_js landed and
          // PV of tile js-3, which reads its P from that buffer, completed
          if (bar_test<kPair>(bar_k_full + 8 * s_kslot, s_kphase) &&
              (js < kNS || bar_test<kPair>(bar_o_done + 8 * s_buf, (s_round + 1) & 1))) {
            // the K operand is a TMA load, ordered by its barrier; the
            // buffer's last reader is a product of the other thread
            if (js >= kNS) tc_fence_after();
            const uint64_t dk = dk0 + static_cast<uint64_t>((s_kslot * P::kKSlot) >> 4);
            const uint32_t dst = tmem + s_buf * 128;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              tc_mma_f16<kPair>(dst, dq + (((ks >> 2) * kHalf + (ks & 3) * 32) >> 4),
                                dk + (((ks >> 2) * kKHalfOffset + (ks & 3) * 32) >> 4), idesc_s,
                                ks > 0);
            commit(bar_s_full + 8 * s_buf);
            if constexpr (!kFreeByS<kPair>) commit(bar_k_empty + 8 * s_kslot);
            ++js;
            if (++s_buf == kNS) {
              s_buf = 0;
              ++s_round;
            }
            if (++s_kslot == kNK) {
              s_kslot = 0;
              s_kphase ^= 1;
            }
            clk.progress();
          } else if (*abort_flag || clk.expired()) {
            give_up();
            ok = false;
          }
        }
      } else {
        const uint32_t idesc_o = instr_desc(1, 128 * kPair);
        const uint64_t dv0 = smem_desc(sbase + P::kVOff, kHalf, 1024);
        int jp = 0, p_buf = 0, p_phase = 0, p_vslot = 0, p_vphase = 0;
        bool ok = true;
        while (ok && jp < nkt) {
          // O += P_jp V_jp once the softmax wrote P_jp (so S(jp) is done)
          // and V_jp is ready
          if (bar_test<kPair>(bar_p_full + 8 * p_buf, p_phase) &&
              bar_test<kPair>(bar_v_ready + 8 * p_vslot, p_vphase)) {
            if (kPair == 2 && jp == tail_tile) fence_acq_rel_cluster();  // the peer's zeroed rows
            tc_fence_after();
            const uint64_t dv = dv0 + static_cast<uint64_t>((p_vslot * P::kVSlot) >> 4);
            const uint32_t ta = tmem + p_buf * 128;
#pragma unroll
            for (int ks = 0; ks < 8; ++ks)
              tc_mma_f16_tmem_a<kPair>(tmem + kTmemO, ta + (ks >> 2) * 64 + (ks & 3) * 8,
                                       dv + ((ks * kBlockBytes) >> 4), idesc_o,
                                       (jp > 0 || ks > 0) ? 1u : 0u);
            commit(bar_o_done + 8 * p_buf);
            if constexpr (!kFreeByPV<kPair>) commit(bar_v_empty + 8 * p_vslot);
            ++jp;
            if (++p_buf == kNS) {
              p_buf = 0;
              p_phase ^= 1;
            }
            if (++p_vslot == kNV) {
              p_vslot = 0;
              p_vphase ^= 1;
            }
            clk.progress();
          } else if (*abort_flag || clk.expired()) {
            give_up();
            ok = false;
          }
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
    if (append && tv > 0) {
      // the slot scatter of this tile's tokens for head kvh, while the first
      // scores are still on their way: K and V rows of 256 bytes, 16 bytes
      // per thread and step (no CTA reads these slots in this launch)
      for (int e = tid; e < tv * 32; e += kSoftmaxWarps * 32) {
        const int i = e >> 5, which = (e >> 4) & 1, piece = e & 15;
        const int pos = p0 + t0 + i;
        const int id = a.block_tables[id_row + pos / kBlockSize];
        if (id < 0 || id >= a.num_blocks) {
          atomicOr(a.err, PA_DEVERR_BLOCK_ID);
          continue;
        }
        const long long slot = static_cast<long long>(id) * kBlockSize + (pos & (kBlockSize - 1));
        const long long row = q0 + t0 + i;
        const uint4* src = reinterpret_cast<const uint4*>(
            which ? a.new_v + row * a.new_v_stride : a.new_k + row * a.new_k_stride);
        uint4* dst = reinterpret_cast<uint4*>((which ? a.v_pool : a.k_pool) +
                                              (slot * Hkv + kvh) * 128);
        dst[piece] = __ldg(src + kvh * 16 + piece);
      }
    }
    const int qd = warp & 3, hc = warp >> 2;
    const int r = qd * 32 + lane;  // query row = tensor-memory lane
    const uint32_t lane_off = static_cast<uint32_t>(qd * 32) << 16;
    const int pos = p0 + t0 + r / G;
    const int lim = min(pos, kmax - 1);  // last visible key of the row
    float m_run = -INFINITY, l_run = 0.f;
    uint32_t v[64];
    for (int j = 0; j < nkt; ++j) {
      const int b = j & 1;        // row maximum exchange buffer
      const int b3 = j % kNS;     // score buffer
      wait_or_abort_warp<kPair>(bar_s_full + 8 * b3, (j / kNS) & 1, abort_flag, a);
      tc_fence_after();
      const int kb = j * kTileKeys + hc * 64;
      const int nvis = lim - kb + 1;  // visible columns of this half (may be <= 0 or > 64)
      // a warp whose rows all see the whole half takes the row maximum from
      // the tensor-memory load itself and skips the per-element masks; the
      // others reduce the visible columns with eight independent partial
      // maxima (short dependency chains)
      const bool full = __all_sync(0xffffffffu, nvis >= 64);
      float mloc;
      if (full) {
        tmem_ld64_max(tmem + lane_off + b3 * 128 + hc * 64, v, mloc);
      } else {
        tmem_ld64(tmem + lane_off + b3 * 128 + hc * 64, v);
        float mp[8];
#pragma unroll
        for (int k = 0; k < 8; ++k) mp[k] = -INFINITY;
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i < nvis) mp[i & 7] = fmaxf(mp[i & 7], __uint_as_float(v[i]));
        mloc = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                     fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
      }
      mloc = mloc * a.scale_log2;  // scale > 0 keeps the order
      red_max[(b * 2 + hc) * 128 + r] = mloc;
      named_barrier(1 + qd, 64);
      const float mx = fmaxf(mloc, red_max[(b * 2 + (hc ^ 1)) * 128 + r]);
      const float m_new = fmaxf(m_run, mx);
      const bool move = m_new > m_run + kRescaleThreshold;  // true on the first tile
      const float m_use = move ? m_new : m_run;
      const float alpha = move ? fast_exp2(m_run - m_use) : 1.f;
      float rsp[4] = {0.f, 0.f, 0.f, 0.f};
      uint32_t pk[32];
      const float sl = a.scale_log2;
      if (full) {
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          // p = 2^(scale*s - m): one FMA per score before the exp
          const float e0 = fast_exp2(fmaf(__uint_as_float(v[i]), sl, -m_use));
          const float e1 = fast_exp2(fmaf(__uint_as_float(v[i + 1]), sl, -m_use));
          rsp[(i >> 1) & 3] += e0 + e1;
          pk[i / 2] = pack_bf16x2(e0, e1);
        }
      } else {
#pragma unroll
        for (int i = 0; i < 64; i += 2) {
          const float e0 = i < nvis ? fast_exp2(fmaf(__uint_as_float(v[i]), sl, -m_use)) : 0.f;
          const float e1 =
              i + 1 < nvis ? fast_exp2(fmaf(__uint_as_float(v[i + 1]), sl, -m_use)) : 0.f;
          rsp[(i >> 1) & 3] += e0 + e1;
          pk[i / 2] = pack_bf16x2(e0, e1);
        }
      }
      const float rs = (rsp[0] + rsp[1]) + (rsp[2] + rsp[3]);
      l_run = l_run * alpha + rs;
      m_run = m_use;

      // O is rescaled only when a row maximum moved; then PV of the previous
      // tile must have landed first
      if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
        wait_or_abort_warp<kPair>(bar_o_done + 8 * ((j - 1) % kNS), ((j - 1) / kNS) & 1,
                                  abort_flag, a);
        tc_fence_after();
        const uint32_t ocol = tmem + lane_off + kTmemO + hc * 64;
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          uint32_t (&w)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32 * cc]);
          tmem_ld32(ocol + 32 * cc, w);
#pragma unroll
          for (int i = 0; i < 32; ++i) w[i] = __float_as_uint(__uint_as_float(w[i]) * alpha);
          tmem_st32(ocol + 32 * cc, w);
        }
      }
      // keys hc*64 .. hc*64+63 of row r -> columns hc*64 .. hc*64+31 of score
      // buffer b3, which this warp alone has read (its partner's half is
      // disjoint); PV of tile j-3 finished with it before S(j) was computed
      tmem_st32(tmem + lane_off + b3 * 128 + hc * 64, pk);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) {
        if (kPair == 2 && !issuer)
          mbar_arrive_remote(mapa_shared(bar_p_full + 8 * b3, 0));
        else
          mbar_arrive(bar_p_full + 8 * b3);
      }
    }

    // ---- epilogue: O / l -> bf16, and lse
    wait_or_abort_warp<kPair>(bar_o_done + 8 * ((nkt - 1) % kNS), ((nkt - 1) / kNS) & 1,
                              abort_flag, a);
    tc_fence_after();
    red_sum[hc * 128 + r] = l_run;
    named_barrier(1 + qd, 64);
    const float l_tot = l_run + red_sum[(hc ^ 1) * 128 + r];
    const int tok = r / G, g = r % G;
    const bool store = tok < tv && !*abort_flag;
    const float inv = l_tot > 0.f ? 1.f / l_tot : 0.f;
    const long long row = static_cast<long long>(q0 + t0 + tok) * a.num_q_heads + kvh * G + g;
    const uint32_t ocol = tmem + lane_off + kTmemO + hc * 64;
#pragma unroll
    for (int cc = 0; cc < 2; ++cc) {
      uint32_t (&w)[32] = *reinterpret_cast<uint32_t(*)[32]>(&v[32 * cc]);
      tmem_ld32(ocol + 32 * cc, w);
      if (store) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          pk[i / 2] = pack_bf16x2(__uint_as_float(w[i]) * inv, __uint_as_float(w[i + 1]) * inv);
        uint4* dst = reinterpret_cast<uint4*>(a.out + row * 128 + hc * 64 + cc * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
    if (store && hc == 0 && a.out_lse)
      a.out_lse[row] = l_tot > 0.f ? (m_run + __log2f(l_tot)) * kLn2 : -INFINITY;
  }
  tc_fence_before();
  if constexpr (kPair == 2)
    cluster_sync();  // neither CTA leaves while the other may still report to it
  else
    __syncthreads();
  tc_fence_after();
  if (warp == 0) tmem_dealloc<kPair>(tmem, kTmemCols);
}

}  // namespace
}  // namespace pre
}  // namespace pa
