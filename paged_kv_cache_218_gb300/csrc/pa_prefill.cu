// pa_prefill.cu -- causal paged prefill chunks on tcgen05 tensor cores (sm_103a).
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
//    tile serves all G heads (128 / G tokens per tile).  Four consecutive
//    query tiles of the same kv head form a cluster and share every K/V tile:
//    each CTA loads a quarter of a tile's paged blocks with TMA multicast into
//    all four, so each SM issues a quarter of the loads (the per-SM TMA
//    request rate, not bandwidth, bounds this pipeline).
//  * Warp roles.  Warp 9 loads: Q once, then K and V tiles of 128 keys, each
//    assembled from eight 16-token paged blocks by TMA (128-byte swizzle), in
//    rings of two K and two V tiles (a K tile is free once its scores are
//    done, a V tile only once its PV product is).  Deeper rings only lengthen
//    the queue: per-tile traces show each SM taking in K/V at about 57 GB/s
//    whatever the depth, the arrival latency growing with the tiles in
//    flight.  Warp 8 issues the tensor-core work from one thread: S = Q K^T
//    into one of three tensor-memory score buffers (tcgen05.mma, M = N = 128,
//    K = 16, bf16 in, fp32 accumulate) and O += P V into a fourth region.
//    Warps 0-7 run the softmax: two warps per tensor-memory lane quadrant,
//    each owning 64 of a row's 128 score columns.
//  * Three score buffers.  Scores of a tile can be computed as soon as its K
//    tile lands (while the softmax still works on the two before it), so a K
//    tile leaves its ring slot soon after it arrives: with two rings of two,
//    how long a tile holds its slot sets the pace, not the tensor cores.
//  * Pipelining.  Loader and MMA issuer poll their barriers and issue
//    whatever is ready, so scores of the next tiles are computed while the
//    softmax works on tile j and PV of tile j-1 runs meanwhile.
//  * Softmax per row: tcgen05.ld of its scores, causal mask, row maximum
//    shared by the two half-row owners, p = 2^(x - m) rounded to bf16 and
//    stored back into tensor memory (tcgen05.st) over the first half of the
//    score columns it came from, where the PV product reads it as its A
//    operand; a score buffer takes new scores once that PV product is done.  The running maximum only
//    moves (and O in tensor memory is only rescaled) when the row maximum
//    grows by more than 2^8, which keeps every p below 256 and the fp32
//    accumulators far from overflow; the final division uses the same
//    reference maximum, so the result is exact up to rounding.
//  * Epilogue: tcgen05.ld of O, divide by the row sum, bf16 store; lse.
// Every mbarrier wait is bounded; after a timeout the roles skip their
// remaining waits, still meet their barriers, and PA_DEVERR_TIMEOUT is set.
#include <math.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kClusterAlone = 4;  // query tiles of one kv head sharing every K/V tile load
static_assert(kClusterAlone <= kMaxCluster, "tile counts are bounded with kMaxCluster");
constexpr int kSoftmaxWarps = 8;
constexpr int kMmaWarp = 8;
constexpr int kLoadWarp = 9;
constexpr int kThreads = 10 * 32;
constexpr int kTileKeys = 128;
constexpr int kHalf = 128 * 128;  // a 64-column half of a 128-row operand: 128 rows x 128 B
constexpr int kQOff = 0;
constexpr int kNK = 2;                  // K tiles in flight (freed as soon as their scores are done)
constexpr int kNV = 2;                  // V tiles in flight (held until their PV product is done)
constexpr int kTileBytes = 2 * kHalf;   // one K or V tile: 128 keys x 128 columns
constexpr int kKOff = kQOff + 2 * kHalf;
constexpr int kVOff = kKOff + kNK * kTileBytes;
constexpr int kIdsOff = kVOff + kNV * kTileBytes;      // block ids of the tiles in flight
constexpr int kRedOff = kIdsOff + 4 * 8 * 4;          // row max / sum exchange
constexpr int kRedOff2 = kRedOff + 2 * 2 * 128 * 4;  // row-sum exchange
constexpr int kBarOff = kRedOff2 + 2 * 128 * 4;
constexpr int kSmemBytes = kBarOff + 256;
static_assert(kNK <= 3 && kNV <= 3, "barrier slots");
// S0 [0,128), S1 [128,256), S2 [256,384), O [384,512); P of a tile (bf16
// pairs) over its scores: keys 64h .. 64h+63 at columns 64h .. 64h+31
constexpr int kNS = 3;  // score buffers
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

// Instruction descriptor, kind::f16: bf16 A and B, fp32 D, M = N = 128;
// A K-major; B K-major (b_mn = 0) or MN-major (b_mn = 1).
__host__ __device__ constexpr uint32_t instr_desc(uint32_t b_mn) {
  return (1u << 4)              // D format: f32
         | (1u << 7)            // A format: bf16
         | (1u << 10)           // B format: bf16
         | (b_mn << 16)         // B major-ness
         | ((128u >> 3) << 17)  // N / 8
         | ((128u >> 4) << 24); // M / 16
}

// Bounded wait that gives up at once after an earlier timeout anywhere in
// the CTA (so every role still reaches its barriers).
__device__ __forceinline__ bool wait_or_abort(uint32_t bar, uint32_t parity, volatile int* abort,
                                              unsigned int* err) {
  if (*abort) return false;
  if (mbar_wait(bar, parity)) return true;
  *abort = 1;
  atomicOr(err, PA_DEVERR_TIMEOUT);
  return false;
}

// wait_or_abort for a whole warp that goes on to warp-synchronous tensor-
// memory loads and stores: the lanes reconverge and agree on the result.
__device__ __forceinline__ bool wait_or_abort_warp(uint32_t bar, uint32_t parity,
                                                   volatile int* abort, unsigned int* err) {
  bool ok = !warp_flag(abort);
  if (ok) ok = mbar_wait_warp(bar, parity);
  if (!ok && !*abort) {
    *abort = 1;
    if ((threadIdx.x & 31) == 0) atomicOr(err, PA_DEVERR_TIMEOUT);
  }
  return ok;
}

// Co-scheduled next to a decode (PrefillArgs::after_decode) the chunk is a
// programmatic dependent of that decode, whose result it does not read: its
// CTAs start as soon as the decode's have started and take the SMs the decode
// leaves free.  Its K/V were scattered by the kernel before the decode, which
// has completed by then.  To keep the stream's order for the kernels after
// it, the last CTA of the chunk to finish waits for the decode before it
// exits (the others exit at once and free their SMs).
__device__ __forceinline__ void chunk_exit(const PrefillArgs& a, int tid) {
  if (!a.after_decode || tid != 0) return;
  if (atomicAdd(a.done_ctr, 1u) == gridDim.x - 1) {
    *a.done_ctr = 0;  // for the next call
    griddep_wait();
  }
}

// kCluster query tiles (4 alone, 1 when co-scheduled: a cluster needs that
// many free SMs of one GPC at once) share each K/V tile load by multicast.
template <int kCluster>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_q = sbase + kBarOff;
  const uint32_t bar_k_full = bar_q + 8;     // [3] (kNK used)
  const uint32_t bar_k_empty = bar_q + 32;   // [3]
  const uint32_t bar_v_full = bar_q + 56;    // [3] (kNV used)
  const uint32_t bar_v_empty = bar_q + 80;   // [3]
  const uint32_t bar_s_full = bar_q + 104;   // [3]: scores of tile j in buffer j % 3
  const uint32_t bar_p_full = bar_q + 128;   // [3]: softmax of tile j done
  const uint32_t bar_o_done = bar_q + 152;   // [3]: PV of tile j done
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 176);
  int* ids_smem = reinterpret_cast<int*>(smem + kIdsOff);      // [4 tiles][8 blocks]
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kBarOff + 180);
  float* red_max = reinterpret_cast<float*>(smem + kRedOff);   // [2 parity][2 half][128]
  float* red_sum = reinterpret_cast<float*>(smem + kRedOff2);  // [2 half][128]

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = a.num_kv_heads, G = a.group;
  const int tpt = kTileKeys / G;  // query tokens per tile
  const int rank = static_cast<int>(blockIdx.x % kCluster);  // rank in the cluster
  const int rest = static_cast<int>(blockIdx.x / kCluster);
  const int kvh = rest % Hkv;
  const int t3 = rest / Hkv;
  const int c = t3 % a.num_chunks;
  const int mg = t3 / a.num_chunks;  // cluster index along the chunk
  const int m = mg * kCluster + rank;
  constexpr uint16_t kMask = (1u << kCluster) - 1;

  // launched as a programmatic dependent of the previous kernel (the scatter
  // of this step's K/V): nothing before this line touches global memory --
  // unless co-scheduled behind a decode (see chunk_exit)
  if (!a.after_decode) griddep_wait();
  // the next kernel on the stream may start launching; it waits for this grid
  griddep_launch_dependents();

  // ---- chunk metadata (uniform over the CTA)
  const int q0 = a.cu_q_lens[c], q1 = a.cu_q_lens[c + 1];
  const int p0 = a.q_start_pos[c], n = a.seq_lens[c];
  const int qlen = q1 - q0;
  if (q0 < 0 || q1 > a.total_q || qlen < 0 || p0 < 0 || p0 + qlen > n ||
      n > a.max_blocks * kBlockSize) {
    if (tid == 0 && m == 0 && kvh == 0) atomicOr(a.err, PA_DEVERR_CHUNK);
    chunk_exit(a, tid);
    return;
  }
  const int t0 = m * tpt;
  const int tc0 = mg * kCluster * tpt;  // first query token of the cluster
  if (tc0 >= qlen) {  // the whole cluster is past the chunk
    chunk_exit(a, tid);
    return;
  }
  const int tv = qlen - t0 < tpt ? qlen - t0 : tpt;  // valid tokens here (<= 0: none)
  // keys [0, kmax) are visible to some row of the cluster; every member walks
  // the same tiles (its own rows mask what they may not see)
  const int kmax = p0 + min(qlen, tc0 + kCluster * tpt);
  const int nkt = (kmax + kTileKeys - 1) / kTileKeys;
  const int nb_vis = (kmax + kBlockSize - 1) / kBlockSize;
  // the loader reads the block ids of its first two K tiles now, so that the
  // table's latency overlaps the set-up below instead of delaying the first load
  int id_t0 = -1, id_t1 = -1;
  if (warp == kLoadWarp && lane < 8 / kCluster) {
    const long long row = static_cast<long long>(c) * a.max_blocks;
    const int jb = lane * kCluster + rank;
    if (jb < nb_vis) id_t0 = a.block_tables[row + jb];
    if (jb + 8 < nb_vis) id_t1 = a.block_tables[row + jb + 8];
  }

  if (tid == 0) {
    mbar_init(bar_q, 1);
    for (int k = 0; k < kNK; ++k) {
      mbar_init(bar_k_full + 8 * k, 1);
      mbar_init(bar_k_empty + 8 * k, kCluster);  // released by every member of the cluster
    }
    for (int k = 0; k < kNV; ++k) {
      mbar_init(bar_v_full + 8 * k, 1);
      mbar_init(bar_v_empty + 8 * k, kCluster);
    }
    for (int k = 0; k < kNS; ++k) {
      mbar_init(bar_s_full + 8 * k, 1);
      mbar_init(bar_p_full + 8 * k, kSoftmaxWarps);
      mbar_init(bar_o_done + 8 * k, 1);
    }
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  cluster_sync();  // every member's barriers exist before any multicast reaches them
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == kLoadWarp) {
    // ------------------------------------------------------------ loader
    // K/V tiles are re-read by every query tile of the chunk: keep them in L2
    const uint64_t pol = l2_policy_evict_last();
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar_q, 2 * kHalf);
      for (int h = 0; h < 2; ++h)
        tma_load_3d(sbase + kQOff + h * kHalf, &tm_q, h * 64, kvh * G, q0 + t0, bar_q, pol);
    }
    // tile j = paged blocks 8j .. 8j+7 (their ids are read once, with the K
    // tile, and kept for the V tile); blocks past the visible keys are read
    // from outside the pool, which fills zeros
    auto issue = [&](int j, bool is_k, uint32_t dst, uint32_t bar) {
      if (lane == 0) mbar_arrive_expect_tx(bar, kTileBytes);  // the whole tile lands here
      __syncwarp();
      if (lane < 8 / kCluster) {
        const int bl = lane * kCluster + rank;  // this CTA's share of the tile's blocks
        int id;
        if (is_k) {
          const int jb = j * 8 + bl;
          id = -1;
          if (jb < nb_vis) {
            id = j == 0   ? id_t0
                 : j == 1 ? id_t1
                          : a.block_tables[static_cast<long long>(c) * a.max_blocks + jb];
            if (id < 0 || id >= a.num_blocks) {
              atomicOr(a.err, PA_DEVERR_BLOCK_ID);
              id = -1;
            }
          }
          ids_smem[(j & 3) * 8 + bl] = id;
        } else {
          id = ids_smem[(j & 3) * 8 + bl];
        }
        const uint32_t d = dst + bl * kBlockSize * 128;
        const int z = id * kBlockSize;
#pragma unroll
        for (int h = 0; h < 2; ++h)
          tma_load_3d_multicast(d + h * kHalf, is_k ? &tm_k : &tm_v, h * 64, kvh, z, bar, kMask,
                                pol);
      }
      __syncwarp();
    };
    int jk = 0, jv = 0;
    uint64_t t_last = global_ns();  // time of the last issue
    while ((jk < nkt || jv < nkt) && !*abort_flag) {
      bool progressed = false;
      if (jk < nkt && jk < jv + 4) {  // the id ring holds four tiles
        const int slot = jk % kNK;
        bool free_slot = jk < kNK;
        if (!free_slot && lane == 0)
          free_slot = mbar_test_wait(bar_k_empty + 8 * slot, ((jk / kNK) - 1) & 1);
        if (__shfl_sync(0xffffffffu, free_slot ? 1 : 0, 0)) {
          issue(jk, true, sbase + kKOff + slot * kTileBytes, bar_k_full + 8 * slot);
          ++jk;
          progressed = true;
        }
      }
      if (jv < jk) {
        const int slot = jv % kNV;
        bool free_slot = jv < kNV;
        if (!free_slot && lane == 0)
          free_slot = mbar_test_wait(bar_v_empty + 8 * slot, ((jv / kNV) - 1) & 1);
        if (__shfl_sync(0xffffffffu, free_slot ? 1 : 0, 0)) {
          issue(jv, false, sbase + kVOff + slot * kTileBytes, bar_v_full + 8 * slot);
          ++jv;
          progressed = true;
        }
      }
      if (progressed) {
        t_last = global_ns();
      } else if (global_ns() - t_last > kWaitLimitNs) {
        if (lane == 0) {
          *abort_flag = 1;
          atomicOr(a.err, PA_DEVERR_TIMEOUT);
        }
        break;
      }
    }
    // every member's release of the last fill of each slot has reached this
    // CTA before it may leave the cluster
    if (lane == 0) {
      for (int sl = 0; sl < kNK && sl < nkt; ++sl)
        wait_or_abort(bar_k_empty + 8 * sl, ((nkt - 1 - sl) / kNK) & 1, abort_flag, a.err);
      for (int sl = 0; sl < kNV && sl < nkt; ++sl)
        wait_or_abort(bar_v_empty + 8 * sl, ((nkt - 1 - sl) / kNV) & 1, abort_flag, a.err);
    }
    __syncwarp();
  } else if (warp == kMmaWarp) {
    // ------------------------------------------------------------ tensor-core issue
    if (lane == 0) {
      const uint32_t idesc_s = instr_desc(0), idesc_o = instr_desc(1);
      bool ok = wait_or_abort(bar_q, 0, abort_flag, a.err);
      int js = 0, jp = 0;  // next score tile / next PV product to issue
      uint64_t t_last = global_ns();  // time of the last issue
      while (ok && jp < nkt) {
        bool progressed = false;
        // S(js) = Q K_js^T into score buffer js % 3, once K_js landed and PV
        // of tile js-3 has read its P from that buffer
        if (js < nkt && mbar_test_wait(bar_k_full + 8 * (js % kNK), (js / kNK) & 1) &&
            (js < kNS || mbar_test_wait(bar_o_done + 8 * (js % kNS), ((js / kNS) - 1) & 1))) {
          tc_fence_after();
          const uint32_t kt = sbase + kKOff + (js % kNK) * kTileBytes;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks) {
            const uint32_t koff = (ks >> 2) * kHalf + (ks & 3) * 32;
            tc_mma_f16(tmem + (js % kNS) * 128, smem_desc(sbase + kQOff + koff, 16, 1024),
                       smem_desc(kt + koff, 16, 1024), idesc_s, ks > 0);
          }
          tc_commit(bar_s_full + 8 * (js % kNS));
          tc_commit_multicast(bar_k_empty + 8 * (js % kNK), kMask);
          ++js;
          progressed = true;
        }
        // O += P_jp V_jp once the softmax wrote P_jp and V_jp landed
        if (jp < js && mbar_test_wait(bar_p_full + 8 * (jp % kNS), (jp / kNS) & 1) &&
            mbar_test_wait(bar_v_full + 8 * (jp % kNV), (jp / kNV) & 1)) {
          tc_fence_after();
          const uint32_t vt = sbase + kVOff + (jp % kNV) * kTileBytes;
#pragma unroll
          for (int ks = 0; ks < 8; ++ks)
            tc_mma_f16_tmem_a(tmem + kTmemO, tmem + (jp % kNS) * 128 + (ks >> 2) * 64 + (ks & 3) * 8,
                              smem_desc(vt + ks * 16 * 128, kHalf, 1024), idesc_o,
                              (jp > 0 || ks > 0) ? 1u : 0u);
          tc_commit(bar_o_done + 8 * (jp % kNS));
          tc_commit_multicast(bar_v_empty + 8 * (jp % kNV), kMask);
          ++jp;
          progressed = true;
        }
        if (progressed) {
          t_last = global_ns();
        } else if (*abort_flag || global_ns() - t_last > kWaitLimitNs) {
          if (!*abort_flag) {
            *abort_flag = 1;
            atomicOr(a.err, PA_DEVERR_TIMEOUT);
          }
          ok = false;
        }
      }
    }
    __syncwarp();
  } else {
    // ------------------------------------------------------------ softmax warps
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
      wait_or_abort_warp(bar_s_full + 8 * b3, (j / kNS) & 1, abort_flag, a.err);
      tc_fence_after();
      tmem_ld64(tmem + lane_off + b3 * 128 + hc * 64, v);

      const int kb = j * kTileKeys + hc * 64;
      const int nvis = lim - kb + 1;  // visible columns of this half (may be <= 0 or > 64)
      // eight independent partial maxima keep the dependency chains short; a
      // warp whose rows all see the whole half skips the per-element masks
      const bool full = __all_sync(0xffffffffu, nvis >= 64);
      float mp[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) mp[k] = -INFINITY;
      if (full) {
#pragma unroll
        for (int i = 0; i < 64; ++i) mp[i & 7] = fmaxf(mp[i & 7], __uint_as_float(v[i]));
      } else {
#pragma unroll
        for (int i = 0; i < 64; ++i)
          if (i < nvis) mp[i & 7] = fmaxf(mp[i & 7], __uint_as_float(v[i]));
      }
      float mloc = fmaxf(fmaxf(fmaxf(mp[0], mp[1]), fmaxf(mp[2], mp[3])),
                         fmaxf(fmaxf(mp[4], mp[5]), fmaxf(mp[6], mp[7])));
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
        wait_or_abort_warp(bar_o_done + 8 * ((j - 1) % kNS), ((j - 1) / kNS) & 1, abort_flag,
                           a.err);
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
      // the sequence's last block may end inside this tile: its slots past
      // seq_len hold no token and must not reach the PV product
      if ((n & (kBlockSize - 1)) != 0) {
        const int jl = (n - 1) / kBlockSize;
        if (jl < nb_vis && jl / 8 == j) {
          wait_or_abort_warp(bar_v_full + 8 * (j % kNV), (j / kNV) & 1, abort_flag, a.err);
          const uint32_t vt = sbase + kVOff + (j % kNV) * kTileBytes;
          const int first = n - jl * kBlockSize;  // rows first..15 of block jl % 8
          const int rows = kBlockSize - first;
          for (int e = tid; e < rows * 2 * 8; e += kSoftmaxWarps * 32) {
            const int row = first + e / 16, h = (e / 8) & 1, chunk = e & 7;
            const uint32_t addr =
                vt + h * kHalf + ((jl & 7) * kBlockSize + row) * 128 + (chunk << 4);
            asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u)
                         : "memory");
          }
        }
      }
      fence_proxy_async_smem();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_p_full + 8 * b3);
    }

    // ---- epilogue: O / l -> bf16, and lse
    wait_or_abort_warp(bar_o_done + 8 * ((nkt - 1) % kNS), ((nkt - 1) / kNS) & 1, abort_flag,
                       a.err);
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
  cluster_sync();  // no member leaves while a partner may still write to it
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
  chunk_exit(a, tid);
}

}  // namespace

size_t prefill_smem_bytes() { return kSmemBytes + 1024; }

int prefill_cluster(bool co_scheduled) { return co_scheduled ? 1 : kClusterAlone; }

namespace {
template <int kCluster>
cudaError_t launch_prefill_as(const PrefillArgs& a, const CUtensorMap* tm_q,
                              const CUtensorMap* tm_k, const CUtensorMap* tm_v, int grid_tiles,
                              cudaStream_t stream) {
  const size_t smem = prefill_smem_bytes();
  // raise the kernel's dynamic shared-memory limit once per device
  static std::mutex mu;
  static bool set_for[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set_for[dev]) {
      e = cudaFuncSetAttribute(prefill_kernel<kCluster>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      set_for[dev] = true;
    }
  }
  // programmatic dependent launch: the CTAs may start while the previous
  // kernel on the stream finishes; they touch no global memory before
  // griddepcontrol.wait (co-scheduled: see chunk_exit)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = kCluster;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, prefill_kernel<kCluster>, *tm_q, *tm_k, *tm_v, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}
}  // namespace

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                           const CUtensorMap* tm_v, int grid_tiles, cudaStream_t stream) {
  return a.after_decode ? launch_prefill_as<1>(a, tm_q, tm_k, tm_v, grid_tiles, stream)
                        : launch_prefill_as<kClusterAlone>(a, tm_q, tm_k, tm_v, grid_tiles, stream);
}

}  // namespace pa
