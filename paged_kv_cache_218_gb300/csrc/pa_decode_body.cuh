// pa_decode_body.cuh -- the paged decode's device code (one CTA's work,
// decode_cta) and its shared-memory plan, included by the decode launcher
// (pa_decode.cu) and by the fused hybrid launch (pa_hybrid.cu).
//
// One query per sequence attends over its paged KV ("03 - Engines Papers",
// section 2 PagedAttention: the kernel gathers K/V from non-contiguous
// 16-token blocks named by the block table).  Design:
//
//  * Persistent CTAs, at most one per SM: 8 consumer warps, 1 producer warp
//    and 1 merge warp (which takes the merge tickets of the balanced split's
//    mid-walk partial pieces).
//  * Work is a list of (sequence, block range) pieces covering *all* kv heads
//    of each block, so one physical block -- 16 tokens x Hkv heads x D,
//    contiguous in the pool -- is streamed as a whole (DRAM-page friendly).
//    The balanced split cuts the batch's blocks into one contiguous range per
//    CTA on a cost coordinate where each sequence adds a fixed cost, so a
//    range that starts sequences (pieces) gets fewer blocks.
//  * Variants: KV8 reads E4M3 pools (converted to f16 in registers); AP
//    writes each sequence's new token into its slot and into the landed
//    stage (the scatter fused into the decode step).
//  * The producer walks the CTA's pieces, prefetches block-table rows 32
//    entries at a time, and lands each block in a ring of shared-memory
//    stages with TMA tensor loads: for K and for V, one box per 64-column
//    half covering 16 tokens x every kv head (the pool is described to TMA as
//    (columns, tokens, heads), so a box lands as [head][token][64 columns]),
//    128-byte swizzled so warp-level matrix loads are bank-conflict free.
//    One mbarrier per stage counts the bytes in.
//  * Consumer warps map to kv heads (with Hkv < 8, several warps share a head
//    and split its blocks).  GQA: the group's q heads are the N=8 columns of
//    a warp MMA, so each K/V byte loaded serves every q head of its group:
//    S^T[16 tok x 8 heads] = K[16 x D] Q^T (mma.m16n8k16, bf16 in, fp32
//    accumulate), a per-head online softmax over the block's 16 scores with
//    warp-shuffle max reductions (the Milakov & Gimelshein recurrence,
//    "References" page), then O^T[D x 8] += V^T P^T.
//  * At the end of a piece the result is written: final bf16 output, a
//    fixed-partition partial for the LSE merge kernel, or (balanced mode) a
//    partial that the last-arriving CTA of that sequence merges in place by
//    log-sum-exp ("03 - Engines Papers", section 12 Cascade Inference;
//    split-K reduction of "The LLM inference engine playbook", Theme 4).
//
// No wait is unbounded: every mbarrier spin gives up after a two-second limit,
// sets PA_DEVERR_TIMEOUT, and the CTA then skips the rest of its work while
// still meeting its named barriers.
#pragma once

#include <math.h>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace dec {
namespace {


constexpr int kConsumerWarps = 8;
constexpr int kConsumerThreads = kConsumerWarps * 32;
constexpr int kProducerWarp = kConsumerWarps;
constexpr int kMergeWarp = kConsumerWarps + 1;  // balanced split: tickets of mid-walk partials
constexpr int kHandOffs = 2;  // partial pieces a CTA's walk can hand to the merge warp
constexpr int kThreads = kConsumerThreads + 64;
constexpr int kBoxBytes = 16 * 128;  // one TMA box: 16 token rows x 64 bf16
constexpr int kMaxStages = 16;
constexpr float kLn2 = 0.6931471805599453f;
constexpr int kLenCache = 512;  // balanced mode keeps the lengths in shared memory up to this batch

// Shared-memory ints of the balanced mode's per-sequence data: the exclusive
// prefix of block counts (S + 1) and, for small batches, the lengths (S).
__host__ __device__ inline int balanced_pre_ints(int S) { return S + 1 + (S <= kLenCache ? S : 0); }

enum PieceKind : int { kFinal = 0, kPartialFixed = 1, kPartialBalanced = 2 };

struct Piece {
  int s, j0, j1, len, nb, kind, part, which, first;
  long long seg_start;
};

struct Cursor {
  long long u, U;         // fixed / single-pass unit walk
  int step;               // fixed / single-pass: CTAs of the decode
  long long idx, lo, hi;  // balanced block range [lo, hi)
  long long mid, end;     // balanced: walk [mid, hi) first, then [lo, mid)
  long long W;            // balanced: total blocks
  long long T;            // balanced: total cost, W + beta * S
  int C;                  // balanced: CTAs that own a range
  int beta;               // balanced: cost of a sequence, in blocks
  int phase;              // balanced: 0 while walking [mid, hi)
};

// Shared-memory carve-up (byte offsets from a 1024-aligned base).
struct Layout {
  int head_bytes;   // K (or V) of one block, one kv head
  int stage_bytes;  // K + V of one block, all kv heads
  int stages;
  int q_bytes;      // one staged query row set: Hq x D bf16
  int q_off, obuf_off, ml_off, nk_off, bar_off, misc_off, pre_off, total;
};

// Append: per consumer warp, its kv head's new K row and V row (D bf16 each)
// and the id of the sequence's last block.
__host__ __device__ constexpr int new_row_bytes(int D) { return 4 * D + 16; }

__host__ __device__ inline Layout make_layout(int D, int Hkv, int Hq, int wph, int stages,
                                              int pre_ints, int elem_bytes, bool append = false) {
  Layout L;
  L.head_bytes = kBlockSize * D * elem_bytes;
  L.stage_bytes = 2 * Hkv * L.head_bytes;
  L.stages = stages;
  L.q_bytes = (Hq * D * 2 + 127) / 128 * 128;
  L.q_off = stages * L.stage_bytes;
  L.obuf_off = L.q_off + 2 * L.q_bytes;
  const int obuf = wph > 1 ? kConsumerWarps * kMaxGroup * (D + 4) * 4 : 0;
  L.ml_off = L.obuf_off + obuf;
  L.nk_off = L.ml_off + kConsumerWarps * kMaxGroup * 2 * 4;
  L.bar_off = L.nk_off + (append ? kConsumerWarps * new_row_bytes(D) : 0);
  L.misc_off = L.bar_off + (kMaxStages * 2 + 8) * 8;
  L.pre_off = L.misc_off + 128;  // misc: flags, tickets, scan partials, per-warp words
  L.total = L.pre_off + pre_ints * 4;
  return L;
}

__device__ __forceinline__ int load_len(const DecodeArgs& a, int s, bool report) {
  int len = __ldcg(a.seq_lens + s);
  const int cap = a.max_blocks * kBlockSize;
  if (len < 0 || len > cap) {
    if (report) atomicOr(a.err, PA_DEVERR_SEQ_LEN);
    len = len < 0 ? 0 : cap;
  }
  return len;
}

// First block of sequence s this launch attends to: 0, or the cascade suffix
// pass's start block (clamped to [0, ceil(len/16)]).
__device__ __forceinline__ int start_block(const DecodeArgs& a, int s, int len, bool report) {
  if (!a.start_blocks) return 0;
  int sb = __ldcg(a.start_blocks + s);
  const int nb = (len + kBlockSize - 1) / kBlockSize;
  if (sb < 0) {
    if (report) atomicOr(a.err, PA_DEVERR_GROUP);
    sb = 0;
  }
  return sb > nb ? nb : sb;
}

// The balanced split charges every sequence a fixed cost of beta blocks on
// top of its blocks: a piece costs its CTA more than its blocks (the queries'
// fragments, the partial result and its merge ticket), so a range that starts
// sequences gets fewer blocks.  Block x of sequence s sits at cost coordinate
// x + beta * (s + 1); CTA c of C owns the costs [c*T/C, (c+1)*T/C) (floors),
// T = W + beta * S.  owner_of_cost: the CTA owning cost point y.
__device__ __forceinline__ long long owner_of_cost(long long y, long long T, int C) {
  return ((y + 1) * C + T - 1) / T - 1;
}

// The smallest block whose cost coordinate is at least y (W if none).
__device__ __forceinline__ long long block_at_cost(const int* pre, int S, int beta, long long y) {
  // the first sequence s whose last cost point pre[s+1] - 1 + beta*(s+1) is >= y
  int lo = 0, hi = S;
  while (lo < hi) {
    const int mid = (lo + hi) >> 1;
    if (pre[mid + 1] + static_cast<long long>(beta) * (mid + 1) > y)
      hi = mid;
    else
      lo = mid + 1;
  }
  if (lo == S) return pre[S];
  const long long x = y - static_cast<long long>(beta) * (lo + 1);
  return x > pre[lo] ? x : pre[lo];
}

// the sequence holding global block x: the largest s with pre[s] <= x
__device__ __forceinline__ int seq_of(const int* pre, int S, long long x) {
  int lo = 0, hi = S - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (pre[mid] <= x) lo = mid; else hi = mid - 1;
  }
  return lo;
}

__device__ bool next_piece(const DecodeArgs& a, const int* pre, const int* lens_c, Cursor& c,
                           Piece& p, bool report) {
  if (a.mode == kModeBalanced) {
    if (c.idx >= c.end) {
      if (c.phase != 0) return false;
      c.phase = 1;
      c.idx = c.lo;
      c.end = c.mid;
      if (c.idx >= c.end) return false;
    }
    const int s = seq_of(pre, a.num_seqs, c.idx);
    p.s = s;
    p.nb = pre[s + 1] - pre[s];
    p.seg_start = pre[s];
    const int r0 = static_cast<int>(c.idx - p.seg_start);
    const long long seg_end = p.seg_start + p.nb;
    const long long end = c.end < seg_end ? c.end : seg_end;
    const int r1 = r0 + static_cast<int>(end - c.idx);
    c.idx = end;
    p.len = lens_c ? lens_c[s] : load_len(a, s, false);
    const int sb = start_block(a, s, p.len, false);
    p.j0 = sb + r0;
    p.j1 = sb + r1;
    p.first = r0 == 0;
    p.kind = (r0 == 0 && r1 == p.nb) ? kFinal : kPartialBalanced;
    p.which = p.seg_start < c.lo ? 0 : 1;
    p.part = 0;
    return true;
  }
  while (c.u < c.U) {
    const long long u = c.u;
    c.u += c.step;
    const int part = static_cast<int>(u % a.max_parts);
    const int s = static_cast<int>(u / a.max_parts);
    const int len = load_len(a, s, report && part == 0);
    const int nb = (len + kBlockSize - 1) / kBlockSize;
    const int sb = start_block(a, s, len, report && part == 0);
    const int ns = nb - sb;
    const int nparts = ns == 0 ? 1 : (ns + a.part_blocks - 1) / a.part_blocks;
    if (part >= nparts) continue;
    p.s = s;
    p.len = len;
    p.nb = nb;
    p.j0 = sb + part * a.part_blocks;
    p.j1 = min(nb, p.j0 + a.part_blocks);
    p.first = part == 0;
    p.kind = nparts == 1 ? kFinal : kPartialFixed;
    p.part = part;
    p.which = 0;
    p.seg_start = 0;
    return true;
  }
  return false;
}

// Block ids jb .. jb+n-1 of sequence s, one per lane (read from L2: lengths
// and tables are metadata a CTA may also read before its grid-dependency
// wait, and a line cached in L1 then could be stale).  load_id_raw issues the
// read; check_id flags a bad id and turns it into -1 (the TMA box then lies
// outside the pool and reads zeros).
__device__ __forceinline__ int load_id_raw(const DecodeArgs& a, int s, int jb, int n, int lane) {
  return lane < n ? __ldcg(a.block_tables + static_cast<long long>(s) * a.max_blocks + jb + lane)
                  : 0;
}

__device__ __forceinline__ int check_id(const DecodeArgs& a, int id, int n, int lane) {
  if (lane < n && (id < 0 || id >= a.num_blocks)) {
    atomicOr(a.err, PA_DEVERR_BLOCK_ID);
    id = -1;
  }
  return id;
}

__device__ __forceinline__ int load_ids(const DecodeArgs& a, int s, int jb, int n, int lane) {
  return check_id(a, load_id_raw(a, s, jb, n, lane), n, lane);
}

// Address of the 16-byte chunk `chunk` (8 bf16) of token row `tok` in one
// head's block.  A stage holds, for K and then for V, one 128-byte-swizzled
// box per 64-column half covering [head][16 tokens][64 columns]; `half` is
// the distance between the two halves (Hkv x 16 rows x 128 B).
__device__ __forceinline__ uint32_t swz(uint32_t base, int tok, int chunk, uint32_t half) {
  return base + (chunk >> 3) * half + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4);
}

// Scores x[e] of S^T for one bf16 block (fragment element e: tokens lane/4
// and lane/4 + 8, heads 2q and 2q + 1) in log2 units, -inf at or past
// `valid`.  Four independent accumulation chains of KS/4 k-steps each cut the
// dependent MMA latency.
template <int D>
__device__ __forceinline__ void bf16_scores(uint32_t kbase, uint32_t half,
                                            const uint32_t (&qf)[D / 16][2], float scale_log2,
                                            int valid, int lane, float (&x)[4]) {
  constexpr int KS = D / 16;
  const int i = lane >> 3, r = lane & 7;
  float sc[4][4];
#pragma unroll
  for (int c = 0; c < 4; ++c) sc[c][0] = sc[c][1] = sc[c][2] = sc[c][3] = 0.f;
  const int ktok = r + ((i & 1) << 3);
#pragma unroll
  for (int ks = 0; ks < KS; ks += 2) {
    uint32_t a0[4], a1[4];
    ldsm_x4(swz(kbase, ktok, ks * 2 + (i >> 1), half), a0);
    ldsm_x4(swz(kbase, ktok, (ks + 1) * 2 + (i >> 1), half), a1);
    mma_bf16_16816(sc[ks & 3], a0, qf[ks][0], qf[ks][1]);
    mma_bf16_16816(sc[(ks + 1) & 3], a1, qf[ks + 1][0], qf[ks + 1][1]);
  }
  const int t0 = lane >> 2;
  const bool v0 = t0 < valid, v1 = t0 + 8 < valid;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    x[e] = (e < 2 ? v0 : v1) ? ((sc[0][e] + sc[1][e]) + (sc[2][e] + sc[3][e])) * scale_log2
                             : -INFINITY;
}

// O^T += V^T P^T for one bf16 block: P^T fragments b0, b1; V rows of tokens at
// or past `valid` zeroed (their p is 0, but their rows may hold anything).
template <int D>
__device__ __forceinline__ void bf16_pv(uint32_t vbase, uint32_t half, uint32_t b0, uint32_t b1,
                                        int valid, int lane, float (&o)[D / 16][4]) {
  constexpr int KS = D / 16;
  const int i = lane >> 3, r = lane & 7;
  const int vtok = r + ((i >> 1) << 3);
  uint32_t keep01 = 0xffffffffu, keep23 = 0xffffffffu;
  if (valid < 16) {
    const int q2 = (lane & 3) * 2;
    keep01 = (q2 < valid ? 0x0000ffffu : 0u) | (q2 + 1 < valid ? 0xffff0000u : 0u);
    keep23 = (q2 + 8 < valid ? 0x0000ffffu : 0u) | (q2 + 9 < valid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    uint32_t a[4];
    ldsm_x4_trans(swz(vbase, vtok, mt * 2 + (i & 1), half), a);
    a[0] &= keep01;
    a[1] &= keep01;
    a[2] &= keep23;
    a[3] &= keep23;
    mma_bf16_16816(o[mt], a, b0, b1);
  }
}

template <int D>
__device__ __forceinline__ void attend_block(uint32_t kbase, uint32_t vbase, uint32_t half,
                                             const uint32_t (&qf)[D / 16][2],
                                             float (&o)[D / 16][4], float& m0, float& m1,
                                             float& l0, float& l1, int valid, float scale_log2,
                                             int lane) {
  constexpr int KS = D / 16;
  float x[4];
  bf16_scores<D>(kbase, half, qf, scale_log2, valid, lane, x);
  float mxa = fmaxf(x[0], x[2]), mxb = fmaxf(x[1], x[3]);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
  }
  const float mna = fmaxf(m0, mxa), mnb = fmaxf(m1, mxb);
  const float aa = fast_exp2(m0 - mna), ab = fast_exp2(m1 - mnb);
  const float pa0 = fast_exp2(x[0] - mna), pb0 = fast_exp2(x[1] - mnb);
  const float pa1 = fast_exp2(x[2] - mna), pb1 = fast_exp2(x[3] - mnb);
  l0 = l0 * aa + pa0 + pa1;
  l1 = l1 * ab + pb0 + pb1;
  m0 = mna;
  m1 = mnb;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    o[mt][0] *= aa;
    o[mt][1] *= ab;
    o[mt][2] *= aa;
    o[mt][3] *= ab;
  }
  // P^T as the B operand (k = token, n = head): transpose the two 8x8 halves
  bf16_pv<D>(vbase, half, movmatrix_trans(pack_bf16x2(pa0, pb0)),
             movmatrix_trans(pack_bf16x2(pa1, pb1)), valid, lane, o);
}

// Two consecutive bf16 blocks of one piece (the first full), as
// attend_pair_fp8 does for E4M3.
template <int D>
__device__ __forceinline__ void attend_pair(uint32_t kbase0, uint32_t vbase0, uint32_t kbase1,
                                            uint32_t vbase1, uint32_t half,
                                            const uint32_t (&qf)[D / 16][2],
                                            float (&o)[D / 16][4], float& m0, float& m1,
                                            float& l0, float& l1, int valid, float scale_log2,
                                            int lane) {
  constexpr int KS = D / 16;
  float x[4], y[4];
  bf16_scores<D>(kbase0, half, qf, scale_log2, 16, lane, x);
  bf16_scores<D>(kbase1, half, qf, scale_log2, valid, lane, y);
  float mxa = fmaxf(fmaxf(x[0], x[2]), fmaxf(y[0], y[2]));
  float mxb = fmaxf(fmaxf(x[1], x[3]), fmaxf(y[1], y[3]));
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
  }
  const float mna = fmaxf(m0, mxa), mnb = fmaxf(m1, mxb);
  const float aa = fast_exp2(m0 - mna), ab = fast_exp2(m1 - mnb);
  const float pa0 = fast_exp2(x[0] - mna), pb0 = fast_exp2(x[1] - mnb);
  const float pa1 = fast_exp2(x[2] - mna), pb1 = fast_exp2(x[3] - mnb);
  const float qa0 = fast_exp2(y[0] - mna), qb0 = fast_exp2(y[1] - mnb);
  const float qa1 = fast_exp2(y[2] - mna), qb1 = fast_exp2(y[3] - mnb);
  l0 = l0 * aa + ((pa0 + pa1) + (qa0 + qa1));
  l1 = l1 * ab + ((pb0 + pb1) + (qb0 + qb1));
  m0 = mna;
  m1 = mnb;
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    o[mt][0] *= aa;
    o[mt][1] *= ab;
    o[mt][2] *= aa;
    o[mt][3] *= ab;
  }
  bf16_pv<D>(vbase0, half, movmatrix_trans(pack_bf16x2(pa0, pb0)),
             movmatrix_trans(pack_bf16x2(pa1, pb1)), 16, lane, o);
  bf16_pv<D>(vbase1, half, movmatrix_trans(pack_bf16x2(qa0, qb0)),
             movmatrix_trans(pack_bf16x2(qa1, qb1)), valid, lane, o);
}

// One 16-token block of E4M3 K/V for one kv head (head_dim 128).  The stage
// holds, for K and then for V, one box [head][token][128 bytes] with the
// 128-byte swizzle.  A lane converts its own bytes to f16 in registers
// (exactly: every E4M3 value is an f16 value) and the contractions run as f16
// warp MMAs.  The head dimension is visited in a permuted order, the same for
// the query fragments (a dot product does not depend on the order), so that a
// lane's bytes are contiguous:
//  * S^T = K Q^T: lane (g, c) holds, at k-step ks, dims 32c + 4ks + {0, 1}
//    (fragment columns 2c, 2c+1) and 32c + 4ks + {2, 3} (columns 2c+8, 2c+9)
//    of tokens g and g + 8: two 16-byte loads per token row;
//  * O^T += V^T P^T: row g of m-tile mt is dim 16g + 2mt and row g + 8 is dim
//    16g + 2mt + 1 (out_dim<true>), so lane (g, c) needs dims [16g, 16g + 16)
//    of tokens 2c, 2c+1, 2c+8, 2c+9: one 16-byte load per token, and byte
//    pairs of two tokens are interleaved with prmt before the conversion.
// The scores come out in units of sl2 (the query's power-of-two scale and the
// K scale folded in); the V scale is applied to the finished output.
// Pieces of the E4M3 block routines below (head_dim 128).
// The block's K bytes of this lane: tokens g and g + 8, 32 bytes each.
__device__ __forceinline__ void fp8_load_k(uint32_t kbase, int lane, uint32_t (&kw)[2][8]) {
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int r = 0; r < 2; ++r) {
    const int tok = g + 8 * r;
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const uint4 v = lds128(kbase + tok * 128 + (((2 * c + h) ^ (tok & 7)) << 4));
      kw[r][4 * h + 0] = v.x;
      kw[r][4 * h + 1] = v.y;
      kw[r][4 * h + 2] = v.z;
      kw[r][4 * h + 3] = v.w;
    }
  }
}

// The block's V bytes of this lane: dims [16g, 16g + 16) of tokens 2c, 2c+1,
// 2c+8, 2c+9.
__device__ __forceinline__ void fp8_load_v(uint32_t vbase, int lane, uint32_t (&vw)[4][4]) {
  const int g = lane >> 2, c = lane & 3;
#pragma unroll
  for (int r = 0; r < 4; ++r) {
    const int tok = 2 * c + (r & 1) + 8 * (r >> 1);
    const uint4 v = lds128(vbase + tok * 128 + ((g ^ (tok & 7)) << 4));
    vw[r][0] = v.x;
    vw[r][1] = v.y;
    vw[r][2] = v.z;
    vw[r][3] = v.w;
  }
}

// Scores x[e] of S^T (fragment element e: tokens lane/4 and lane/4 + 8, heads
// 2c and 2c + 1) in sl2 units, -inf for tokens at or past `valid`.  Four
// independent MMA chains of two k-steps each: this path is bound by the
// latency of a consumer warp's work per block.
__device__ __forceinline__ void fp8_scores(const uint32_t (&kw)[2][8], const uint32_t (&qf)[8][2],
                                           float sl2, int valid, int lane, float (&x)[4]) {
  float sc[4][4];
#pragma unroll
  for (int i = 0; i < 4; ++i) sc[i][0] = sc[i][1] = sc[i][2] = sc[i][3] = 0.f;
#pragma unroll
  for (int ks = 0; ks < 8; ++ks) {
    uint32_t ka[4];
    ka[0] = e4m3x2_to_f16x2(kw[0][ks]);
    ka[1] = e4m3x2_to_f16x2(kw[1][ks]);
    ka[2] = e4m3x2_to_f16x2(kw[0][ks] >> 16);
    ka[3] = e4m3x2_to_f16x2(kw[1][ks] >> 16);
    mma_f16_16816(sc[ks & 3], ka, qf[ks][0], qf[ks][1]);
  }
  const int t0 = lane >> 2;
  const bool v0 = t0 < valid, v1 = t0 + 8 < valid;
#pragma unroll
  for (int e = 0; e < 4; ++e)
    x[e] = (e < 2 ? v0 : v1) ? ((sc[0][e] + sc[1][e]) + (sc[2][e] + sc[3][e])) * sl2 : -INFINITY;
}

// O^T += V^T P^T for one block: P^T fragments b0, b1; V halves of tokens at or
// past `valid` zeroed (their p is 0, but their bytes may hold anything).
__device__ __forceinline__ void fp8_pv(const uint32_t (&vw)[4][4], uint32_t b0, uint32_t b1,
                                       int valid, int lane, float (&o)[8][4]) {
  uint32_t keep01 = 0xffffffffu, keep23 = 0xffffffffu;
  if (valid < 16) {
    const int q2 = (lane & 3) * 2;
    keep01 = (q2 < valid ? 0x0000ffffu : 0u) | (q2 + 1 < valid ? 0xffff0000u : 0u);
    keep23 = (q2 + 8 < valid ? 0x0000ffffu : 0u) | (q2 + 9 < valid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    const int j = mt >> 1;
    const uint32_t sel = (mt & 1) ? 0x7362u : 0x5140u;  // bytes 2mt, 2mt+1 of two tokens
    const uint32_t t01 = prmt(vw[0][j], vw[1][j], sel);
    const uint32_t t23 = prmt(vw[2][j], vw[3][j], sel);
    uint32_t va[4];
    va[0] = e4m3x2_to_f16x2(t01) & keep01;
    va[1] = e4m3x2_to_f16x2(t01 >> 16) & keep01;
    va[2] = e4m3x2_to_f16x2(t23) & keep23;
    va[3] = e4m3x2_to_f16x2(t23 >> 16) & keep23;
    mma_f16_16816(o[mt], va, b0, b1);
  }
}

template <int D>
__device__ __forceinline__ void attend_block_fp8(uint32_t kbase, uint32_t vbase,
                                                 const uint32_t (&qf)[D / 16][2],
                                                 float (&o)[D / 16][4], float& m0, float& m1,
                                                 float& l0, float& l1, int valid, float sl2,
                                                 int lane) {
  static_assert(D == 128, "the E4M3 path has 128-byte token rows");
  uint32_t kw[2][8], vw[4][4];
  fp8_load_k(kbase, lane, kw);
  fp8_load_v(vbase, lane, vw);  // read now: the latency hides under the scores
  float x[4];
  fp8_scores(kw, qf, sl2, valid, lane, x);
  float mxa = fmaxf(x[0], x[2]), mxb = fmaxf(x[1], x[3]);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
  }
  const float mna = fmaxf(m0, mxa), mnb = fmaxf(m1, mxb);
  const float aa = fast_exp2(m0 - mna), ab = fast_exp2(m1 - mnb);
  const float pa0 = fast_exp2(x[0] - mna), pb0 = fast_exp2(x[1] - mnb);
  const float pa1 = fast_exp2(x[2] - mna), pb1 = fast_exp2(x[3] - mnb);
  l0 = l0 * aa + pa0 + pa1;
  l1 = l1 * ab + pb0 + pb1;
  m0 = mna;
  m1 = mnb;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    o[mt][0] *= aa;
    o[mt][1] *= ab;
    o[mt][2] *= aa;
    o[mt][3] *= ab;
  }
  fp8_pv(vw, movmatrix_trans(pack_f16x2(pa0, pb0)), movmatrix_trans(pack_f16x2(pa1, pb1)), valid,
         lane, o);
}

// Two consecutive blocks of one piece (the first one full, the second with
// `valid` tokens) in one step: both score chains at once, one online-softmax
// update over the 32 tokens, one rescale of the accumulators, then both PV
// products.  Twice the independent work per dependency chain.
template <int D>
__device__ __forceinline__ void attend_pair_fp8(uint32_t kbase0, uint32_t vbase0, uint32_t kbase1,
                                                uint32_t vbase1, const uint32_t (&qf)[D / 16][2],
                                                float (&o)[D / 16][4], float& m0, float& m1,
                                                float& l0, float& l1, int valid, float sl2,
                                                int lane) {
  static_assert(D == 128, "the E4M3 path has 128-byte token rows");
  float x[4], y[4];
  {
    uint32_t kw[2][8], kv[2][8];
    fp8_load_k(kbase0, lane, kw);
    fp8_load_k(kbase1, lane, kv);
    fp8_scores(kw, qf, sl2, 16, lane, x);
    fp8_scores(kv, qf, sl2, valid, lane, y);
  }
  float mxa = fmaxf(fmaxf(x[0], x[2]), fmaxf(y[0], y[2]));
  float mxb = fmaxf(fmaxf(x[1], x[3]), fmaxf(y[1], y[3]));
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
  }
  const float mna = fmaxf(m0, mxa), mnb = fmaxf(m1, mxb);
  const float aa = fast_exp2(m0 - mna), ab = fast_exp2(m1 - mnb);
  const float pa0 = fast_exp2(x[0] - mna), pb0 = fast_exp2(x[1] - mnb);
  const float pa1 = fast_exp2(x[2] - mna), pb1 = fast_exp2(x[3] - mnb);
  const float qa0 = fast_exp2(y[0] - mna), qb0 = fast_exp2(y[1] - mnb);
  const float qa1 = fast_exp2(y[2] - mna), qb1 = fast_exp2(y[3] - mnb);
  l0 = l0 * aa + ((pa0 + pa1) + (qa0 + qa1));
  l1 = l1 * ab + ((pb0 + pb1) + (qb0 + qb1));
  m0 = mna;
  m1 = mnb;
#pragma unroll
  for (int mt = 0; mt < 8; ++mt) {
    o[mt][0] *= aa;
    o[mt][1] *= ab;
    o[mt][2] *= aa;
    o[mt][3] *= ab;
  }
  uint32_t vw[4][4];
  fp8_load_v(vbase0, lane, vw);
  fp8_pv(vw, movmatrix_trans(pack_f16x2(pa0, pb0)), movmatrix_trans(pack_f16x2(pa1, pb1)), 16,
         lane, o);
  fp8_load_v(vbase1, lane, vw);
  fp8_pv(vw, movmatrix_trans(pack_f16x2(qa0, qb0)), movmatrix_trans(pack_f16x2(qa1, qb1)), valid,
         lane, o);
}

// Head-dimension index of output fragment row g (+8 when half = 1) of m-tile
// mt: natural order for bf16, the permuted order of attend_block_fp8 for E4M3.
template <bool KV8>
__device__ __forceinline__ int out_dim(int mt, int g, int half) {
  return KV8 ? 16 * g + 2 * mt + half : mt * 16 + g + 8 * half;
}

// Log-sum-exp merge of a sequence's partial pieces, held in the slots of CTAs
// c_first (its "after" slot) and c_first+1 .. c_first+npieces-1 ("before"
// slots); writes the final bf16 output (and lse).  Each thread owns kNI float4
// groups of the output and keeps, per group, the running maximum M, the sum
// S = sum_k exp(lse_k - M) and the weighted sum of the pieces' outputs.  The
// pieces are read kKB at a time with all their loads issued together, so a
// merge of up to kKB pieces costs about one L2 round trip.  NT threads take
// part (ctid in [0, NT)): the consumers, or the merge warp.  Inlined: it runs
// inside the piece loop, where a call would save the loop's live registers to
// the stack around it.
template <int D, int NT>
__device__ __forceinline__ void merge_pieces(const DecodeArgs& a, int s, long long c_first,
                                             int npieces, int ctid) {
  const int Hq = a.num_q_heads;
  constexpr int kNI = NT >= 256 ? 4 : 2;  // float4 groups per thread per batch
  constexpr int kKB = NT >= 256 ? 4 : 2;  // pieces per round
  const int nf = Hq * D / 4;
  const long long row0 = static_cast<long long>(s) * Hq;
  for (int fb0 = 0; fb0 < nf; fb0 += kNI * NT) {
    float4 acc[kNI];
    float M[kNI], S[kNI];
#pragma unroll
    for (int i = 0; i < kNI; ++i) {
      acc[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      M[i] = -INFINITY;
      S[i] = 0.f;
    }
#pragma unroll 1
    for (int k0 = 0; k0 < npieces; k0 += kKB) {
      float4 ok[kKB][kNI];
      float lk[kKB][kNI];
#pragma unroll
      for (int u = 0; u < kKB; ++u) {
        const int k = k0 + u;
        const float* sl =
            a.part_o + ((c_first + (k < npieces ? k : 0)) * 2 + (k == 0 ? 1 : 0)) * a.slot_floats;
#pragma unroll
        for (int i = 0; i < kNI; ++i) {
          const int f = fb0 + ctid + i * NT;
          if (k < npieces && f < nf) {
            lk[u][i] = __ldcg(sl + Hq * D + (f * 4) / D);
            ok[u][i] = __ldcg(reinterpret_cast<const float4*>(sl) + f);
          } else {
            lk[u][i] = -INFINITY;
            ok[u][i] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
#pragma unroll
      for (int i = 0; i < kNI; ++i) {
        float mx = M[i];
#pragma unroll
        for (int u = 0; u < kKB; ++u) mx = fmaxf(mx, lk[u][i]);
        if (mx == -INFINITY) continue;
        const float sc = __expf(M[i] - mx);  // 0 while M is still -inf
        acc[i].x *= sc;
        acc[i].y *= sc;
        acc[i].z *= sc;
        acc[i].w *= sc;
        S[i] *= sc;
#pragma unroll
        for (int u = 0; u < kKB; ++u) {
          const float w = __expf(lk[u][i] - mx);  // 0 for absent pieces
          acc[i].x += w * ok[u][i].x;
          acc[i].y += w * ok[u][i].y;
          acc[i].z += w * ok[u][i].z;
          acc[i].w += w * ok[u][i].w;
          S[i] += w;
        }
        M[i] = mx;
      }
    }
#pragma unroll
    for (int i = 0; i < kNI; ++i) {
      const int f = fb0 + ctid + i * NT;
      if (f < nf) {
        const float inv = S[i] > 0.f ? 1.f / S[i] : 0.f;
        const uint2 pk = make_uint2(pack_bf16x2(acc[i].x * inv, acc[i].y * inv),
                                    pack_bf16x2(acc[i].z * inv, acc[i].w * inv));
        *reinterpret_cast<uint2*>(a.out + row0 * D + static_cast<long long>(f) * 4) = pk;
        if ((f * 4) % D == 0 && a.out_lse)
          a.out_lse[row0 + (f * 4) / D] = S[i] > 0.f ? M[i] + __logf(S[i]) : -INFINITY;
      }
    }
  }
}

// One CTA of the decode: CTA `cta` of `ncta` (a decode launch's block index
// and grid, or the decode role's share of a fused hybrid launch).  Uses the
// first kThreads threads of its CTA and the dynamic shared memory.
template <int D, bool KV8, bool AP>
__device__ __forceinline__ void decode_cta(const CUtensorMap& tm_k, const CUtensorMap& tm_v,
                                           const DecodeArgs& a, const int cta, const int ncta) {
  constexpr int KS = D / 16;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);

  const int Hkv = a.num_kv_heads, G = a.group, Hq = a.num_q_heads;
  const int wph = a.warps_per_head;
  const Layout L = make_layout(D, Hkv, Hq, wph, a.stages, 0, KV8 ? 1 : 2, AP);
  float* obuf = reinterpret_cast<float*>(smem + L.obuf_off);
  float* mlbuf = reinterpret_cast<float*>(smem + L.ml_off);
  int* misc = reinterpret_cast<int*>(smem + L.misc_off);
  int* pre = reinterpret_cast<int*>(smem + L.pre_off);
  const uint32_t bar_full = sbase + L.bar_off;
  const uint32_t bar_empty = bar_full + kMaxStages * 8;
  const uint32_t bar_qfull = bar_empty + kMaxStages * 8;  // two query slots
  const uint32_t bar_qempty = bar_qfull + 16;
  const uint32_t bar_hand = bar_qempty + 16;   // two: a mid-walk partial handed to the merge warp
  const uint32_t bar_tdone = bar_hand + 16;    // two: the merge warp took that piece's ticket
  const int NS = L.stages;
  const int active_warps = Hkv * wph < kConsumerWarps ? Hkv * wph : kConsumerWarps;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(bar_full + st * 8, 1);
      mbar_init(bar_empty + st * 8, Hkv);  // one arrival per kv head's warp
    }
    for (int k = 0; k < 2; ++k) {
      mbar_init(bar_qfull + k * 8, 1);
      mbar_init(bar_qempty + k * 8, active_warps);
      mbar_init(bar_hand + k * 8, kConsumerWarps);  // one arrival per consumer warp
      mbar_init(bar_tdone + k * 8, 1);
    }
    misc[0] = 0;   // abort flag
    misc[15] = 0;  // the walk's own pending merge (record kHandOffs), none yet
    fence_mbar_init();
  }
  named_barrier(4, kThreads);  // barriers initialized before any warp uses them
  // Launched as a programmatic dependent of the previous kernel on the stream,
  // the CTA may get here while that kernel still runs.  Until griddep_wait()
  // returns it writes no global memory, and it reads only lengths and start
  // blocks, for a plan that is checked after the wait (below).  It also asks
  // L2 for the lines of this launch's lengths, block tables and queries (at
  // most 4 MB of each), spread over every thread of the grid, so that the
  // reads after the wait hit L2.
  {
    const long long nthr = static_cast<long long>(ncta) * kThreads;
    const long long me = static_cast<long long>(cta) * kThreads + tid;
    auto warm = [&](const void* base, long long bytes) {
      bytes = bytes < (4ll << 20) ? bytes : (4ll << 20);
      for (long long off = me * 128; off < bytes; off += nthr * 128)
        prefetch_l2(static_cast<const char*>(base) + off);
    };
    warm(a.seq_lens, static_cast<long long>(a.num_seqs) * 4);
    warm(a.block_tables, static_cast<long long>(a.num_seqs) * a.max_blocks * 4);
    warm(a.q, static_cast<long long>(a.num_seqs) * Hq * D * 2);
  }
  // ---- balanced mode: the plan (exclusive prefix of block counts over
  // sequences, the CTA's range, its first piece and chunk), made by the
  // producer warp.  For batches whose lengths fit in shared memory it is made
  // before the grid-dependency wait, from lengths that the previous kernel
  // could still be writing: after the wait the producer reads the first
  // chunk's table row and, at the same time, the lengths and start blocks
  // once more; the plan stands if they read the same, and is made again if
  // not.  The first loads of the launch thus wait on one L2 round trip after
  // the previous kernel, not on three.
  const int S = a.num_seqs;
  int* lens_w = (a.mode == kModeBalanced && S <= kLenCache) ? pre + S + 1 : nullptr;
  const int* lens_c = lens_w;
  const int per = (S + 31) / 32;
  const int sl0 = min(S, lane * per), sl1 = min(S, sl0 + per);
  // prefix over the sequences (producer warp; lane takes [sl0, sl1))
  auto prefix = [&](bool report) {
    int local = 0;
    for (int s = sl0; s < sl1; ++s) {
      const int len = load_len(a, s, report);
      if (lens_w) lens_w[s] = len;
      local += (len + kBlockSize - 1) / kBlockSize - start_block(a, s, len, report);
    }
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    int run = incl - local;
    for (int s = sl0; s < sl1; ++s) {
      pre[s] = run;
      const int len = lens_w ? lens_w[s] : load_len(a, s, false);
      run += (len + kBlockSize - 1) / kBlockSize - start_block(a, s, len, false);
    }
    if (lane == 31) pre[S] = incl;
    __syncwarp();
  };
  Cursor cur{};
  auto init_cursor = [&]() {
    cur = Cursor{};
    cur.W = pre[S];
    cur.C = static_cast<int>(cur.W < ncta ? cur.W : ncta);
    // the per-sequence cost only once every CTA has a few blocks to stream
    cur.beta = cur.W >= 2ll * ncta ? a.piece_cost : 0;
    cur.T = cur.W + static_cast<long long>(cur.beta) * S;
    if (cta < cur.C) {
      cur.lo = block_at_cost(pre, S, cur.beta, static_cast<long long>(cta) * cur.T / cur.C);
      cur.hi = block_at_cost(pre, S, cur.beta, static_cast<long long>(cta + 1) * cur.T / cur.C);
    } else {
      cur.lo = cur.hi = 0;
    }
    // When the range's last sequence runs on into the next CTA's range, that
    // piece is walked first ([mid, hi), then [lo, mid)): the range's first
    // piece is also the first of [lo, mid), so both partial pieces of a
    // sequence split between neighbouring CTAs finish early in both, and its
    // merge happens while other blocks still stream, not at the launch's end.
    cur.mid = cur.lo;
    if (cur.hi > cur.lo) {
      const int sl = seq_of(pre, S, cur.hi - 1);
      if (pre[sl + 1] > cur.hi && pre[sl] > cur.lo) cur.mid = pre[sl];
    }
    cur.phase = cur.mid > cur.lo ? 0 : 1;
    cur.idx = cur.phase == 0 ? cur.mid : cur.lo;
    cur.end = cur.hi;
  };
  // the producer's walk: piece p, next block jbp of it, the first chunk
  Piece p{};
  int jbp = 0, c_s = 0, c_jb = 0, c_n = 0;
  bool have_p = false, have_c = false;
  auto first_chunk = [&]() {
    have_p = next_piece(a, pre, lens_c, cur, p, false);
    jbp = have_p ? p.j0 : 0;
    have_c = have_p && jbp < p.j1;  // a balanced piece holds at least one block
    if (have_c) {
      c_s = p.s;
      c_jb = jbp;
      c_n = min(32, p.j1 - jbp);
      jbp += c_n;
    }
  };
  if (warp == kProducerWarp && lens_w) {
    prefix(false);
    init_cursor();
    first_chunk();
  }

  griddep_wait();
  // The next kernel on the stream may start launching now: its CTAs take SMs
  // as these exit, and it waits for this grid before it reads memory.
  griddep_launch_dependents();

  int ids_raw = 0;
  if (a.mode == kModeBalanced) {
    // the consumers wait on a named barrier that the producer passes without
    // waiting
    if (warp == kProducerWarp) {
      bool same = false;
      if (lens_w) {
        ids_raw = have_c ? load_id_raw(a, c_s, c_jb, c_n, lane) : 0;
        same = true;
        for (int s = sl0; s < sl1; ++s) {
          const int len = load_len(a, s, true);
          const int nb = (len + kBlockSize - 1) / kBlockSize - start_block(a, s, len, true);
          same = same && len == lens_w[s] && nb == pre[s + 1] - pre[s];
        }
        same = __all_sync(0xffffffffu, same);
      }
      if (!same) {
        prefix(true);
        init_cursor();
        first_chunk();
        ids_raw = have_c ? load_id_raw(a, c_s, c_jb, c_n, lane) : 0;
      }
      asm volatile("bar.arrive 2, %0;" ::"n"(kThreads) : "memory");
    } else {
      asm volatile("bar.sync 2, %0;" ::"n"(kThreads) : "memory");
      init_cursor();
    }
  } else {
    cur.u = cta;
    cur.step = ncta;
    cur.U = static_cast<long long>(a.num_seqs) * a.max_parts;
  }

  if (warp == kProducerWarp) {
    // ------------------------------------------------------------ producer
    // a stalled test launch issues nothing: every consumer wait runs out
    // with no copy in flight
    if (a.stall_loads) return;
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    const uint64_t pol = l2_policy_evict_first();
    const uint32_t qrow_bytes = static_cast<uint32_t>(Hq) * D * 2;
    bool ok = true;
    // query rows of the piece's sequence into query slot qi & 1 (lane 0)
    auto stage_q = [&](const Piece& pp, int qi) {
      if (lane != 0 || !ok) return;
      const int k = qi & 1;
      if (qi >= 2 && !mbar_wait(bar_qempty + k * 8, ((qi >> 1) - 1) & 1, a.wait_ns)) {
        atomicOr(a.err, PA_DEVERR_TIMEOUT);
        ok = false;
        return;
      }
      // one copy per kv head's rows (G x D, at most 2 KB) on the same
      // barrier: a single copy of the whole row set (16 KB at 64 q heads)
      // into this two-slot ring gave nondeterministic query rows when pieces
      // were one block long; per-head copies do not
      mbar_arrive_expect_tx(bar_qfull + k * 8, qrow_bytes);
      const uint32_t chunk = static_cast<uint32_t>(G) * D * 2;
      for (int h = 0; h < Hkv; ++h)
        bulk_load(sbase + L.q_off + k * L.q_bytes + h * chunk,
                  a.q + static_cast<long long>(pp.s) * Hq * D + h * G * D, chunk,
                  bar_qfull + k * 8);
    };
    int qi = 0;
    if (a.mode != kModeBalanced) {
      have_p = next_piece(a, pre, lens_c, cur, p, false);
      jbp = have_p ? p.j0 : 0;
    }
    if (have_p) stage_q(p, qi++);
    // next chunk of up to 32 blocks, staging the queries of every piece reached
    auto next_chunk2 = [&](int& s, int& jb, int& n) -> bool {
      while (have_p) {
        if (jbp < p.j1) {
          s = p.s;
          jb = jbp;
          n = min(32, p.j1 - jbp);
          jbp += n;
          return true;
        }
        have_p = next_piece(a, pre, lens_c, cur, p, false);
        if (!have_p) return false;
        stage_q(p, qi++);
        jbp = p.j0;
      }
      return false;
    };
    int s, jb, n, ids;
    bool have;
    if (a.mode == kModeBalanced) {
      have = have_c;
      s = c_s;
      jb = c_jb;
      n = c_n;
      ids = have ? check_id(a, ids_raw, n, lane) : 0;
    } else {
      have = next_chunk2(s, jb, n);
      ids = have ? load_ids(a, s, jb, n, lane) : 0;
    }
    uint32_t g = 0;
    ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
    while (have && ok) {
      // the next chunk (its table row, and the queries of a new piece) is
      // prepared once the current chunk's first ring's worth of blocks is
      // issued, so the first loads of a launch go out without waiting on it
      int s2 = 0, jb2 = 0, n2 = 0, ids2 = 0;
      bool have2 = false, got2 = false;
      for (int i = 0; i < n && ok; ++i, ++g) {
        const int blk = __shfl_sync(0xffffffffu, ids, i);
        const uint32_t st = g % NS;
        const uint32_t fb = bar_full + st * 8;
        if (lane == 0) {
          if (g >= static_cast<uint32_t>(NS) &&
              !mbar_wait(bar_empty + st * 8, ((g / NS) - 1) & 1, a.wait_ns)) {
            atomicOr(a.err, PA_DEVERR_TIMEOUT);
            ok = false;
          } else {
            mbar_arrive_expect_tx(fb, L.stage_bytes);
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
        // one box per 64-column half and pool (16 tokens x every kv head of
        // the block), each issued by its own lane: the TMA unit takes boxes
        // from several threads at once, one thread's boxes one after another
        constexpr int kBoxes = KV8 ? 2 : 2 * (D / 64);
        if (lane < kBoxes) {
          const uint32_t kdst = sbase + st * L.stage_bytes;
          const uint32_t vdst = kdst + Hkv * L.head_bytes;
          const int y = blk * kBlockSize;
          const bool is_v = lane & 1;
          const int h = lane >> 1;  // 64-column half (E4M3: the whole 128-byte row)
          tma_load_3d((is_v ? vdst : kdst) + (KV8 ? 0 : h * Hkv * kBoxBytes), is_v ? &tm_v : &tm_k,
                      KV8 ? 0 : h * 64, y, 0, fb, pol);
        }
        if (!got2 && (i + 1 == n || i + 1 == NS)) {
          have2 = next_chunk2(s2, jb2, n2);
          ids2 = have2 ? load_ids(a, s2, jb2, n2, lane) : 0;
          got2 = true;
          ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        }
      }
      if (!got2) break;  // stopped early (a failed wait): nothing more is issued
      s = s2;
      jb = jb2;
      n = n2;
      ids = ids2;
      have = have2;
    }
    // queries of pieces without blocks (empty sequences) still get staged
    while (ok && have_p) {
      have_p = next_piece(a, pre, lens_c, cur, p, false);
      if (have_p) stage_q(p, qi++);
    }
    if (!ok) *reinterpret_cast<volatile int*>(misc) = 1;
    return;
  }

  if (warp == kMergeWarp) {
    // -------------------------------------------------------------- merge warp
    // Balanced split: a partial piece that is not the last of the CTA's walk
    // is handed over here once the consumers have published it (hand-off k
    // on barrier k, with the sequence, its first CTA and its piece count in
    // shared memory), so that they go on streaming the next piece while this
    // warp takes the sequence's ticket (an L2 round trip).  A ticket taken by
    // the consumers themselves stalled the stream: decode CTAs of two pieces
    // streamed 8 % slower than those of one.  If the ticket is the last one,
    // the merge is left pending for the consumers, who make it with the same
    // code as every other merge (bitwise the same result) once their stream
    // has ended.  A record with no pieces ends the hand-offs.  If a wait runs
    // out, the remaining records go back to the consumers (state 2: "take
    // the ticket yourselves"), so every published piece draws one ticket.
    if (a.mode == kModeBalanced) {
      for (int k = 0; k < kHandOffs; ++k) {
        if (!mbar_wait_warp(bar_hand + k * 8, 0, a.wait_ns)) {
          if (lane == 0) {
            atomicOr(a.err, PA_DEVERR_TIMEOUT);
            for (int j = k; j < kHandOffs; ++j) {
              misc[7 + 4 * j] = 2;
              mbar_arrive(bar_tdone + j * 8);
            }
          }
          __syncwarp();
          break;
        }
        volatile int* rec = misc + 4 + 4 * k;
        if (rec[2] == 0) break;
        if (lane == 0) {
          const int t = atom_add_acq_rel_gpu(a.counters + rec[1], 1);
          rec[3] = t == rec[2] - 1 ? 1 : 0;  // pending merge
          mbar_arrive(bar_tdone + k * 8);
        }
        __syncwarp();
      }
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  const int ctid = tid;  // 0..255
  if (a.mode == kModeBalanced) {
    // sequences without tokens to attend produce out = 0, lse = -inf -- or,
    // in a cascade suffix pass, the prefix pass's result
    for (int s = cta; s < a.num_seqs; s += ncta) {
      const int len = load_len(a, s, warp == 0);
      if ((len + kBlockSize - 1) / kBlockSize - start_block(a, s, len, warp == 0) != 0) continue;
      const long long base = static_cast<long long>(s) * Hq;
      for (int e = ctid; e < Hq * D; e += kConsumerThreads)
        a.out[base * D + e] = __float2bfloat16(a.init_o ? a.init_o[base * D + e] : 0.f);
      if (a.out_lse)
        for (int h = ctid; h < Hq; h += kConsumerThreads)
          a.out_lse[base + h] = a.init_o ? a.init_lse[base + h] : -INFINITY;
    }
  }

  const bool active = warp < active_warps;
  const int hw = warp % Hkv;   // this warp's kv head
  const float vsc = KV8 && active ? a.v_scales[hw] : 1.f;  // E4M3: V dequantization scale
  const int sub = warp / Hkv;  // which of the head's warps
  const int q4 = lane & 3;
  const int d0 = lane >> 2;
  const int hq = lane >> 2;
  volatile int* abort_flag = misc;
  Piece pc;
  uint32_t g = 0;
  int qi = 0;
  int hand = 0;  // partial pieces handed to the merge warp so far
  // the report flag is uniform over a warp: lanes of one warp must take the
  // same path here, or the warp-synchronous MMA and matrix loads below could
  // be reached at different instructions
  while (next_piece(a, pre, lens_c, cur, pc, warp == 0)) {
    __syncwarp();
    const long long head0 = static_cast<long long>(pc.s) * Hq + hw * G;
    uint32_t qf[KS][2];
    float sl2 = a.scale_log2;  // scores to log2 units (E4M3: scales folded in)
    if (active) {
      // query fragments of the group (B operand: k = dim, n = head) from the
      // piece's staged query rows
      const int k = qi & 1;
      if (!warp_flag(abort_flag) && !mbar_wait_warp(bar_qfull + k * 8, (qi >> 1) & 1, a.wait_ns)) {
        if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
      }
      const uint32_t qrow = sbase + L.q_off + k * L.q_bytes + (hw * G + hq) * D * 2;
      if constexpr (KV8) {
        // f16 fragments in the permuted dim order of attend_block_fp8:
        // k-step ks takes dims 32c + 4ks + {0,1} and {2,3}.  The group's
        // queries are scaled by one power of two 2^e that puts their largest
        // magnitude in [2^14, 2^15): exact in fp32, no f16 overflow; 2^-e and
        // the K scale go into sl2.
        uint32_t w[KS][2];
        float mx = 0.f;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          uint32_t x0 = 0u, x1 = 0u;
          if (hq < G)
            asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];"
                         : "=r"(x0), "=r"(x1)
                         : "r"(qrow + (32 * q4 + 4 * ks) * 2));
          w[ks][0] = x0;
          w[ks][1] = x1;
          mx = fmaxf(mx, fmaxf(fmaxf(fabsf(__uint_as_float(x0 << 16)),
                                     fabsf(__uint_as_float(x0 & 0xffff0000u))),
                               fmaxf(fabsf(__uint_as_float(x1 << 16)),
                                     fabsf(__uint_as_float(x1 & 0xffff0000u)))));
        }
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, off));
        int ex = 0;
        if (mx > 0.f && isfinite(mx)) frexpf(mx, &ex);  // mx < 2^ex
        const int e = ex == 0 ? 0 : min(126, max(-126, 15 - ex));
        const float p2 = ldexpf(1.f, e);
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          qf[ks][0] = pack_f16x2(__uint_as_float(w[ks][0] << 16) * p2,
                                 __uint_as_float(w[ks][0] & 0xffff0000u) * p2);
          qf[ks][1] = pack_f16x2(__uint_as_float(w[ks][1] << 16) * p2,
                                 __uint_as_float(w[ks][1] & 0xffff0000u) * p2);
        }
        sl2 = a.scale_log2 * a.k_scales[hw] * ldexpf(1.f, -e);
      } else {
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) {
          const uint32_t c = (ks * 16 + q4 * 2) * 2;
          uint32_t x0 = 0u, x1 = 0u;
          if (hq < G) {
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(x0) : "r"(qrow + c));
            asm volatile("ld.shared.b32 %0, [%1];" : "=r"(x1) : "r"(qrow + c + 16));
          }
          qf[ks][0] = x0;
          qf[ks][1] = x1;
        }
      }
      // The slot is released below and the next bulk copy (async proxy) may
      // overwrite it at once.  Every loaded value goes into one word stored
      // to this warp's scratch slot -- an instruction that cannot issue
      // before all the loads have returned -- then a proxy fence orders the
      // reads before the copy that the release lets the producer issue.
      {
        uint32_t dep = 0u;
#pragma unroll
        for (int ks = 0; ks < KS; ++ks) dep ^= qf[ks][0] ^ qf[ks][1];
        asm volatile("st.shared.u32 [%0], %1;" ::"r"(smem_u32(misc + 16 + warp)), "r"(dep)
                     : "memory");
        fence_proxy_async_smem();
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_qempty + k * 8);
    }
    ++qi;
    float o[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;
    if (a.init_o && pc.first && active && sub == 0) {
      // cascade suffix pass: the sequence's first piece starts from the prefix
      // pass's result: accumulator o_pre (before the V scale), running max
      // lse in log2 units, running sum 1 (held by one lane of the 8 that
      // share a head column; the sums are reduced across them at the end)
      const float l2e = 1.4426950408889634f;
      const float inv_v = 1.f / vsc;
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int hk = 2 * q4 + k;
        if (hk >= G) continue;
        const long long row = head0 + hk;
        const float lse = a.init_lse[row];
        if (!(lse > -INFINITY)) continue;
        if (k == 0) {
          m0 = lse * l2e;
          l0 = d0 == 0 ? 1.f : 0.f;
        } else {
          m1 = lse * l2e;
          l1 = d0 == 0 ? 1.f : 0.f;
        }
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          o[mt][k] = a.init_o[row * D + out_dim<KV8>(mt, d0, 0)] * inv_v;
          o[mt][2 + k] = a.init_o[row * D + out_dim<KV8>(mt, d0, 1)] * inv_v;
        }
      }
    }

    // Append: the warp that will attend the sequence's last block tb fetches
    // its kv head's row of the new token (and the block's id) into its
    // shared-memory slot now, asynchronously; when block tb has landed it
    // writes the row over position seq_len-1 of the stage -- so the token is
    // attended whatever the pool held there -- and into the pool's slot.
    int tail_j = -1;  // the sequence's last block, when this warp attends it
    if constexpr (AP) {
      const int tb = (pc.len - 1) / kBlockSize;
      const uint32_t nbuf = sbase + L.nk_off + warp * new_row_bytes(D);
      if (active && pc.len > 0 && tb >= pc.j0 && tb < pc.j1 &&
          static_cast<int>((g + static_cast<uint32_t>(tb - pc.j0)) % wph) == sub) {
        tail_j = tb;
        if (lane < D / 4) {  // K chunks, then V chunks, of 16 bytes
          const bool isv = lane >= D / 8;
          const int ch = lane % (D / 8);
          const __nv_bfloat16* src =
              (isv ? a.new_v + pc.s * a.new_v_stride : a.new_k + pc.s * a.new_k_stride) +
              hw * D + ch * 8;
          cp_async_16(nbuf + (isv ? 2 * D : 0) + ch * 16, src);
        }
        if (lane == 0)
          cp_async_4(nbuf + 4 * D, a.block_tables + static_cast<long long>(pc.s) * a.max_blocks + tb);
      }
    }
    auto patch_tail = [&](uint32_t stg) {
      const uint32_t nbuf = sbase + L.nk_off + warp * new_row_bytes(D);
      cp_async_wait_all();
      __syncwarp();
      const int t = (pc.len - 1) & (kBlockSize - 1);
      if (lane < D / 4) {
        const bool isv = lane >= D / 8;
        const int ch = lane % (D / 8);
        const uint4 v = lds128(nbuf + (isv ? 2 * D : 0) + ch * 16);
        const uint32_t base =
            sbase + stg * L.stage_bytes + hw * kBoxBytes + (isv ? Hkv * L.head_bytes : 0);
        sts128(swz(base, t, ch, Hkv * kBoxBytes), v);
        int id;
        asm volatile("ld.shared.u32 %0, [%1];" : "=r"(id) : "r"(nbuf + 4 * D) : "memory");
        if (id >= 0 && id < a.num_blocks)
          *reinterpret_cast<uint4*>((isv ? a.v_pool : a.k_pool) +
                                    (static_cast<long long>(id) * kBlockSize + t) * Hkv * D +
                                    hw * D + ch * 8) = v;
      }
      // the stage is refilled by TMA (async proxy) once released
      fence_proxy_async_smem();
      __syncwarp();
    };

    if (active) {
      for (int j = pc.j0; j < pc.j1; ++j, ++g) {
        if (static_cast<int>(g % wph) != sub) continue;
        if (warp_flag(abort_flag)) continue;
        const uint32_t st = g % NS;
        if (!mbar_wait_warp(bar_full + st * 8, (g / NS) & 1, a.wait_ns)) {
          if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
          *abort_flag = 1;
          continue;
        }
        if constexpr (AP)
          if (j == tail_j) patch_tail(st);
        const int valid = min(kBlockSize, pc.len - j * kBlockSize);
        if (!AP && wph == 1 && NS >= 4 && j + 1 < pc.j1) {
          // the piece's next block too (this warp holds every block of its kv
          // head): both in one step.  The first one is full, since the piece
          // goes on past it.  Only with a ring of four stages or more (the
          // E4M3 pools' six): holding two of three stages starves the
          // producer (measured 48.8 -> 51.9 us on the Llama-3-8B layer).
          const uint32_t st2 = (g + 1) % NS;
          if (!mbar_wait_warp(bar_full + st2 * 8, ((g + 1) / NS) & 1, a.wait_ns)) {
            if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
            *abort_flag = 1;
            __syncwarp();
            if (lane == 0) mbar_arrive(bar_empty + st * 8);
            continue;
          }

          const int valid2 = min(kBlockSize, pc.len - (j + 1) * kBlockSize);
          if constexpr (KV8) {
            const uint32_t kb = sbase + st * L.stage_bytes + hw * L.head_bytes;
            const uint32_t kb2 = sbase + st2 * L.stage_bytes + hw * L.head_bytes;
            attend_pair_fp8<D>(kb, kb + Hkv * L.head_bytes, kb2, kb2 + Hkv * L.head_bytes, qf, o,
                               m0, m1, l0, l1, valid2, sl2, lane);
          } else {
            const uint32_t kb = sbase + st * L.stage_bytes + hw * kBoxBytes;
            const uint32_t kb2 = sbase + st2 * L.stage_bytes + hw * kBoxBytes;
            attend_pair<D>(kb, kb + Hkv * L.head_bytes, kb2, kb2 + Hkv * L.head_bytes,
                           Hkv * kBoxBytes, qf, o, m0, m1, l0, l1, valid2, a.scale_log2, lane);
          }
          __syncwarp();
          if (lane == 0) {
            mbar_arrive(bar_empty + st * 8);
            mbar_arrive(bar_empty + st2 * 8);
          }
          ++j;
          ++g;
          continue;
        }
        if constexpr (KV8) {
          const uint32_t kb = sbase + st * L.stage_bytes + hw * L.head_bytes;
          attend_block_fp8<D>(kb, kb + Hkv * L.head_bytes, qf, o, m0, m1, l0, l1, valid, sl2,
                              lane);
        } else {
          const uint32_t kb = sbase + st * L.stage_bytes + hw * kBoxBytes;
          attend_block<D>(kb, kb + Hkv * L.head_bytes, Hkv * kBoxBytes, qf, o, m0, m1, l0, l1,
                          valid, a.scale_log2, lane);
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_empty + st * 8);
      }
    } else {
      g += pc.j1 - pc.j0;
    }
    if constexpr (AP)
      if (tail_j >= 0) cp_async_wait_all();  // no copy left in flight (an aborted walk skips blocks)

    // ---- per-head result of this piece: normalized o and lse (log2 units)
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    float fa, fb, lsea, lseb;
    if (wph > 1) {
      // several warps share the head: merge their (m, l, O) through smem
      if (active && lane < 4) {
        mlbuf[(warp * kMaxGroup + 2 * q4) * 2 + 0] = m0;
        mlbuf[(warp * kMaxGroup + 2 * q4) * 2 + 1] = l0;
        mlbuf[(warp * kMaxGroup + 2 * q4 + 1) * 2 + 0] = m1;
        mlbuf[(warp * kMaxGroup + 2 * q4 + 1) * 2 + 1] = l1;
      }
      named_barrier(1, kConsumerThreads);
      float f[2], ls[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int h = 2 * q4 + k;
        float M = -INFINITY;
        for (int w2 = 0; w2 < wph; ++w2)
          M = fmaxf(M, mlbuf[((w2 * Hkv + hw) * kMaxGroup + h) * 2]);
        float Ls = 0.f;
        if (M != -INFINITY)
          for (int w2 = 0; w2 < wph; ++w2)
            Ls += mlbuf[((w2 * Hkv + hw) * kMaxGroup + h) * 2 + 1] *
                  fast_exp2(mlbuf[((w2 * Hkv + hw) * kMaxGroup + h) * 2] - M);
        const float mine = k == 0 ? m0 : m1;
        f[k] = Ls > 0.f ? fast_exp2(mine - M) / Ls : 0.f;
        ls[k] = Ls > 0.f ? (M + __log2f(Ls)) * kLn2 : -INFINITY;
      }
      fa = f[0];
      fb = f[1];
      if constexpr (KV8) {
        fa *= vsc;
        fb *= vsc;
      }
      lsea = ls[0];
      lseb = ls[1];
      if (active) {
        float* ob = obuf + warp * kMaxGroup * (D + 4);
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d = out_dim<KV8>(mt, d0, 0), d8 = out_dim<KV8>(mt, d0, 1);
          ob[(2 * q4) * (D + 4) + d] = o[mt][0] * fa;
          ob[(2 * q4 + 1) * (D + 4) + d] = o[mt][1] * fb;
          ob[(2 * q4) * (D + 4) + d8] = o[mt][2] * fa;
          ob[(2 * q4 + 1) * (D + 4) + d8] = o[mt][3] * fb;
        }
      }
      named_barrier(1, kConsumerThreads);
      // the head's first warp sums its partners' contributions into registers
      if (active && sub == 0) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d = out_dim<KV8>(mt, d0, 0), d8 = out_dim<KV8>(mt, d0, 1);
          float s0 = 0.f, s1 = 0.f, s2 = 0.f, s3 = 0.f;
          for (int w2 = 0; w2 < wph; ++w2) {
            const float* ob = obuf + (w2 * Hkv + hw) * kMaxGroup * (D + 4);
            s0 += ob[(2 * q4) * (D + 4) + d];
            s1 += ob[(2 * q4 + 1) * (D + 4) + d];
            s2 += ob[(2 * q4) * (D + 4) + d8];
            s3 += ob[(2 * q4 + 1) * (D + 4) + d8];
          }
          o[mt][0] = s0;
          o[mt][1] = s1;
          o[mt][2] = s2;
          o[mt][3] = s3;
        }
      }
      named_barrier(1, kConsumerThreads);
    } else {
      fa = l0 > 0.f ? 1.f / l0 : 0.f;
      fb = l1 > 0.f ? 1.f / l1 : 0.f;
      if constexpr (KV8) {
        fa *= vsc;
        fb *= vsc;
      }
      lsea = l0 > 0.f ? (m0 + __log2f(l0)) * kLn2 : -INFINITY;
      lseb = l1 > 0.f ? (m1 + __log2f(l1)) * kLn2 : -INFINITY;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        o[mt][0] *= fa;
        o[mt][1] *= fb;
        o[mt][2] *= fa;
        o[mt][3] *= fb;
      }
    }
    // lanes own o^T[out_dim(mt, d0, 0 / 1)][head 2*q4 (+1)] of kv head hw
    const bool writer = active && sub == 0;
    const int ha = 2 * q4, hb = 2 * q4 + 1;
    if (pc.kind == kFinal) {
      if constexpr (KV8) {
        if (writer) {
          // E4M3 layout: the lane holds dims [16 d0, 16 d0 + 16) of both heads,
          // stored as two 16-byte pieces each
          if (ha < G) {
            uint4* dst = reinterpret_cast<uint4*>(a.out + (head0 + ha) * D + 16 * d0);
            dst[0] = make_uint4(pack_bf16x2(o[0][0], o[0][2]), pack_bf16x2(o[1][0], o[1][2]),
                                pack_bf16x2(o[2][0], o[2][2]), pack_bf16x2(o[3][0], o[3][2]));
            dst[1] = make_uint4(pack_bf16x2(o[4][0], o[4][2]), pack_bf16x2(o[5][0], o[5][2]),
                                pack_bf16x2(o[6][0], o[6][2]), pack_bf16x2(o[7][0], o[7][2]));
          }
          if (hb < G) {
            uint4* dst = reinterpret_cast<uint4*>(a.out + (head0 + hb) * D + 16 * d0);
            dst[0] = make_uint4(pack_bf16x2(o[0][1], o[0][3]), pack_bf16x2(o[1][1], o[1][3]),
                                pack_bf16x2(o[2][1], o[2][3]), pack_bf16x2(o[3][1], o[3][3]));
            dst[1] = make_uint4(pack_bf16x2(o[4][1], o[4][3]), pack_bf16x2(o[5][1], o[5][3]),
                                pack_bf16x2(o[6][1], o[6][3]), pack_bf16x2(o[7][1], o[7][3]));
          }
          if (a.out_lse && d0 == 0) {
            if (ha < G) a.out_lse[head0 + ha] = lsea;
            if (hb < G) a.out_lse[head0 + hb] = lseb;
          }
        }
      } else if (writer) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d = out_dim<KV8>(mt, d0, 0), d8 = out_dim<KV8>(mt, d0, 1);
          if (ha < G) {
            a.out[(head0 + ha) * D + d] = __float2bfloat16(o[mt][0]);
            a.out[(head0 + ha) * D + d8] = __float2bfloat16(o[mt][2]);
          }
          if (hb < G) {
            a.out[(head0 + hb) * D + d] = __float2bfloat16(o[mt][1]);
            a.out[(head0 + hb) * D + d8] = __float2bfloat16(o[mt][3]);
          }
        }
        if (a.out_lse && d0 == 0) {
          if (ha < G) a.out_lse[head0 + ha] = lsea;
          if (hb < G) a.out_lse[head0 + hb] = lseb;
        }
      }
    } else if (pc.kind == kPartialFixed) {
      if (writer) {
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d = out_dim<KV8>(mt, d0, 0), d8 = out_dim<KV8>(mt, d0, 1);
          if (ha < G) {
            const long long row = (head0 + ha) * a.max_parts + pc.part;
            a.part_o[row * D + d] = o[mt][0];
            a.part_o[row * D + d8] = o[mt][2];
            if (mt == 0 && d0 == 0) a.part_lse[row] = lsea;
          }
          if (hb < G) {
            const long long row = (head0 + hb) * a.max_parts + pc.part;
            a.part_o[row * D + d] = o[mt][1];
            a.part_o[row * D + d8] = o[mt][3];
            if (mt == 0 && d0 == 0) a.part_lse[row] = lseb;
          }
        }
      }
    } else {
      // balanced partial: publish to this CTA's slot [Hq][D] + lse[Hq]
      float* slot = a.part_o + (static_cast<long long>(cta) * 2 + pc.which) * a.slot_floats;
      if constexpr (KV8) {
        if (writer) {
          // E4M3 layout: dims [16 d0, 16 d0 + 16) of both heads, as four
          // 16-byte pieces each (scattered 4-byte stores cost the L1 one
          // transaction per lane)
          const int hga = hw * G + ha, hgb = hw * G + hb;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            if (ha < G)
              *reinterpret_cast<float4*>(slot + hga * D + 16 * d0 + 4 * i) =
                  make_float4(o[2 * i][0], o[2 * i][2], o[2 * i + 1][0], o[2 * i + 1][2]);
            if (hb < G)
              *reinterpret_cast<float4*>(slot + hgb * D + 16 * d0 + 4 * i) =
                  make_float4(o[2 * i][1], o[2 * i][3], o[2 * i + 1][1], o[2 * i + 1][3]);
          }
          if (d0 == 0) {
            if (ha < G) slot[Hq * D + hga] = lsea;
            if (hb < G) slot[Hq * D + hgb] = lseb;
          }
        }
      } else if (writer) {
        const int hga = hw * G + ha, hgb = hw * G + hb;
#pragma unroll
        for (int mt = 0; mt < KS; ++mt) {
          const int d = out_dim<KV8>(mt, d0, 0), d8 = out_dim<KV8>(mt, d0, 1);
          if (ha < G) {
            slot[hga * D + d] = o[mt][0];
            slot[hga * D + d8] = o[mt][2];
          }
          if (hb < G) {
            slot[hgb * D + d] = o[mt][1];
            slot[hgb * D + d8] = o[mt][3];
          }
        }
        if (d0 == 0) {
          if (ha < G) slot[Hq * D + hga] = lsea;
          if (hb < G) slot[Hq * D + hgb] = lseb;
        }
      }
      const long long c0 = pc.seg_start + static_cast<long long>(cur.beta) * (pc.s + 1);
      const long long cf = owner_of_cost(c0, cur.T, cur.C);
      const int np = static_cast<int>(owner_of_cost(c0 + pc.nb - 1, cur.T, cur.C) - cf + 1);
      // a piece before the walk's last: hand it to the merge warp (each
      // warp's slot stores, ordered by __syncwarp, are released by its
      // arrival) and go on with the next piece
      if (hand < kHandOffs && (cur.idx < cur.end || (cur.phase == 0 && cur.lo < cur.mid))) {
        if (ctid == 0) {
          misc[4 + 4 * hand] = pc.s;
          misc[5 + 4 * hand] = static_cast<int>(cf);
          misc[6 + 4 * hand] = np;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(bar_hand + hand * 8);
        ++hand;
        continue;
      }
      // the walk's last piece: take the sequence's ticket (release of the
      // slot stores above); the last of its pieces to draw one merges them
      // all, right after the walk (below)
      named_barrier(1, kConsumerThreads);
      if (ctid == 0) {
        const int t = atom_add_acq_rel_gpu(a.counters + cf, 1);
        int* rec = misc + 4 + 4 * kHandOffs;
        rec[0] = pc.s;
        rec[1] = static_cast<int>(cf);
        rec[2] = np;
        rec[3] = t == np - 1 ? 1 : 0;
      }
    }
  }
  if (a.mode == kModeBalanced) {
    // no more hand-offs: a record without pieces lets the merge warp exit
    if (hand < kHandOffs) {
      if (ctid == 0) misc[6 + 4 * hand] = 0;
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_hand + hand * 8);
    }
    // the merges whose last ticket this CTA drew: those of the merge warp's
    // hand-offs, then the walk's last piece's (one merge site, so every
    // merge rounds the same way)
    named_barrier(1, kConsumerThreads);  // record kHandOffs (ctid 0's) is visible
    for (int k = 0; k <= kHandOffs; ++k) {
      const volatile int* rec = misc + 4 + 4 * k;
      // the record's state, read by every consumer thread between named
      // barriers, so that all of them take the same branches below
      int st;
      if (k < kHandOffs) {
        if (k >= hand) continue;  // hand is the same in every consumer thread
        // one thread waits for the merge warp's answer and shares it
        if (ctid == 0) {
          const bool ok = mbar_wait(bar_tdone + k * 8, 0, a.wait_ns);
          if (!ok) atomicOr(a.err, PA_DEVERR_TIMEOUT);
          misc[2] = ok ? rec[3] : 0;
        }
        named_barrier(1, kConsumerThreads);
        st = misc[2];
      } else {
        st = rec[3];  // ctid 0's, before the barrier above the loop
      }
      named_barrier(1, kConsumerThreads);  // read before misc[2] changes again
      if (st == 2) {  // the merge warp gave up before this hand-off's ticket
        if (ctid == 0) misc[2] = atom_add_acq_rel_gpu(a.counters + rec[1], 1) == rec[2] - 1 ? 1 : 0;
        named_barrier(1, kConsumerThreads);
        st = misc[2];
        named_barrier(1, kConsumerThreads);
      }
      if (st == 1) {
        merge_pieces<D, kConsumerThreads>(a, rec[0], rec[1], rec[2], ctid);
        named_barrier(1, kConsumerThreads);
        if (ctid == 0) a.counters[rec[1]] = 0;
      }
    }
  }
}

inline int warps_per_head(int Hkv) { return Hkv >= kConsumerWarps ? 1 : kConsumerWarps / Hkv; }

inline int pick_stages(int D, int Hkv, int Hq, int pre_ints, int elem_bytes, bool append) {
  const int wph = warps_per_head(Hkv);
  const int budget = 227 * 1024 - 1024;  // minus alignment slack
  int st = kMaxStages;
  while (st > 2 && make_layout(D, Hkv, Hq, wph, st, pre_ints, elem_bytes, append).total > budget)
    --st;
  return st;
}

}  // namespace
}  // namespace dec
}  // namespace pa
