// pa_decode.cu -- paged decode attention for sm_103a.
//
// One query per sequence attends over its paged KV ("03 - Engines Papers",
// section 2 PagedAttention: the kernel gathers K/V from non-contiguous
// 16-token blocks named by the block table).  Design:
//
//  * Persistent CTAs, one per SM: 4 consumer warps + 1 producer warp.
//  * The producer walks the CTA's work (a list of block ranges of
//    (sequence, kv head) segments), prefetches block-table rows 32 entries at
//    a time, and streams each 16-token block of one kv head into a ring of
//    shared-memory stages with TMA tensor loads (two 64-column boxes per
//    row of 128 bf16, 128-byte swizzled), signalling an mbarrier per stage.
//  * Consumer warp w takes every 4th stage.  GQA: the group's q heads are the
//    N=8 columns of a warp MMA, so each K/V byte loaded is used by every q
//    head of its group: S^T[16 tokens x 8 heads] = K[16 x D] Q^T[D x 8]
//    (mma.m16n8k16, bf16 in, fp32 accumulate), online softmax over the
//    block's 16 scores per head with warp-shuffle max reductions (Milakov &
//    Gimelshein recurrence, "References" page), then O^T[D x 8] += V^T P^T.
//  * At the end of a segment piece the 4 warps' running (m, l, O) are merged
//    through shared memory and the result is written: final bf16 output, a
//    fixed-partition partial for the LSE merge kernel, or (balanced mode) a
//    partial that the last-arriving CTA of that segment merges in place by
//    log-sum-exp ("03 - Engines Papers", section 12 Cascade Inference;
//    split-K reduction of "The LLM inference engine playbook", Theme 4).
//
// No wait is unbounded: every mbarrier spin gives up after kWaitLimit tries,
// sets PA_DEVERR_TIMEOUT and stops the CTA's work.
#include <math.h>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kConsumerWarps = 4;
constexpr int kThreads = (kConsumerWarps + 1) * 32;
constexpr int kBoxBytes = 16 * 128;  // one TMA box: 16 token rows x 64 bf16
constexpr float kLn2 = 0.6931471805599453f;

template <int D>
struct Cfg {
  static constexpr int kStages = D == 128 ? 16 : 24;
  static constexpr int kHalves = D / 64;
  static constexpr int kKBytes = kHalves * kBoxBytes;  // K of one block, one kv head
  static constexpr int kStageBytes = 2 * kKBytes;      // K + V
  static constexpr int kObufStride = D + 4;            // padded head row (bank spread)
  static constexpr int kObufFloats = kConsumerWarps * kMaxGroup * kObufStride;
  static constexpr int kStageOff = 0;
  static constexpr int kObufOff = kStages * kStageBytes;
  static constexpr int kMlOff = kObufOff + kObufFloats * 4;
  static constexpr int kLseOff = kMlOff + kConsumerWarps * kMaxGroup * 2 * 4;
  static constexpr int kBarOff = kLseOff + kMaxGroup * 2 * 4;
  static constexpr int kMiscOff = kBarOff + kStages * 2 * 8;
  static constexpr int kPreOff = kMiscOff + 64;
};

enum PieceKind : int { kFinal = 0, kPartialFixed = 1, kPartialBalanced = 2 };

struct Piece {
  int s, kvh, j0, j1, len, nb, kind, part, which;
  long long seg_start;
};

struct Cursor {
  long long u, U;          // fixed / single-pass unit walk
  long long idx, lo, hi;   // balanced block range [lo, hi)
  long long W;             // balanced: total blocks
  int C;                   // balanced: CTAs that own a non-empty range
};

__device__ __forceinline__ int load_len(const DecodeArgs& a, int s, bool report) {
  int len = a.seq_lens[s];
  const int cap = a.max_blocks * kBlockSize;
  if (len < 0 || len > cap) {
    if (report) atomicOr(a.err, PA_DEVERR_SEQ_LEN);
    len = len < 0 ? 0 : cap;
  }
  return len;
}

__device__ __forceinline__ long long cta_of(long long x, long long W, int C) {
  // owner of global block x when CTA c owns [c*W/C, (c+1)*W/C)
  return ((x + 1) * C + W - 1) / W - 1;
}

__device__ bool next_piece(const DecodeArgs& a, const int* pre, Cursor& c, Piece& p,
                           bool report) {
  if (a.mode == kModeBalanced) {
    if (c.idx >= c.hi) return false;
    const long long Hkv = a.num_kv_heads;
    int lo = 0, hi = a.num_seqs - 1;  // largest s with Hkv*pre[s] <= idx
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (Hkv * pre[mid] <= c.idx) lo = mid; else hi = mid - 1;
    }
    const int s = lo;
    const int nb = pre[s + 1] - pre[s];
    const long long base = Hkv * pre[s];
    const long long r = c.idx - base;
    p.s = s;
    p.nb = nb;
    p.kvh = static_cast<int>(r / nb);
    p.j0 = static_cast<int>(r % nb);
    p.seg_start = base + static_cast<long long>(p.kvh) * nb;
    const long long seg_end = p.seg_start + nb;
    const long long end = c.hi < seg_end ? c.hi : seg_end;
    p.j1 = p.j0 + static_cast<int>(end - c.idx);
    c.idx = end;
    p.len = load_len(a, s, false);
    p.kind = (p.j0 == 0 && p.j1 == nb) ? kFinal : kPartialBalanced;
    p.which = p.seg_start < c.lo ? 0 : 1;
    p.part = 0;
    return true;
  }
  while (c.u < c.U) {
    const long long u = c.u;
    c.u += gridDim.x;
    const int kvh = static_cast<int>(u % a.num_kv_heads);
    const long long t = u / a.num_kv_heads;
    const int part = static_cast<int>(t % a.max_parts);
    const int s = static_cast<int>(t / a.max_parts);
    const int len = load_len(a, s, report && part == 0 && kvh == 0);
    const int nb = (len + kBlockSize - 1) / kBlockSize;
    const int nparts = nb == 0 ? 1 : (nb + a.part_blocks - 1) / a.part_blocks;
    if (part >= nparts) continue;
    p.s = s;
    p.kvh = kvh;
    p.len = len;
    p.nb = nb;
    p.j0 = part * a.part_blocks;
    p.j1 = min(nb, p.j0 + a.part_blocks);
    p.kind = nparts == 1 ? kFinal : kPartialFixed;
    p.part = part;
    p.which = 0;
    p.seg_start = 0;
    return true;
  }
  return false;
}

// Chunks of up to 32 consecutive blocks of the CTA's piece sequence.
struct ChunkIter {
  Cursor cur;
  Piece pc;
  int jb;
  bool valid;
};

__device__ __forceinline__ bool next_chunk(const DecodeArgs& a, const int* pre, ChunkIter& it,
                                           int& s, int& kvh, int& jb, int& n) {
  while (true) {
    if (it.valid && it.jb < it.pc.j1) {
      s = it.pc.s;
      kvh = it.pc.kvh;
      jb = it.jb;
      n = min(32, it.pc.j1 - it.jb);
      it.jb += n;
      return true;
    }
    if (!next_piece(a, pre, it.cur, it.pc, false)) return false;
    it.valid = true;
    it.jb = it.pc.j0;
  }
}

__device__ __forceinline__ int load_ids(const DecodeArgs& a, int s, int jb, int n, int lane) {
  int id = 0;
  if (lane < n) {
    id = a.block_tables[static_cast<long long>(s) * a.max_blocks + jb + lane];
    if (id < 0 || id >= a.num_blocks) {
      atomicOr(a.err, PA_DEVERR_BLOCK_ID);
      id = -1;  // the TMA box then lies outside the pool and reads zeros
    }
  }
  return id;
}

// Address of the 16-byte chunk `chunk` (8 bf16) of token row `tok` in a
// block staged as kHalves 128-byte-swizzled boxes of 16 rows.
__device__ __forceinline__ uint32_t swz(uint32_t base, int tok, int chunk) {
  return base + (chunk >> 3) * kBoxBytes + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4);
}

template <int D>
__device__ __forceinline__ void attend_block(uint32_t kbase, uint32_t vbase,
                                             const uint32_t (&qf)[D / 16][2],
                                             float (&o)[D / 16][4], float& m0, float& m1,
                                             float& l0, float& l1, int valid, float scale_log2,
                                             int lane) {
  constexpr int KS = D / 16;
  const int i = lane >> 3, r = lane & 7;
  float sacc[4] = {0.f, 0.f, 0.f, 0.f};
  const int ktok = r + ((i & 1) << 3);
#pragma unroll
  for (int ks = 0; ks < KS; ++ks) {
    uint32_t a[4];
    ldsm_x4(swz(kbase, ktok, ks * 2 + (i >> 1)), a);
    mma_bf16_16816(sacc, a, qf[ks][0], qf[ks][1]);
  }
  // sacc: [token lane/4][heads 2q, 2q+1], [token lane/4 + 8][same heads]
  const int t0 = lane >> 2;
  const bool v0 = t0 < valid, v1 = t0 + 8 < valid;
  const float x0 = v0 ? sacc[0] * scale_log2 : -INFINITY;
  const float x1 = v0 ? sacc[1] * scale_log2 : -INFINITY;
  const float x2 = v1 ? sacc[2] * scale_log2 : -INFINITY;
  const float x3 = v1 ? sacc[3] * scale_log2 : -INFINITY;
  float mxa = fmaxf(x0, x2), mxb = fmaxf(x1, x3);
#pragma unroll
  for (int off = 4; off < 32; off <<= 1) {
    mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
    mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
  }
  const float mna = fmaxf(m0, mxa), mnb = fmaxf(m1, mxb);
  const float aa = fast_exp2(m0 - mna), ab = fast_exp2(m1 - mnb);
  const float pa0 = fast_exp2(x0 - mna), pb0 = fast_exp2(x1 - mnb);
  const float pa1 = fast_exp2(x2 - mna), pb1 = fast_exp2(x3 - mnb);
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
  const uint32_t b0 = movmatrix_trans(pack_bf16x2(pa0, pb0));
  const uint32_t b1 = movmatrix_trans(pack_bf16x2(pa1, pb1));
  const int vtok = r + ((i >> 1) << 3);
  uint32_t keep01 = 0xffffffffu, keep23 = 0xffffffffu;
  if (valid < 16) {  // masked tokens have p = 0, but their V rows may hold anything
    const int q2 = (lane & 3) * 2;
    keep01 = (q2 < valid ? 0x0000ffffu : 0u) | (q2 + 1 < valid ? 0xffff0000u : 0u);
    keep23 = (q2 + 8 < valid ? 0x0000ffffu : 0u) | (q2 + 9 < valid ? 0xffff0000u : 0u);
  }
#pragma unroll
  for (int mt = 0; mt < KS; ++mt) {
    uint32_t a[4];
    ldsm_x4_trans(swz(vbase, vtok, mt * 2 + (i & 1)), a);
    a[0] &= keep01;
    a[1] &= keep01;
    a[2] &= keep23;
    a[3] &= keep23;
    mma_bf16_16816(o[mt], a, b0, b1);
  }
}

template <int D>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeArgs a) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  float* obuf = reinterpret_cast<float*>(smem + C::kObufOff);
  float* mlbuf = reinterpret_cast<float*>(smem + C::kMlOff);
  float* lsebuf = reinterpret_cast<float*>(smem + C::kLseOff);
  int* misc = reinterpret_cast<int*>(smem + C::kMiscOff);
  int* pre = reinterpret_cast<int*>(smem + C::kPreOff);
  const uint32_t bar_full = sbase + C::kBarOff;
  const uint32_t bar_empty = bar_full + C::kStages * 8;

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int G = a.group;

  if (tid == 0) {
    for (int st = 0; st < C::kStages; ++st) {
      mbar_init(bar_full + st * 8, 1);
      mbar_init(bar_empty + st * 8, 1);
    }
    misc[0] = 0;  // abort flag
    fence_mbar_init();
  }

  Cursor cur{};
  if (a.mode == kModeBalanced) {
    // exclusive prefix of block counts over sequences (every thread of the CTA)
    const int S = a.num_seqs;
    const int per = (S + kThreads - 1) / kThreads;
    const int s0 = min(S, tid * per), s1 = min(S, s0 + per);
    int local = 0;
    for (int s = s0; s < s1; ++s) local += (load_len(a, s, false) + kBlockSize - 1) / kBlockSize;
    int incl = local;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      int v = __shfl_up_sync(0xffffffffu, incl, off);
      if (lane >= off) incl += v;
    }
    if (lane == 31) misc[8 + warp] = incl;
    __syncthreads();
    int warp_base = 0;
    for (int w = 0; w < warp; ++w) warp_base += misc[8 + w];
    int run = warp_base + incl - local;
    for (int s = s0; s < s1; ++s) {
      pre[s] = run;
      run += (load_len(a, s, false) + kBlockSize - 1) / kBlockSize;
    }
    if (tid == kThreads - 1) pre[S] = run;
    __syncthreads();
    cur.W = static_cast<long long>(a.num_kv_heads) * pre[S];
    cur.C = static_cast<int>(cur.W < gridDim.x ? cur.W : gridDim.x);
    if (static_cast<int>(blockIdx.x) < cur.C) {
      cur.lo = static_cast<long long>(blockIdx.x) * cur.W / cur.C;
      cur.hi = static_cast<long long>(blockIdx.x + 1) * cur.W / cur.C;
    } else {
      cur.lo = cur.hi = 0;
    }
    cur.idx = cur.lo;
  } else {
    cur.u = blockIdx.x;
    cur.U = static_cast<long long>(a.num_seqs) * a.max_parts * a.num_kv_heads;
    __syncthreads();
  }

  if (warp == kConsumerWarps) {
    // ------------------------------------------------------------ producer
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
    }
    const uint64_t pol = l2_policy_evict_first();
    ChunkIter it{cur, Piece{}, 0, false};
    int s, kvh, jb, n;
    bool have = next_chunk(a, pre, it, s, kvh, jb, n);
    int ids = have ? load_ids(a, s, jb, n, lane) : 0;
    uint32_t g = 0;
    bool ok = true;
    while (have && ok) {
      int s2, kvh2, jb2, n2;
      const bool have2 = next_chunk(a, pre, it, s2, kvh2, jb2, n2);
      const int ids2 = have2 ? load_ids(a, s2, jb2, n2, lane) : 0;
      for (int i = 0; i < n; ++i, ++g) {
        const int blk = __shfl_sync(0xffffffffu, ids, i);
        if (lane == 0 && ok) {
          const uint32_t st = g % C::kStages;
          if (g >= static_cast<uint32_t>(C::kStages) &&
              !mbar_wait(bar_empty + st * 8, ((g / C::kStages) - 1) & 1)) {
            atomicOr(a.err, PA_DEVERR_TIMEOUT);
            *reinterpret_cast<volatile int*>(misc) = 1;
            ok = false;
          } else {
            const uint32_t fb = bar_full + st * 8;
            mbar_arrive_expect_tx(fb, C::kStageBytes);
            const uint32_t kdst = sbase + C::kStageOff + st * C::kStageBytes;
            const uint32_t vdst = kdst + C::kKBytes;
            const int z = blk * kBlockSize;
#pragma unroll
            for (int h = 0; h < C::kHalves; ++h) {
              tma_load_3d(kdst + h * kBoxBytes, &tm_k, h * 64, kvh, z, fb, pol);
              tma_load_3d(vdst + h * kBoxBytes, &tm_v, h * 64, kvh, z, fb, pol);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
        if (!ok) break;
      }
      s = s2;
      kvh = kvh2;
      jb = jb2;
      n = n2;
      ids = ids2;
      have = have2;
    }
    return;
  }

  // -------------------------------------------------------------- consumers
  constexpr int KS = D / 16;
  const int ctid = tid;  // 0..127
  if (a.mode == kModeBalanced) {
    // sequences without tokens produce out = 0, lse = -inf
    for (int s = blockIdx.x; s < a.num_seqs; s += gridDim.x) {
      if (load_len(a, s, ctid == 0) != 0) continue;
      for (int e = ctid; e < a.num_q_heads * D; e += kConsumerWarps * 32)
        a.out[static_cast<long long>(s) * a.num_q_heads * D + e] = __float2bfloat16(0.f);
      if (a.out_lse)
        for (int h = ctid; h < a.num_q_heads; h += kConsumerWarps * 32)
          a.out_lse[static_cast<long long>(s) * a.num_q_heads + h] = -INFINITY;
    }
  }

  // After a timeout every consumer warp keeps walking its pieces (skipping
  // the waits and the math) so that all of them still meet at each named
  // barrier; nothing waits without a bound.
  volatile int* abort_flag = misc;
  Piece pc;
  uint32_t g = 0;
  while (next_piece(a, pre, cur, pc, ctid == 0)) {
    // query fragments of the group: B operand (k = dim, n = head)
    uint32_t qf[KS][2];
    {
      const int hq = lane >> 2;
      const __nv_bfloat16* qrow =
          a.q + (static_cast<long long>(pc.s) * a.num_q_heads + pc.kvh * G + hq) * D;
#pragma unroll
      for (int ks = 0; ks < KS; ++ks) {
        const int c = ks * 16 + (lane & 3) * 2;
        qf[ks][0] = hq < G ? *reinterpret_cast<const uint32_t*>(qrow + c) : 0u;
        qf[ks][1] = hq < G ? *reinterpret_cast<const uint32_t*>(qrow + c + 8) : 0u;
      }
    }
    float o[KS][4];
#pragma unroll
    for (int mt = 0; mt < KS; ++mt) o[mt][0] = o[mt][1] = o[mt][2] = o[mt][3] = 0.f;
    float m0 = -INFINITY, m1 = -INFINITY, l0 = 0.f, l1 = 0.f;

    for (int j = pc.j0; j < pc.j1; ++j, ++g) {
      if (static_cast<int>(g & (kConsumerWarps - 1)) != warp) continue;
      if (*abort_flag) continue;
      const uint32_t st = g % C::kStages;
      if (!mbar_wait(bar_full + st * 8, (g / C::kStages) & 1)) {
        atomicOr(a.err, PA_DEVERR_TIMEOUT);
        *abort_flag = 1;
        continue;
      }
      const int valid = min(kBlockSize, pc.len - j * kBlockSize);
      const uint32_t kb = sbase + C::kStageOff + st * C::kStageBytes;
      attend_block<D>(kb, kb + C::kKBytes, qf, o, m0, m1, l0, l1, valid, a.scale_log2, lane);
      __syncwarp();
      if (lane == 0) mbar_arrive(bar_empty + st * 8);
    }

    // ---- merge the 4 warps' running states
#pragma unroll
    for (int off = 4; off < 32; off <<= 1) {
      l0 += __shfl_xor_sync(0xffffffffu, l0, off);
      l1 += __shfl_xor_sync(0xffffffffu, l1, off);
    }
    const int q4 = lane & 3;
    if (lane < 4) {
      mlbuf[(warp * kMaxGroup + 2 * q4) * 2 + 0] = m0;
      mlbuf[(warp * kMaxGroup + 2 * q4) * 2 + 1] = l0;
      mlbuf[(warp * kMaxGroup + 2 * q4 + 1) * 2 + 0] = m1;
      mlbuf[(warp * kMaxGroup + 2 * q4 + 1) * 2 + 1] = l1;
    }
    named_barrier(1, kConsumerWarps * 32);
    float fa, fb;
    {
      float f[2];
#pragma unroll
      for (int k = 0; k < 2; ++k) {
        const int h = 2 * q4 + k;
        float M = -INFINITY;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w) M = fmaxf(M, mlbuf[(w * kMaxGroup + h) * 2]);
        float L = 0.f;
        if (M != -INFINITY) {
#pragma unroll
          for (int w = 0; w < kConsumerWarps; ++w)
            L += mlbuf[(w * kMaxGroup + h) * 2 + 1] *
                 fast_exp2(mlbuf[(w * kMaxGroup + h) * 2] - M);
        }
        const float mine = k == 0 ? m0 : m1;
        f[k] = L > 0.f ? fast_exp2(mine - M) / L : 0.f;
        if (warp == 0 && lane < 4)
          lsebuf[h] = L > 0.f ? (M + __log2f(L)) * kLn2 : -INFINITY;
      }
      fa = f[0];
      fb = f[1];
    }
    {
      const int d0 = lane >> 2;
      float* ob = obuf + warp * kMaxGroup * C::kObufStride;
#pragma unroll
      for (int mt = 0; mt < KS; ++mt) {
        const int d = mt * 16 + d0;
        ob[(2 * q4) * C::kObufStride + d] = o[mt][0] * fa;
        ob[(2 * q4 + 1) * C::kObufStride + d] = o[mt][1] * fb;
        ob[(2 * q4) * C::kObufStride + d + 8] = o[mt][2] * fa;
        ob[(2 * q4 + 1) * C::kObufStride + d + 8] = o[mt][3] * fb;
      }
    }
    named_barrier(1, kConsumerWarps * 32);

    const long long head0 = static_cast<long long>(pc.s) * a.num_q_heads + pc.kvh * G;
    if (pc.kind == kFinal || pc.kind == kPartialFixed) {
      for (int e = ctid; e < G * D; e += kConsumerWarps * 32) {
        const int h = e / D, d = e % D;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
          v += obuf[(w * kMaxGroup + h) * C::kObufStride + d];
        if (pc.kind == kFinal) {
          a.out[(head0 + h) * D + d] = __float2bfloat16(v);
          if (d == 0 && a.out_lse) a.out_lse[head0 + h] = lsebuf[h];
        } else {
          const long long row = (head0 + h) * a.max_parts + pc.part;
          a.part_o[row * D + d] = v;
          if (d == 0) a.part_lse[row] = lsebuf[h];
        }
      }
    } else {
      // balanced partial: publish to this CTA's slot, then the last of the
      // segment's pieces merges them all
      float* slot = a.part_o + (static_cast<long long>(blockIdx.x) * 2 + pc.which) * a.slot_floats;
      for (int e = ctid; e < G * D; e += kConsumerWarps * 32) {
        const int h = e / D, d = e % D;
        float v = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumerWarps; ++w)
          v += obuf[(w * kMaxGroup + h) * C::kObufStride + d];
        slot[e] = v;
        if (d == 0) slot[G * D + h] = lsebuf[h];
      }
      __threadfence();
      named_barrier(1, kConsumerWarps * 32);
      const long long c_first = cta_of(pc.seg_start, cur.W, cur.C);
      const long long c_last = cta_of(pc.seg_start + pc.nb - 1, cur.W, cur.C);
      const int npieces = static_cast<int>(c_last - c_first + 1);
      if (ctid == 0) misc[1] = atomicAdd(a.counters + c_first, 1);
      named_barrier(1, kConsumerWarps * 32);
      if (misc[1] == npieces - 1) {
        __threadfence();
        for (int e = ctid; e < G * D; e += kConsumerWarps * 32) {
          const int h = e / D, d = e % D;
          float L = -INFINITY;
          for (int k = 0; k < npieces; ++k) {
            const float* sl = a.part_o + ((c_first + k) * 2 + (k == 0 ? 1 : 0)) * a.slot_floats;
            L = fmaxf(L, __ldcg(sl + G * D + h));
          }
          float wsum = 0.f, acc = 0.f;
          if (L != -INFINITY) {
            for (int k = 0; k < npieces; ++k) {
              const float* sl = a.part_o + ((c_first + k) * 2 + (k == 0 ? 1 : 0)) * a.slot_floats;
              const float w = __expf(__ldcg(sl + G * D + h) - L);
              wsum += w;
              acc += w * __ldcg(sl + e);
            }
          }
          a.out[(head0 + h) * D + d] = __float2bfloat16(wsum > 0.f ? acc / wsum : 0.f);
          if (d == 0 && a.out_lse) a.out_lse[head0 + h] = wsum > 0.f ? L + __logf(wsum) : -INFINITY;
        }
        if (ctid == 0) a.counters[c_first] = 0;
      }
    }
  }
}

}  // namespace

size_t balanced_slot_floats(int group, int head_dim) {
  const size_t f = static_cast<size_t>(group) * head_dim + group;
  return (f + 63) / 64 * 64;
}

size_t balanced_workspace_bytes(int grid, int group, int head_dim) {
  const size_t counters = (static_cast<size_t>(grid) * 4 + 255) / 256 * 256;
  return counters + static_cast<size_t>(grid) * 2 * balanced_slot_floats(group, head_dim) * 4;
}

int decode_grid(int num_sms, int mode) {
  (void)mode;
  return num_sms;
}

size_t decode_smem_bytes(int head_dim, int mode, int num_seqs) {
  const size_t pre = mode == kModeBalanced ? static_cast<size_t>(num_seqs + 1) * 4 : 0;
  const size_t fixed = head_dim == 128 ? Cfg<128>::kPreOff : Cfg<64>::kPreOff;
  return fixed + pre + 1024;
}

cudaError_t launch_decode(const DecodeArgs& a, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                          int head_dim, int grid, cudaStream_t stream) {
  const size_t smem = decode_smem_bytes(head_dim, a.mode, a.num_seqs);
  cudaError_t e;
  if (head_dim == 128) {
    e = cudaFuncSetAttribute(decode_kernel<128>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    decode_kernel<128><<<grid, kThreads, smem, stream>>>(*tm_k, *tm_v, a);
  } else {
    e = cudaFuncSetAttribute(decode_kernel<64>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(smem));
    if (e != cudaSuccess) return e;
    decode_kernel<64><<<grid, kThreads, smem, stream>>>(*tm_k, *tm_v, a);
  }
  return cudaGetLastError();
}

}  // namespace pa
