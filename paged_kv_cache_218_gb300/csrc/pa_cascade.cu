// pa_cascade.cu -- shared-prefix pass of cascade decode for sm_103a.
//
// Cascade inference ("03 - Engines Papers", section 12 Cascade Inference /
// Multi-Query Cascade Attention): when several requests share a prefix, the
// attention over the shared prefix is computed once for all of them, batched
// across their queries, and combined with each request's private-suffix
// attention by log-sum-exp.  This kernel is the batched prefix pass; the
// suffix pass is the paged decode started from this pass's result
// (DecodeArgs::init_o / init_lse), which is the log-sum-exp merge.
//
// One CTA per (group, subset of kv heads) -- or, when there are too few of
// those to fill the GPU, a few CTAs each taking an equal share of the
// prefix's blocks, whose partial results the last of them to finish merges
// by log-sum-exp.  The producer warp streams the CTA's prefix blocks once --
// per block one TMA box per 64-column half and
// pool covering 16 tokens x the subset's kv heads -- and every consumer warp
// uses each block for 16 query rows, a row being one (member, q head) pair of
// one kv head.  So a prefix byte read from HBM serves every member.
// S = Q K^T and O += P V are warp MMAs (m16n8k16, bf16 in, fp32 accumulate)
// with the query rows on M: the queries stay in registers for the CTA's life,
// K comes by ldmatrix and V by ldmatrix.trans from the swizzled stage, P goes
// from the score accumulators straight into the A fragment of PV.  Each row
// sees the prefix up to its own member's length; V rows of tokens no row sees
// are zeroed, so NaN in unused slots cannot leak in.  The result per (member,
// q head) is normalized o (fp32) and lse (natural log).
#include <math.h>

#include <mutex>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kCW = 8;  // consumer warps
constexpr int kCThreads = kCW * 32 + 32;
constexpr int kCMaxStages = 8;
constexpr int kHeadBox = 16 * 128;  // one head, 16 tokens, one 64-column half (bf16)
constexpr float kLn2C = 0.6931471805599453f;

struct CLayout {
  int stage_bytes, q_off, q_row_bytes, q_bytes, bar_off, misc_off, total;
};

__host__ __device__ inline CLayout cascade_layout(int KH, int Mmax, int G, int stages) {
  CLayout L;
  L.stage_bytes = 2 * 2 * KH * kHeadBox;  // K and V, two 64-column halves each
  L.q_off = stages * L.stage_bytes;
  L.q_row_bytes = KH * G * 128 * 2;  // one member's q rows of the subset
  L.q_bytes = Mmax * L.q_row_bytes;
  L.bar_off = L.q_off + L.q_bytes;
  L.misc_off = L.bar_off + (2 * kCMaxStages + 1) * 8;
  L.total = L.misc_off + (8 + Mmax) * 4;
  return L;
}

__device__ __forceinline__ uint32_t swz2(uint32_t base, int tok, int chunk, uint32_t half) {
  return base + (chunk >> 3) * half + tok * 128 + (((chunk & 7) ^ (tok & 7)) << 4);
}

__global__ void __launch_bounds__(kCThreads, 1)
    cascade_prefix_kernel(const __grid_constant__ CUtensorMap tm_k,
                          const __grid_constant__ CUtensorMap tm_v, const CascadeArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);

  const int KH = a.kv_per_cta, G = a.group, Mmax = a.max_group, wpk = a.warps_per_kv;
  const int Hq = a.num_q_heads;
  const int nsub = a.num_kv_heads / KH;
  const int part = blockIdx.x % a.parts, unit = blockIdx.x / a.parts;
  const int grp = unit / nsub, hs = unit % nsub;
  const int NS = a.stages;
  const CLayout L = cascade_layout(KH, Mmax, G, NS);
  const uint32_t bar_full = sbase + L.bar_off;
  const uint32_t bar_empty = bar_full + kCMaxStages * 8;
  const uint32_t bar_q = bar_empty + kCMaxStages * 8;
  int* misc = reinterpret_cast<int*>(smem + L.misc_off);  // 0 abort, 1 nbp, 2 M, 3 s0, 4 Lmax, 8.. limits
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;

  if (tid == 0) {
    for (int st = 0; st < NS; ++st) {
      mbar_init(bar_full + st * 8, 1);
      mbar_init(bar_empty + st * 8, kCW);
    }
    mbar_init(bar_q, 1);
    fence_mbar_init();
  }
  griddep_wait();
  griddep_launch_dependents();
  if (tid == 0) {
    int s0 = a.group_offsets[grp], s1 = a.group_offsets[grp + 1];
    int M = s1 - s0;
    if (s0 < 0 || M < 0 || M > Mmax || s1 > a.num_seqs) {
      atomicOr(a.err, PA_DEVERR_GROUP);
      M = 0;
      s0 = 0;
    }
    int nbp = 0, lmax = 0;
    for (int m = 0; m < M; ++m) {
      int len = a.seq_lens[s0 + m];
      int sb = a.shared_blocks[s0 + m];
      if (sb < 0 || sb > a.max_prefix_blocks) {
        atomicOr(a.err, PA_DEVERR_GROUP);
        sb = sb < 0 ? 0 : a.max_prefix_blocks;
      }
      if (len < 0) len = 0;
      const int lim = min(len, sb * kBlockSize);
      misc[8 + m] = lim;
      lmax = max(lmax, lim);
      nbp = max(nbp, (lim + kBlockSize - 1) / kBlockSize);
    }
    misc[0] = 0;
    misc[1] = nbp;
    misc[2] = M;
    misc[3] = s0;
    misc[4] = lmax;
  }
  __syncthreads();
  const int nbp = misc[1], M = misc[2], s0 = misc[3], lmax = misc[4];
  // this CTA's share of the prefix blocks
  const int j_lo = part * nbp / a.parts, j_hi = (part + 1) * nbp / a.parts;
  volatile int* abort_flag = misc;

  if (warp == kCW) {
    // ------------------------------------------------------------ producer
    bool ok = true;
    if (lane == 0) {
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      // one copy per (member, kv head): G rows of 256 bytes, at most 2 KB
      mbar_arrive_expect_tx(bar_q, static_cast<uint32_t>(M) * L.q_row_bytes);
      for (int m = 0; m < M; ++m)
        for (int h = 0; h < KH; ++h)
          bulk_load(sbase + L.q_off + m * L.q_row_bytes + h * G * 256,
                    a.q + (static_cast<long long>(s0 + m) * Hq + (hs * KH + h) * G) * 128,
                    G * 256, bar_q);
    }
    const uint64_t pol = l2_policy_evict_first();
    for (int jb = j_lo; jb < j_hi && ok; jb += 32) {
      const int n = min(32, j_hi - jb);
      int id = 0;
      if (lane < n) {
        id = a.prefix_tables[static_cast<long long>(grp) * a.max_prefix_blocks + jb + lane];
        if (id < 0 || id >= a.num_blocks) {
          atomicOr(a.err, PA_DEVERR_BLOCK_ID);
          id = -1;  // the box lies outside the pool and reads zeros
        }
      }
      for (int i = 0; i < n && ok; ++i) {
        const int blk = __shfl_sync(0xffffffffu, id, i);
        const int jj = jb + i - j_lo;  // place in this CTA's stream
        const int st = jj % NS;
        if (lane == 0) {
          if (jj >= NS && !mbar_wait(bar_empty + st * 8, ((jj / NS) - 1) & 1)) {
            atomicOr(a.err, PA_DEVERR_TIMEOUT);
            ok = false;
          } else {
            const uint32_t fb = bar_full + st * 8;
            mbar_arrive_expect_tx(fb, L.stage_bytes);
            const uint32_t kdst = sbase + st * L.stage_bytes;
            const uint32_t vdst = kdst + 2 * KH * kHeadBox;
            const int y = blk * kBlockSize;
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              tma_load_3d(kdst + h * KH * kHeadBox, &tm_k, h * 64, y, hs * KH, fb, pol);
              tma_load_3d(vdst + h * KH * kHeadBox, &tm_v, h * 64, y, hs * KH, fb, pol);
            }
          }
        }
        ok = __shfl_sync(0xffffffffu, ok ? 1 : 0, 0) != 0;
      }
    }
    if (!ok) *abort_flag = 1;
    return;
  }

  // -------------------------------------------------------------- consumers
  // rows of absent members read zeros (their results are discarded)
  for (int e = M * L.q_row_bytes / 16 + tid; e < Mmax * L.q_row_bytes / 16; e += kCW * 32)
    *reinterpret_cast<uint4*>(smem + L.q_off + e * 16) = make_uint4(0u, 0u, 0u, 0u);
  named_barrier(1, kCW * 32);
  const int kh = warp / wpk, t = warp % wpk;
  const bool active = kh < KH;
  if (!mbar_wait_warp(bar_q, 0)) {
    if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
    *abort_flag = 1;
  }
  const int g = lane >> 2, c = lane & 3;
  // query A fragments of this warp's 16 rows, kept for every block
  uint32_t qa[8][4];
  {
    const int r = (lane & 7) + ((lane >> 3) & 1) * 8;
    int R = t * 16 + r;
    int mR = R / G;
    if (mR >= Mmax) R = 0, mR = 0;
    const uint32_t row = sbase + L.q_off + mR * L.q_row_bytes +
                         ((active ? kh : 0) * G + (R % G)) * 256;
#pragma unroll
    for (int ks = 0; ks < 8; ++ks) ldsm_x4(row + (ks * 16 + (lane >> 4) * 8) * 2, qa[ks]);
  }
  const int Ra = t * 16 + g, Rb = Ra + 8;
  const int ma = Ra / G, mb = Rb / G;
  const int La = ma < M ? misc[8 + ma] : 0, Lb = mb < M ? misc[8 + mb] : 0;
  float o[16][4];
#pragma unroll
  for (int nd = 0; nd < 16; ++nd) o[nd][0] = o[nd][1] = o[nd][2] = o[nd][3] = 0.f;
  float mA = -INFINITY, mB = -INFINITY, lA = 0.f, lB = 0.f;
  const float sl2 = a.scale_log2;
  const uint32_t half = KH * kHeadBox;

  for (int j = j_lo; j < j_hi; ++j) {
    const int st = (j - j_lo) % NS;
    if (warp_flag(abort_flag)) break;
    if (!mbar_wait_warp(bar_full + st * 8, ((j - j_lo) / NS) & 1)) {
      if (lane == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
      *abort_flag = 1;
      break;
    }
    if (active) {
      const uint32_t kb = sbase + st * L.stage_bytes + kh * kHeadBox;
      const uint32_t vb = kb + 2 * KH * kHeadBox;
      float sc[2][2][4];
#pragma unroll
      for (int x = 0; x < 2; ++x)
#pragma unroll
        for (int y = 0; y < 2; ++y) sc[x][y][0] = sc[x][y][1] = sc[x][y][2] = sc[x][y][3] = 0.f;
      const int ktok = (lane & 7) + ((lane >> 4) << 3);
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        uint32_t kf[4];
        ldsm_x4(swz2(kb, ktok, ks * 2 + ((lane >> 3) & 1), half), kf);
        mma_bf16_16816(sc[0][ks & 1], qa[ks], kf[0], kf[1]);
        mma_bf16_16816(sc[1][ks & 1], qa[ks], kf[2], kf[3]);
      }
      // scores of rows g (a) and g + 8 (b) at tokens 16j + 8nt + 2c + e
      float xa[2][2], xb[2][2];
      float mxa = -INFINITY, mxb = -INFINITY;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          const int tok = j * kBlockSize + nt * 8 + 2 * c + e;
          xa[nt][e] = tok < La ? (sc[nt][0][e] + sc[nt][1][e]) * sl2 : -INFINITY;
          xb[nt][e] = tok < Lb ? (sc[nt][0][2 + e] + sc[nt][1][2 + e]) * sl2 : -INFINITY;
          mxa = fmaxf(mxa, xa[nt][e]);
          mxb = fmaxf(mxb, xb[nt][e]);
        }
#pragma unroll
      for (int off = 1; off < 4; off <<= 1) {
        mxa = fmaxf(mxa, __shfl_xor_sync(0xffffffffu, mxa, off));
        mxb = fmaxf(mxb, __shfl_xor_sync(0xffffffffu, mxb, off));
      }
      const float na = fmaxf(mA, mxa), nb = fmaxf(mB, mxb);
      const float ua = na == -INFINITY ? 0.f : na, ub = nb == -INFINITY ? 0.f : nb;
      const float alA = fast_exp2(mA - ua), alB = fast_exp2(mB - ub);
      float pa_[2][2], pb_[2][2];
      float ra = 0.f, rb = 0.f;
#pragma unroll
      for (int nt = 0; nt < 2; ++nt)
#pragma unroll
        for (int e = 0; e < 2; ++e) {
          pa_[nt][e] = fast_exp2(xa[nt][e] - ua);
          pb_[nt][e] = fast_exp2(xb[nt][e] - ub);
          ra += pa_[nt][e];
          rb += pb_[nt][e];
        }
      lA = lA * alA + ra;
      lB = lB * alB + rb;
      mA = na;
      mB = nb;
#pragma unroll
      for (int nd = 0; nd < 16; ++nd) {
        o[nd][0] *= alA;
        o[nd][1] *= alA;
        o[nd][2] *= alB;
        o[nd][3] *= alB;
      }
      uint32_t pk[4];
      pk[0] = pack_bf16x2(pa_[0][0], pa_[0][1]);
      pk[1] = pack_bf16x2(pb_[0][0], pb_[0][1]);
      pk[2] = pack_bf16x2(pa_[1][0], pa_[1][1]);
      pk[3] = pack_bf16x2(pb_[1][0], pb_[1][1]);
      // tokens no row of the group sees may hold anything: zero their V halves
      const int vis = min(kBlockSize, lmax - j * kBlockSize);
      uint32_t keep01 = 0xffffffffu, keep23 = 0xffffffffu;
      if (vis < kBlockSize) {
        const int q2 = 2 * c;
        keep01 = (q2 < vis ? 0x0000ffffu : 0u) | (q2 + 1 < vis ? 0xffff0000u : 0u);
        keep23 = (q2 + 8 < vis ? 0x0000ffffu : 0u) | (q2 + 9 < vis ? 0xffff0000u : 0u);
      }
      const int vtok = (lane & 7) + (((lane >> 3) & 1) << 3);
#pragma unroll
      for (int np = 0; np < 8; ++np) {
        uint32_t vf[4];
        ldsm_x4_trans(swz2(vb, vtok, 2 * np + (lane >> 4), half), vf);
        vf[0] &= keep01;
        vf[1] &= keep23;
        vf[2] &= keep01;
        vf[3] &= keep23;
        mma_bf16_16816(o[2 * np], pk, vf[0], vf[1]);
        mma_bf16_16816(o[2 * np + 1], pk, vf[2], vf[3]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(bar_empty + st * 8);
  }

  // ---- normalized o and lse per row, for present members
#pragma unroll
  for (int off = 1; off < 4; off <<= 1) {
    lA += __shfl_xor_sync(0xffffffffu, lA, off);
    lB += __shfl_xor_sync(0xffffffffu, lB, off);
  }
  // part 0 writes into the prefix result itself, the others into their own
  // partial buffers (a row without a visible token gets o = 0, lse = -inf)
  const size_t rows_all = static_cast<size_t>(a.num_seqs) * Hq;
  float* dst_o = part == 0 ? a.pre_o : a.part_o + (part - 1) * rows_all * 128;
  float* dst_l = part == 0 ? a.pre_lse : a.part_lse + (part - 1) * rows_all;
  if (active) {
    const float ia = lA > 0.f ? 1.f / lA : 0.f, ib = lB > 0.f ? 1.f / lB : 0.f;
    const int kvg = hs * KH + kh;
    if (ma < M) {
      const long long row = static_cast<long long>(s0 + ma) * Hq + kvg * G + (Ra % G);
#pragma unroll
      for (int nd = 0; nd < 16; ++nd)
        *reinterpret_cast<float2*>(dst_o + row * 128 + nd * 8 + 2 * c) =
            make_float2(o[nd][0] * ia, o[nd][1] * ia);
      if (c == 0) dst_l[row] = lA > 0.f ? (mA + __log2f(lA)) * kLn2C : -INFINITY;
    }
    if (mb < M) {
      const long long row = static_cast<long long>(s0 + mb) * Hq + kvg * G + (Rb % G);
#pragma unroll
      for (int nd = 0; nd < 16; ++nd)
        *reinterpret_cast<float2*>(dst_o + row * 128 + nd * 8 + 2 * c) =
            make_float2(o[nd][2] * ib, o[nd][3] * ib);
      if (c == 0) dst_l[row] = lB > 0.f ? (mB + __log2f(lB)) * kLn2C : -INFINITY;
    }
  }
  if (a.parts == 1) return;
  // ---- the last part of this (group, subset) to finish merges all parts of
  // its rows by log-sum-exp, in part order, into the prefix result
  const int ctid = tid;
  named_barrier(1, kCW * 32);
  if (ctid == 0) misc[5] = atom_add_acq_rel_gpu(a.tickets + unit, 1);
  named_barrier(1, kCW * 32);
  if (misc[5] != a.parts - 1) return;
  const int rows = M * KH * G;  // member-major: (m, kv head of the subset, q head)
  for (int e = ctid; e < rows * 32; e += kCW * 32) {
    const int r = e >> 5, f4 = e & 31;
    const int m = r / (KH * G), h = (r / G) % KH, gq = r % G;
    const long long row = static_cast<long long>(s0 + m) * Hq + (hs * KH + h) * G + gq;
    float lse[kMaxPrefixParts];
    float4 ov[kMaxPrefixParts];
    float L = -INFINITY;
#pragma unroll
    for (int p = 0; p < kMaxPrefixParts; ++p) {
      if (p < a.parts) {
        const float* po = p == 0 ? a.pre_o : a.part_o + (p - 1) * rows_all * 128;
        const float* pl = p == 0 ? a.pre_lse : a.part_lse + (p - 1) * rows_all;
        lse[p] = __ldcg(pl + row);
        ov[p] = __ldcg(reinterpret_cast<const float4*>(po + row * 128) + f4);
        L = fmaxf(L, lse[p]);
      }
    }
    float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
    float wsum = 0.f;
    if (L > -INFINITY) {
#pragma unroll
      for (int p = 0; p < kMaxPrefixParts; ++p) {
        if (p < a.parts) {
          const float w = __expf(lse[p] - L);
          acc.x += w * ov[p].x;
          acc.y += w * ov[p].y;
          acc.z += w * ov[p].z;
          acc.w += w * ov[p].w;
          wsum += w;
        }
      }
    }
    const float inv = wsum > 0.f ? 1.f / wsum : 0.f;
    __syncwarp();  // a warp holds one row: every lane has read part 0's lse
    reinterpret_cast<float4*>(a.pre_o + row * 128)[f4] =
        make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
    if (f4 == 0) a.pre_lse[row] = wsum > 0.f ? L + __logf(wsum) : -INFINITY;
  }
  if (ctid == 0) a.tickets[unit] = 0;
}

}  // namespace

bool cascade_shape(int num_kv_heads, int group, int max_group, int* kv_per_cta, int* warps_per_kv,
                   int* stages) {
  if (max_group < 1 || group < 1 || max_group * group > 32) return false;
  const int wpk = (max_group * group + 15) / 16;
  int kh = 0;
  for (int d = 1; d <= num_kv_heads && d * wpk <= kCW; ++d)
    if (num_kv_heads % d == 0) kh = d;
  if (kh == 0) return false;
  int st = kCMaxStages;
  while (st > 2 && cascade_layout(kh, max_group, group, st).total + 1024 > 227 * 1024) --st;
  if (cascade_layout(kh, max_group, group, st).total + 1024 > 227 * 1024) return false;
  *kv_per_cta = kh;
  *warps_per_kv = wpk;
  *stages = st;
  return true;
}

cudaError_t launch_cascade_prefix(const CascadeArgs& a, const CUtensorMap* tm_k,
                                  const CUtensorMap* tm_v, cudaStream_t stream) {
  const size_t smem = cascade_layout(a.kv_per_cta, a.max_group, a.group, a.stages).total + 1024;
  static std::mutex mu;
  static bool set_for[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set_for[dev]) {
      e = cudaFuncSetAttribute(cascade_prefix_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               227 * 1024);
      if (e != cudaSuccess) return e;
      set_for[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(a.num_groups * (a.num_kv_heads / a.kv_per_cta) *
                                          a.parts));
  cfg.blockDim = dim3(kCThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, cascade_prefix_kernel, *tm_k, *tm_v, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
