// pa_prefill.cu -- causal paged prefill chunks on tcgen05 tensor cores (sm_103a).
//
// A Sarathi hybrid batch carries prefill chunks next to decodes ("03 -
// Engines Papers", section 3 Sarathi / Sarathi-Serve); a chunk's query at
// absolute position p attends over keys 0..p of its own paged KV, the K/V of
// later chunks not being there yet.  This is the one dense contraction of the
// path, so it runs on the 5th-generation tensor cores:
//
//  * One CTA (4 warps) per (128-row query tile, chunk, kv head).  GQA packs
//    the group's q heads into the tile's rows: row r = token (r / G), head
//    (r % G), so each K/V tile serves all G heads (128 / G tokens per tile).
//  * Q lands in shared memory once (TMA, 128-byte swizzle).  K/V tiles of 128
//    keys are assembled from eight 16-token paged blocks by TMA, double
//    buffered behind an mbarrier each.
//  * S = Q K^T: eight tcgen05.mma (M=128, N=128, K=16, bf16 in, fp32
//    accumulate) into tensor memory columns [0, 128); one elected thread
//    issues them and commits to an mbarrier.
//  * Each thread owns one tensor-memory lane = one query row: tcgen05.ld of
//    its 128 scores, causal mask, online-softmax update (running max and
//    sum, FlashAttention-style tiling with the Milakov & Gimelshein
//    recurrence, "References" page), P rounded to bf16 into shared memory
//    (swizzled K-major operand), and the accumulator O rescaled in tensor
//    memory when its row maximum moved.
//  * O += P V: eight tcgen05.mma into columns [128, 256), V read as an
//    MN-major operand straight from the paged tile.
//  * Epilogue: tcgen05.ld of O, divide by the row sum, bf16 store; lse.
// Every mbarrier wait is bounded; a timeout sets PA_DEVERR_TIMEOUT and the
// CTA leaves its loop together (the decision is taken at a block barrier).
#include <math.h>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

constexpr int kThreads = 128;
constexpr int kTileKeys = 128;
constexpr int kHalf = 128 * 128;  // one 64-column half of a 128-row operand: 128 rows x 128 B
constexpr int kQOff = 0;
constexpr int kPOff = kQOff + 2 * kHalf;
constexpr int kStageOff = kPOff + 2 * kHalf;
constexpr int kStageBytes = 4 * kHalf;  // K (two halves) + V (two halves)
constexpr int kVOff = 2 * kHalf;        // V within a stage
constexpr int kBarOff = kStageOff + 2 * kStageBytes;
constexpr int kSmemBytes = kBarOff + 128;
constexpr uint32_t kTmemCols = 256;  // S in [0, 128), O in [128, 256)
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
  return (1u << 4)            // D format: f32
         | (1u << 7)          // A format: bf16
         | (1u << 10)         // B format: bf16
         | (b_mn << 16)       // B major-ness
         | ((128u >> 3) << 17)  // N / 8
         | ((128u >> 4) << 24); // M / 16
}

__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  extern __shared__ uint8_t smem_raw[];
  const uint32_t raw_addr = smem_u32(smem_raw);
  uint8_t* smem = smem_raw + ((1024u - (raw_addr & 1023u)) & 1023u);
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_q = sbase + kBarOff;
  const uint32_t bar_kv = bar_q + 8;  // two stages
  const uint32_t bar_s = bar_q + 24;
  const uint32_t bar_o = bar_q + 32;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kBarOff + 64);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int Hkv = a.num_kv_heads, G = a.group;
  const int tpt = kTileKeys / G;  // query tokens per tile
  const int kvh = blockIdx.x % Hkv;
  const int t2 = blockIdx.x / Hkv;
  const int c = t2 % a.num_chunks;
  const int m = t2 / a.num_chunks;

  // ---- chunk metadata (uniform over the CTA)
  const int q0 = a.cu_q_lens[c], q1 = a.cu_q_lens[c + 1];
  const int p0 = a.q_start_pos[c], n = a.seq_lens[c];
  const int qlen = q1 - q0;
  if (qlen < 0 || p0 < 0 || p0 + qlen > n || n > a.max_blocks * kBlockSize) {
    if (tid == 0 && m == 0 && kvh == 0) atomicOr(a.err, PA_DEVERR_CHUNK);
    return;
  }
  const int t0 = m * tpt;
  if (t0 >= qlen) return;
  const int tv = min(tpt, qlen - t0);  // valid query tokens in this tile
  const int kmax = p0 + t0 + tv;       // keys [0, kmax) are visible to some row
  const int nkt = (kmax + kTileKeys - 1) / kTileKeys;
  const int nb_vis = (kmax + kBlockSize - 1) / kBlockSize;

  if (tid == 0) {
    mbar_init(bar_q, 1);
    mbar_init(bar_kv, 1);
    mbar_init(bar_kv + 8, 1);
    mbar_init(bar_s, 1);
    mbar_init(bar_o, 1);
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const uint32_t tmem_s = tmem;
  const uint32_t tmem_o = tmem + 128;
  const uint32_t lane_off = static_cast<uint32_t>(warp * 32) << 16;

  // K/V tiles are re-read by every query tile of the chunk: keep them in L2
  const uint64_t pol = l2_policy_evict_last();
  // K/V tile j (8 paged blocks) into stage st; blocks past the visible keys
  // are read from outside the pool, which fills zeros
  auto load_tile = [&](int j, int st) {
    const uint32_t fb = bar_kv + st * 8;
    if (lane == 0) mbar_arrive_expect_tx(fb, kStageBytes);
    __syncwarp();
    if (lane < 8) {
      const int jb = j * 8 + lane;
      int id = -1;
      if (jb < nb_vis) {
        id = a.block_tables[static_cast<long long>(c) * a.max_blocks + jb];
        if (id < 0 || id >= a.num_blocks) {
          atomicOr(a.err, PA_DEVERR_BLOCK_ID);
          id = -1;
        }
      }
      const uint32_t kd = sbase + kStageOff + st * kStageBytes + lane * kBlockSize * 128;
      const int z = id * kBlockSize;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        tma_load_3d(kd + h * kHalf, &tm_k, h * 64, kvh, z, fb, pol);
        tma_load_3d(kd + kVOff + h * kHalf, &tm_v, h * 64, kvh, z, fb, pol);
      }
    }
  };

  if (warp == 0) {
    if (lane == 0) {
      tma_prefetch_desc(&tm_q);
      tma_prefetch_desc(&tm_k);
      tma_prefetch_desc(&tm_v);
      mbar_arrive_expect_tx(bar_q, 2 * kHalf);
      for (int h = 0; h < 2; ++h)
        tma_load_3d(sbase + kQOff + h * kHalf, &tm_q, h * 64, kvh * G, q0 + t0, bar_q, pol);
    }
    load_tile(0, 0);
  }

  // this thread's query row
  const int r = tid;
  const int pos = p0 + t0 + r / G;
  const int lim = min(pos, kmax - 1);  // last visible key of the row
  float m_run = -INFINITY, l_run = 0.f;
  bool timed_out = false;
  const uint32_t idesc_s = instr_desc(0), idesc_o = instr_desc(1);

  if (tid == 0 && !mbar_wait(bar_q, 0)) timed_out = true;

  int j = 0;
  for (; j < nkt; ++j) {
    const int st = j & 1;
    const uint32_t stage = sbase + kStageOff + st * kStageBytes;
    // ---- S = Q K_j^T
    if (tid == 0 && !timed_out) {
      if (!mbar_wait(bar_kv + st * 8, (j >> 1) & 1)) {
        timed_out = true;
      } else {
        tc_fence_after();
#pragma unroll
        for (int ks = 0; ks < 8; ++ks) {
          const uint32_t koff = (ks >> 2) * kHalf + (ks & 3) * 32;
          tc_mma_f16(tmem_s, smem_desc(sbase + kQOff + koff, 16, 1024),
                     smem_desc(stage + koff, 16, 1024), idesc_s, ks > 0);
        }
        tc_commit(bar_s);
      }
    }
    // ---- prefetch tile j+1 into the other stage once PV_{j-1} released it
    if (warp == 0 && j + 1 < nkt) {
      bool free_ok = true;
      if (j >= 1 && lane == 0) free_ok = mbar_wait(bar_o, (j - 1) & 1);
      free_ok = __shfl_sync(0xffffffffu, free_ok ? 1 : 0, 0) != 0;
      if (free_ok) load_tile(j + 1, st ^ 1);
      else timed_out = true;
    }
    if (!timed_out && !mbar_wait(bar_s, j & 1)) timed_out = true;
    if (!timed_out && !mbar_wait(bar_kv + st * 8, (j >> 1) & 1)) timed_out = true;
    tc_fence_after();

    // ---- pass 1: row maximum of the visible scores
    const int kb = j * kTileKeys;
    uint32_t v[32];
    float mx = -INFINITY;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      tmem_ld32(tmem_s + lane_off + cc * 32, v);
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const int k = kb + cc * 32 + i;
        const float x = k <= lim ? __uint_as_float(v[i]) * a.scale_log2 : -INFINITY;
        mx = fmaxf(mx, x);
      }
    }
    const float m_new = fmaxf(m_run, mx);
    const float alpha = fast_exp2(m_run - m_new);

    // ---- PV_{j-1} must be done before O and the P buffer are touched
    if (j >= 1 && !timed_out && !mbar_wait(bar_o, (j - 1) & 1)) timed_out = true;
    tc_fence_after();
    if (j >= 1 && __any_sync(0xffffffffu, alpha != 1.f)) {
#pragma unroll
      for (int cc = 0; cc < 4; ++cc) {
        tmem_ld32(tmem_o + lane_off + cc * 32, v);
#pragma unroll
        for (int i = 0; i < 32; ++i) v[i] = __float_as_uint(__uint_as_float(v[i]) * alpha);
        tmem_st32(tmem_o + lane_off + cc * 32, v);
      }
    }

    // ---- pass 2: p = 2^(x - m_new), row sum, P (bf16) into shared memory
    float rs = 0.f;
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      tmem_ld32(tmem_s + lane_off + cc * 32, v);
      uint32_t pk[16];
#pragma unroll
      for (int i = 0; i < 32; i += 2) {
        const int k = kb + cc * 32 + i;
        const float x0 = k <= lim ? __uint_as_float(v[i]) * a.scale_log2 : -INFINITY;
        const float x1 = k + 1 <= lim ? __uint_as_float(v[i + 1]) * a.scale_log2 : -INFINITY;
        const float e0 = fast_exp2(x0 - m_new), e1 = fast_exp2(x1 - m_new);
        rs += e0 + e1;
        pk[i / 2] = pack_bf16x2(e0, e1);
      }
      // keys cc*32 .. cc*32+31 = half cc/2, 16-byte chunks (cc%2)*4 .. +3 of row r
      const uint32_t rowbase = sbase + kPOff + (cc >> 1) * kHalf + r * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int chunk = (cc & 1) * 4 + q;
        const uint32_t addr = rowbase + ((chunk ^ (r & 7)) << 4);
        asm volatile("st.shared.v4.b32 [%0], {%1, %2, %3, %4};" ::"r"(addr), "r"(pk[4 * q]),
                     "r"(pk[4 * q + 1]), "r"(pk[4 * q + 2]), "r"(pk[4 * q + 3])
                     : "memory");
      }
    }
    l_run = l_run * alpha + rs;
    m_run = m_new;

    // ---- the sequence's last block may end inside this tile: its slots past
    // seq_len hold no token and must not reach the PV product
    if ((n & (kBlockSize - 1)) != 0) {
      const int jl = (n - 1) / kBlockSize;
      if (jl < nb_vis && jl / 8 == j) {
        const int first = n - jl * kBlockSize;  // rows first..15 of block jl % 8
        const int rows = kBlockSize - first;
        for (int e = tid; e < rows * 2 * 8; e += kThreads) {
          const int row = first + e / 16, h = (e / 8) & 1, chunk = e & 7;
          const uint32_t addr =
              stage + kVOff + h * kHalf + ((jl & 7) * kBlockSize + row) * 128 + (chunk << 4);
          asm volatile("st.shared.v4.b32 [%0], {%1, %1, %1, %1};" ::"r"(addr), "r"(0u) : "memory");
        }
      }
    }
    fence_proxy_async_smem();
    tc_fence_before();
    if (__syncthreads_or(timed_out ? 1 : 0)) break;

    // ---- O += P V_j
    if (tid == 0) {
      tc_fence_after();
#pragma unroll
      for (int ks = 0; ks < 8; ++ks) {
        const uint32_t poff = (ks >> 2) * kHalf + (ks & 3) * 32;
        tc_mma_f16(tmem_o, smem_desc(sbase + kPOff + poff, 16, 1024),
                   smem_desc(stage + kVOff + ks * 16 * 128, kHalf, 1024), idesc_o,
                   (j > 0 || ks > 0) ? 1u : 0u);
      }
      tc_commit(bar_o);
    }
  }

  bool bad = !(j == nkt && !timed_out);
  if (!bad && !mbar_wait(bar_o, (nkt - 1) & 1)) bad = true;
  bad = __syncthreads_or(bad ? 1 : 0) != 0;  // uniform: tcgen05.ld below is warp-collective
  tc_fence_after();
  if (bad) {
    if (tid == 0) atomicOr(a.err, PA_DEVERR_TIMEOUT);
  } else {
    // ---- epilogue: O / l -> bf16, and lse
    const int tok = r / G, g = r % G;
    const bool store = tok < tv;
    const float inv = l_run > 0.f ? 1.f / l_run : 0.f;
    const long long row = static_cast<long long>(q0 + t0 + tok) * a.num_q_heads + kvh * G + g;
    uint32_t v[32];
#pragma unroll
    for (int cc = 0; cc < 4; ++cc) {
      tmem_ld32(tmem_o + lane_off + cc * 32, v);
      if (store) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 32; i += 2)
          pk[i / 2] = pack_bf16x2(__uint_as_float(v[i]) * inv, __uint_as_float(v[i + 1]) * inv);
        uint4* dst = reinterpret_cast<uint4*>(a.out + row * 128 + cc * 32);
#pragma unroll
        for (int q = 0; q < 4; ++q)
          dst[q] = make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
    }
    if (store && a.out_lse)
      a.out_lse[row] = l_run > 0.f ? (m_run + __log2f(l_run)) * kLn2 : -INFINITY;
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

size_t prefill_smem_bytes() { return kSmemBytes + 1024; }

cudaError_t launch_prefill(const PrefillArgs& a, const CUtensorMap* tm_q, const CUtensorMap* tm_k,
                           const CUtensorMap* tm_v, int grid_tiles, cudaStream_t stream) {
  const size_t smem = prefill_smem_bytes();
  cudaError_t e = cudaFuncSetAttribute(prefill_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       static_cast<int>(smem));
  if (e != cudaSuccess) return e;
  prefill_kernel<<<grid_tiles, kThreads, smem, stream>>>(*tm_q, *tm_k, *tm_v, a);
  return cudaGetLastError();
}

}  // namespace pa
