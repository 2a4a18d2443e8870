// pa_api.cu -- the C ABI of libpa.so (declared in include/pa.h): argument
// checks, TMA descriptor setup, launch selection, and the small kernels
// (slot scatter, block copy, log-sum-exp merge).
#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <math.h>
#include <stdint.h>
#include <string.h>

#include <mutex>
#include <unordered_set>

#include "../../include/pa.h"
#include "pa_internal.h"
#include "pa_ptx.cuh"

namespace pa {
namespace {

// Device error word (PA_DEVERR_* bits), one per device that loads the library.
__device__ unsigned int g_device_error;

constexpr int kMaxDevices = 64;

struct DeviceInfo {
  bool ready = false;
  int num_sms = 0;
  unsigned int* err = nullptr;
};

std::mutex g_mu;
DeviceInfo g_dev[kMaxDevices];
PFN_cuTensorMapEncodeTiled_v12000 g_encode = nullptr;

int current_device_info(DeviceInfo** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return PA_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_mu);
  DeviceInfo& d = g_dev[dev];
  if (!d.ready) {
    if (cudaDeviceGetAttribute(&d.num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
      return PA_ERR_CUDA;
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_device_error) != cudaSuccess) return PA_ERR_CUDA;
    d.err = static_cast<unsigned int*>(p);
    d.ready = true;
  }
  if (!g_encode) {
    void* fn = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &fn, 12000, cudaEnableDefault, &q) !=
            cudaSuccess ||
        q != cudaDriverEntryPointSuccess || fn == nullptr)
      return PA_ERR_CUDA;
    g_encode = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(fn);
  }
  *out = &d;
  return PA_OK;
}

bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }

// Paged pool [num_blocks * 16 tokens, Hkv, D] as a 3-D tensor; box = 64
// columns x 1 head x `rows` tokens, 128-byte swizzle.
// rows > 0: box = 64 columns x 1 head x `rows` tokens (one head of a block).
// rows == 0: the same pool seen as (D, tokens, heads), box = 64 columns x 16
// tokens x Hkv heads -- one whole block, every head, in a single load that
// lands as [head][token][64 columns].
// elem = 1: an E4M3 pool (bytes); only the all-heads view, whose box is a
// whole 128-byte token row (head_dim 128) x 16 tokens x Hkv heads.
// rows == kPool2D: the pool as a 2-D tensor (Hkv * D columns, tokens), box =
// 64 columns x 16 tokens: one head's half of a block, as the 3-D box with
// rows = 16 but cheaper for the TMA unit.
// rows == kPoolKeyTile (bf16, D = 128): the pool as a 4-D tensor (64 columns,
// 8 tokens, 2 * Hkv column chunks of 64, num_blocks * 2 groups of 8 tokens),
// box 64 x 8 x 2 x 2: one head's whole block in one load, landing as
// [token group][64-column half][8 tokens][64 columns].  Every 8-token group
// of a 64-column half then sits 2 KB after the previous one, block after
// block, a uniform stride for a K-major operand descriptor.
constexpr int kPool2D = 1 << 20;
constexpr int kPoolKeyTile = kPool2D + 1;
int encode_pool_map_uncached(CUtensorMap* m, const void* pool, int64_t num_blocks, int Hkv, int D,
                             int rows, int elem) {
  if (rows == kPoolKeyTile) {
    if (D != 128 || elem != 2) return PA_ERR_UNSUPPORTED;
    const cuuint64_t row_bytes = static_cast<cuuint64_t>(Hkv) * D * elem;
    cuuint64_t dims4[4] = {64, 8, 2 * static_cast<cuuint64_t>(Hkv),
                           static_cast<cuuint64_t>(num_blocks) * 2};
    cuuint64_t strides4[3] = {row_bytes, 128, 8 * row_bytes};
    cuuint32_t box4[4] = {64, 8, 2, 2};
    cuuint32_t estr4[4] = {1, 1, 1, 1};
    CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(pool), dims4,
                          strides4, box4, estr4, CU_TENSOR_MAP_INTERLEAVE_NONE,
                          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
  }
  if (rows == kPool2D) {
    cuuint64_t dims2[2] = {static_cast<cuuint64_t>(Hkv) * D,
                           static_cast<cuuint64_t>(num_blocks) * kBlockSize};
    cuuint64_t strides2[1] = {static_cast<cuuint64_t>(Hkv) * D * elem};
    cuuint32_t box2[2] = {static_cast<cuuint32_t>(128 / elem), static_cast<cuuint32_t>(kBlockSize)};
    cuuint32_t estr2[2] = {1, 1};
    CUresult r = g_encode(m, elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                          2, const_cast<void*>(pool), dims2, strides2, box2, estr2,
                          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
  }
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hkv),
                        static_cast<cuuint64_t>(num_blocks) * kBlockSize};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * elem,
                           static_cast<cuuint64_t>(Hkv) * D * elem};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(128 / elem), 1, static_cast<cuuint32_t>(rows)};
  if (rows <= 0) {  // rows < 0: the same view, a box of -rows kv heads
    dims[1] = static_cast<cuuint64_t>(num_blocks) * kBlockSize;
    dims[2] = static_cast<cuuint64_t>(Hkv);
    strides[0] = static_cast<cuuint64_t>(Hkv) * D * elem;
    strides[1] = static_cast<cuuint64_t>(D) * elem;
    box[1] = kBlockSize;
    box[2] = static_cast<cuuint32_t>(rows == 0 ? Hkv : -rows);
  }
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, elem == 1 ? CU_TENSOR_MAP_DATA_TYPE_UINT8 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16,
                        3, const_cast<void*>(pool), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// A serving loop passes the same pools every step: keep the last few pool
// descriptors (they are pure functions of pointer and shape) so a call does
// not re-encode them.
struct PoolMapEntry {
  const void* pool;
  int64_t num_blocks;
  int Hkv, D, rows, elem;
  CUtensorMap map;
};
constexpr int kPoolMapCache = 32;
std::mutex g_map_mu;
PoolMapEntry g_map_cache[kPoolMapCache];
int g_map_next = 0;

int encode_pool_map(CUtensorMap* m, const void* pool, int64_t num_blocks, int Hkv, int D,
                    int rows, int elem = 2) {
  std::lock_guard<std::mutex> lock(g_map_mu);
  for (int i = 0; i < kPoolMapCache; ++i) {
    const PoolMapEntry& e = g_map_cache[i];
    if (e.pool == pool && e.num_blocks == num_blocks && e.Hkv == Hkv && e.D == D &&
        e.rows == rows && e.elem == elem) {
      *m = e.map;
      return PA_OK;
    }
  }
  if (int rc = encode_pool_map_uncached(m, pool, num_blocks, Hkv, D, rows, elem)) return rc;
  PoolMapEntry& e = g_map_cache[g_map_next];
  g_map_next = (g_map_next + 1) % kPoolMapCache;
  e.pool = pool;
  e.num_blocks = num_blocks;
  e.Hkv = Hkv;
  e.D = D;
  e.rows = rows;
  e.elem = elem;
  e.map = *m;
  return PA_OK;
}

// q [T, Hq, D] as a 3-D tensor; box = 64 columns x `heads` heads x `rows` tokens.
int encode_q_map(CUtensorMap* m, const void* q, int64_t T, int Hq, int D, int heads, int rows) {
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(D), static_cast<cuuint64_t>(Hq),
                        static_cast<cuuint64_t>(T)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * 2, static_cast<cuuint64_t>(Hq) * D * 2};
  cuuint32_t box[3] = {64, static_cast<cuuint32_t>(heads), static_cast<cuuint32_t>(rows)};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = g_encode(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(q), dims,
                        strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
                        CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

// A chunk's new K / V rows [T, Hkv, 128] (token strides in elements), read
// by the prefill in place of the pool's slots they are being written to:
// K as (64 columns, T tokens, 2 * Hkv column chunks), box 64 x 8 x 2 -- 8
// tokens of one head's whole row, landing as [64-column half][8 tokens][64
// columns], one token group of a K block in the prefill's layout; V as
// (Hkv * 128 columns, T tokens), box 64 x 16, as the pool's 2-D view.
int encode_new_row_maps(CUtensorMap* nk, CUtensorMap* nv, const void* key, const void* value,
                        int64_t T, int Hkv, int64_t k_stride, int64_t v_stride) {
  cuuint64_t kd[3] = {64, static_cast<cuuint64_t>(T), 2 * static_cast<cuuint64_t>(Hkv)};
  cuuint64_t ks[2] = {static_cast<cuuint64_t>(k_stride) * 2, 128};
  cuuint32_t kb[3] = {64, 8, 2};
  cuuint32_t e3[3] = {1, 1, 1};
  CUresult r = g_encode(nk, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(key), kd, ks,
                        kb, e3, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                        CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS) return PA_ERR_CUDA;
  cuuint64_t vd[2] = {static_cast<cuuint64_t>(Hkv) * 128, static_cast<cuuint64_t>(T)};
  cuuint64_t vs[1] = {static_cast<cuuint64_t>(v_stride) * 2};
  cuuint32_t vb[2] = {64, static_cast<cuuint32_t>(kBlockSize)};
  cuuint32_t e2[2] = {1, 1};
  r = g_encode(nv, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(value), vd, vs, vb, e2,
               CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
               CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? PA_OK : PA_ERR_CUDA;
}

int check_shape(int Hq, int Hkv, int D, int block_size) {
  if (Hq <= 0 || Hkv <= 0 || D <= 0 || block_size <= 0) return PA_ERR_INVALID;
  if (Hq % Hkv != 0) return PA_ERR_INVALID;
  if (block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (D != 64 && D != 128) return PA_ERR_UNSUPPORTED;
  if (Hq / Hkv > kMaxGroup) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// ------------------------------------------------------------------ kernels

// One thread copies 16 bytes (8 bf16) of K and of V for one (token, head).
__global__ void reshape_and_cache_kernel(const uint4* __restrict__ key,
                                         const uint4* __restrict__ value, int64_t key_stride16,
                                         int64_t value_stride16, uint4* __restrict__ k_cache,
                                         uint4* __restrict__ v_cache,
                                         const int64_t* __restrict__ slots, int num_tokens,
                                         int vec_per_token, int64_t num_slots,
                                         unsigned int* err) {
  // the decode / prefill launched after this may begin its prologue now; it
  // waits for this kernel's writes before reading any global memory
  griddep_launch_dependents();
  // launched as a programmatic dependent itself: the previous kernel on the
  // stream (say the last step's decode, still reading the pool) must finish
  // before any slot is written
  griddep_wait();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(num_tokens) * vec_per_token) return;
  const int t = static_cast<int>(i / vec_per_token);
  const int c = static_cast<int>(i % vec_per_token);
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (c == 0) atomicOr(err, PA_DEVERR_SLOT);
    return;
  }
  k_cache[slot * vec_per_token + c] = key[t * key_stride16 + c];
  v_cache[slot * vec_per_token + c] = value[t * value_stride16 + c];
}

// Quantizing scatter into E4M3 pools: one thread turns 8 bf16 of K and of V
// for one (token, head) into 8 bytes each: code = RNE_sat(x / scale[head]),
// the division in IEEE fp32, then round to nearest even onto the E4M3 grid,
// finite values beyond +-448 saturating to +-448.
__global__ void reshape_and_cache_fp8_kernel(const uint4* __restrict__ key,
                                             const uint4* __restrict__ value, int64_t key_stride16,
                                             int64_t value_stride16, uint2* __restrict__ k_cache,
                                             uint2* __restrict__ v_cache,
                                             const int64_t* __restrict__ slots,
                                             const float* __restrict__ k_scales,
                                             const float* __restrict__ v_scales, int num_tokens,
                                             int vec_per_token, int vec_per_head,
                                             int64_t num_slots, unsigned int* err) {
  griddep_launch_dependents();
  griddep_wait();
  const int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (i >= static_cast<int64_t>(num_tokens) * vec_per_token) return;
  const int t = static_cast<int>(i / vec_per_token);
  const int c = static_cast<int>(i % vec_per_token);
  const int64_t slot = slots[t];
  if (slot < 0) return;
  if (slot >= num_slots) {
    if (c == 0) atomicOr(err, PA_DEVERR_SLOT);
    return;
  }
  const int h = c / vec_per_head;
  auto quant8 = [](uint4 x, float sc) {
    const uint32_t w[4] = {x.x, x.y, x.z, x.w};
    uint32_t out[2];
#pragma unroll
    for (int k = 0; k < 2; ++k) {
      uint32_t r = 0;
#pragma unroll
      for (int p = 0; p < 2; ++p) {
        const uint32_t u = w[2 * k + p];
        const float lo = __fdiv_rn(__uint_as_float(u << 16), sc);
        const float hi = __fdiv_rn(__uint_as_float(u & 0xffff0000u), sc);
        r |= static_cast<uint32_t>(f32x2_to_e4m3x2(lo, hi)) << (16 * p);
      }
      out[k] = r;
    }
    return make_uint2(out[0], out[1]);
  };
  k_cache[slot * vec_per_token + c] = quant8(key[t * key_stride16 + c], k_scales[h]);
  v_cache[slot * vec_per_token + c] = quant8(value[t * value_stride16 + c], v_scales[h]);
}

__global__ void copy_blocks_kernel(uint4* __restrict__ k_cache, uint4* __restrict__ v_cache,
                                   const int64_t* __restrict__ pairs, int64_t vec_per_block,
                                   int64_t num_blocks, unsigned int* err) {
  const int p = blockIdx.y;
  const int64_t src = pairs[2 * p], dst = pairs[2 * p + 1];
  if (src < 0 || src >= num_blocks || dst < 0 || dst >= num_blocks) {
    if (blockIdx.x == 0 && threadIdx.x == 0) atomicOr(err, PA_DEVERR_BLOCK_ID);
    return;
  }
  for (int64_t i = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < vec_per_block;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    k_cache[dst * vec_per_block + i] = k_cache[src * vec_per_block + i];
    v_cache[dst * vec_per_block + i] = v_cache[src * vec_per_block + i];
  }
}

// Log-sum-exp merge: one CTA of 128 threads per (sequence, q head); warp w
// takes parts w, w+4, ...; each lane holds head_dim/32 output columns.
template <int D>
__global__ void __launch_bounds__(128) merge_kernel(const MergeArgs a) {
  constexpr int V = D / 32;
  const int s = blockIdx.x / a.num_q_heads;
  const int h = blockIdx.x % a.num_q_heads;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  int np;
  if (a.num_parts) {
    np = a.num_parts[s];
    np = np < 0 ? 0 : (np > a.max_parts ? a.max_parts : np);
  } else {
    int len = a.seq_lens[s];
    const int cap = a.max_blocks * kBlockSize;
    len = len < 0 ? 0 : (len > cap ? cap : len);
    int nb = (len + kBlockSize - 1) / kBlockSize;
    if (a.start_blocks) {
      const int sb = a.start_blocks[s];
      nb = sb <= 0 ? nb : (sb >= nb ? 0 : nb - sb);
    }
    np = nb == 0 ? 1 : (nb + a.part_blocks - 1) / a.part_blocks;
    if (a.skip_single && np == 1) return;
  }
  const int64_t row = static_cast<int64_t>(s) * a.num_q_heads + h;
  const float* lse = a.part_lse + row * a.max_parts;
  const float* po = a.part_o + row * a.max_parts * D;
  __shared__ float red[4];
  __shared__ float acc_s[4][D];
  __shared__ float wsum_s[4];
  float L = -INFINITY;
  for (int p = threadIdx.x; p < np; p += 128) L = fmaxf(L, lse[p]);
#pragma unroll
  for (int off = 16; off > 0; off >>= 1) L = fmaxf(L, __shfl_xor_sync(0xffffffffu, L, off));
  if (lane == 0) red[warp] = L;
  __syncthreads();
  L = fmaxf(fmaxf(red[0], red[1]), fmaxf(red[2], red[3]));
  float acc[V];
#pragma unroll
  for (int v = 0; v < V; ++v) acc[v] = 0.f;
  float wsum = 0.f;
  if (L != -INFINITY) {
    for (int p = warp; p < np; p += 4) {
      const float w = __expf(lse[p] - L);
      wsum += w;
      const float* src = po + static_cast<int64_t>(p) * D + lane * V;
      if constexpr (V == 4) {
        const float4 x = *reinterpret_cast<const float4*>(src);
        acc[0] += w * x.x;
        acc[1] += w * x.y;
        acc[2] += w * x.z;
        acc[3] += w * x.w;
      } else {
        const float2 x = *reinterpret_cast<const float2*>(src);
        acc[0] += w * x.x;
        acc[1] += w * x.y;
      }
    }
  }
#pragma unroll
  for (int v = 0; v < V; ++v) acc_s[warp][lane * V + v] = acc[v];
  if (lane == 0) wsum_s[warp] = wsum;
  __syncthreads();
  const float W = wsum_s[0] + wsum_s[1] + wsum_s[2] + wsum_s[3];
  for (int d = threadIdx.x; d < D; d += 128) {
    const float o = acc_s[0][d] + acc_s[1][d] + acc_s[2][d] + acc_s[3][d];
    a.out[row * a.head_dim + d] = __float2bfloat16(W > 0.f ? o / W : 0.f);
  }
  if (threadIdx.x == 0 && a.out_lse) a.out_lse[row] = W > 0.f ? L + __logf(W) : -INFINITY;
}

}  // namespace

cudaError_t launch_merge(const MergeArgs& a, cudaStream_t stream) {
  const int grid = a.num_seqs * a.num_q_heads;
  if (grid == 0) return cudaSuccess;
  if (a.head_dim == 128)
    merge_kernel<128><<<grid, 128, 0, stream>>>(a);
  else
    merge_kernel<64><<<grid, 128, 0, stream>>>(a);
  return cudaGetLastError();
}

}  // namespace pa

using namespace pa;

extern "C" {

const char* pa_status_string(int status) {
  switch (status) {
    case PA_OK: return "PA_OK";
    case PA_ERR_INVALID: return "PA_ERR_INVALID";
    case PA_ERR_UNSUPPORTED: return "PA_ERR_UNSUPPORTED";
    case PA_ERR_CUDA: return "PA_ERR_CUDA";
    case PA_ERR_WORKSPACE: return "PA_ERR_WORKSPACE";
    case PA_ERR_SCRATCH_LIMIT: return "PA_ERR_SCRATCH_LIMIT";
    default: return "PA_ERR_UNKNOWN";
  }
}

int pa_version(void) { return (1 << 16) | 0; }

int pa_reshape_and_cache(const void* key, const void* value, int64_t key_token_stride,
                         int64_t value_token_stride, void* k_cache, void* v_cache,
                         const int64_t* slot_mapping, int num_tokens, int num_kv_heads,
                         int head_dim, int block_size, int64_t num_blocks, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0) return PA_ERR_INVALID;
  if (block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping) return PA_ERR_INVALID;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 ||
      value_token_stride % 8)
    return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(slot_mapping, 8))
    return PA_ERR_INVALID;
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  const int vec = static_cast<int>(row / 8);
  const int64_t total = static_cast<int64_t>(num_tokens) * vec;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  // programmatic dependent launch: the CTAs may be scheduled while the
  // previous kernel drains, and wait for it inside (griddepcontrol.wait)
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, reshape_and_cache_kernel, static_cast<const uint4*>(key),
                         static_cast<const uint4*>(value), key_token_stride / 8,
                         value_token_stride / 8, static_cast<uint4*>(k_cache),
                         static_cast<uint4*>(v_cache), slot_mapping, num_tokens, vec,
                         num_blocks * block_size, d->err) != cudaSuccess)
    return PA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_reshape_and_cache_fp8(const void* key, const void* value, int64_t key_token_stride,
                             int64_t value_token_stride, void* k_cache, void* v_cache,
                             const int64_t* slot_mapping, const float* k_scales,
                             const float* v_scales, int num_tokens, int num_kv_heads,
                             int head_dim, int block_size, int64_t num_blocks, void* stream) {
  if (num_tokens < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0) return PA_ERR_INVALID;
  if (block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if (head_dim % 8 != 0) return PA_ERR_UNSUPPORTED;
  if (num_tokens == 0) return PA_OK;
  if (!key || !value || !k_cache || !v_cache || !slot_mapping || !k_scales || !v_scales)
    return PA_ERR_INVALID;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 ||
      value_token_stride % 8)
    return PA_ERR_INVALID;
  if (!aligned(key, 16) || !aligned(value, 16) || !aligned(k_cache, 8) || !aligned(v_cache, 8) ||
      !aligned(slot_mapping, 8) || !aligned(k_scales, 4) || !aligned(v_scales, 4))
    return PA_ERR_INVALID;
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  const int vec = static_cast<int>(row / 8);
  const int64_t total = static_cast<int64_t>(num_tokens) * vec;
  const int threads = 256;
  const int64_t blocks = (total + threads - 1) / threads;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(static_cast<unsigned>(blocks));
  cfg.blockDim = dim3(threads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = static_cast<cudaStream_t>(stream);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, reshape_and_cache_fp8_kernel, static_cast<const uint4*>(key),
                         static_cast<const uint4*>(value), key_token_stride / 8,
                         value_token_stride / 8, static_cast<uint2*>(k_cache),
                         static_cast<uint2*>(v_cache), slot_mapping, k_scales, v_scales,
                         num_tokens, vec, head_dim / 8, num_blocks * block_size,
                         d->err) != cudaSuccess)
    return PA_ERR_CUDA;
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

static int copy_blocks_bytes(void* k_cache, void* v_cache, const int64_t* block_pairs,
                             int num_pairs, int num_kv_heads, int head_dim, int block_size,
                             int64_t num_blocks, int elem, void* stream) {
  if (num_pairs < 0 || num_kv_heads <= 0 || head_dim <= 0 || num_blocks <= 0) return PA_ERR_INVALID;
  if (block_size != kBlockSize) return PA_ERR_UNSUPPORTED;
  if ((head_dim * elem) % 16 != 0) return PA_ERR_UNSUPPORTED;
  if (num_pairs == 0) return PA_OK;
  if (num_pairs > 65535) return PA_ERR_UNSUPPORTED;
  if (!k_cache || !v_cache || !block_pairs) return PA_ERR_INVALID;
  if (!aligned(k_cache, 16) || !aligned(v_cache, 16) || !aligned(block_pairs, 8))
    return PA_ERR_INVALID;
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  const int64_t vec = static_cast<int64_t>(block_size) * num_kv_heads * head_dim * elem / 16;
  dim3 grid(static_cast<unsigned>((vec + 255) / 256 < 64 ? (vec + 255) / 256 : 64), num_pairs);
  copy_blocks_kernel<<<grid, 256, 0, static_cast<cudaStream_t>(stream)>>>(
      static_cast<uint4*>(k_cache), static_cast<uint4*>(v_cache), block_pairs, vec, num_blocks,
      d->err);
  return cudaGetLastError() == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

int pa_copy_blocks(void* k_cache, void* v_cache, const int64_t* block_pairs, int num_pairs,
                   int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                   void* stream) {
  return copy_blocks_bytes(k_cache, v_cache, block_pairs, num_pairs, num_kv_heads, head_dim,
                           block_size, num_blocks, 2, stream);
}

int pa_copy_blocks_fp8(void* k_cache, void* v_cache, const int64_t* block_pairs, int num_pairs,
                       int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                       void* stream) {
  return copy_blocks_bytes(k_cache, v_cache, block_pairs, num_pairs, num_kv_heads, head_dim,
                           block_size, num_blocks, 1, stream);
}

static int decode_mode(int partition_tokens) {
  return partition_tokens < 0 ? kModeSinglePass
                              : (partition_tokens == 0 ? kModeBalanced : kModeFixedSplit);
}

static size_t fixed_workspace_bytes(int num_seqs, int Hq, int D, int max_parts) {
  const size_t rows = static_cast<size_t>(num_seqs) * Hq * max_parts;
  const size_t o = (rows * D * 4 + 255) / 256 * 256;
  return o + (rows * 4 + 255) / 256 * 256;
}

size_t pa_decode_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                int max_blocks_per_seq, int block_size, int partition_tokens) {
  if (num_seqs < 0 || max_blocks_per_seq <= 0) return 0;
  if (check_shape(num_q_heads, num_kv_heads, head_dim, block_size) != PA_OK) return 0;
  const int mode = decode_mode(partition_tokens);
  if (mode == kModeSinglePass) return 0;
  if (mode == kModeFixedSplit) {
    if (partition_tokens % block_size) return 0;
    const int pb = partition_tokens / block_size;
    const int max_parts = (max_blocks_per_seq + pb - 1) / pb;
    return fixed_workspace_bytes(num_seqs, num_q_heads, head_dim, max_parts);
  }
  int num_sms = 0, dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess ||
      cudaDeviceGetAttribute(&num_sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess ||
      num_sms <= 0) {
    cudaGetLastError();
    num_sms = 1024;  // no device visible: an upper bound
  }
  // sized for the largest grid a launch may use: one CTA per SM
  return balanced_workspace_bytes(num_sms, num_q_heads, head_dim);
}

// Argument checks of a decode call (everything but the workspace), made
// before anything is enqueued.  PA_OK with num_seqs == 0: nothing to do.
static int decode_check(const void* out, const void* q, const void* k_cache, const void* v_cache,
                        const float* k_scales, const float* v_scales, bool kv_fp8,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* seq_lens, int num_seqs, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                        float scale, int partition_tokens, const float* out_lse,
                        bool append = false) {
  if (int rc = check_shape(num_q_heads, num_kv_heads, head_dim, block_size)) return rc;
  if (kv_fp8 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_seqs < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0) return PA_ERR_INVALID;
  if (num_blocks * kBlockSize > (int64_t)INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_ERR_INVALID;
  if (kv_fp8 && (!k_scales || !v_scales || !aligned(k_scales, 4) || !aligned(v_scales, 4)))
    return PA_ERR_INVALID;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16) ||
      !aligned(block_tables, 4) || !aligned(seq_lens, 4) || (out_lse && !aligned(out_lse, 4)))
    return PA_ERR_INVALID;
  const int mode = decode_mode(partition_tokens);
  if (mode == kModeFixedSplit && partition_tokens % block_size) return PA_ERR_INVALID;
  if (mode == kModeBalanced && num_seqs > kMaxSeqsBalanced) return PA_ERR_UNSUPPORTED;
  if (!decode_supported(head_dim, num_kv_heads, num_q_heads, mode, num_seqs, kv_fp8, append))
    return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// A launch's arguments and tensor maps, built by decode_impl / prefill_impl
// without launching when the hybrid call fuses the two into one kernel.
struct DecodePlan {
  DecodeArgs a;
  CUtensorMap tk, tv;
  int grid;
};
struct PrefillPlan {
  PrefillArgs a;
  CUtensorMap tq, tk, tv;
  CUtensorMap tnk, tnv;  // the chunks' new rows (append only)
  int tiles;
};

// pa_decode and pa_decode_fp8: the same launch; kv_fp8 selects E4M3 pools.
// plan non-null (balanced bf16 only): fill it and launch nothing.
static int decode_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                       const float* k_scales, const float* v_scales, bool kv_fp8,
                       const int32_t* block_tables, int max_blocks_per_seq,
                       const int32_t* seq_lens, int num_seqs, int num_q_heads,
                       int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                       float scale, int partition_tokens, float* out_lse, void* workspace,
                       size_t workspace_bytes, void* stream, const int32_t* start_blocks = nullptr,
                       const float* init_o = nullptr, const float* init_lse = nullptr,
                       int grid_override = 0, int stall_loads = 0, uint64_t wait_ns = 0,
                       const void* new_k = nullptr, const void* new_v = nullptr,
                       int64_t new_k_stride = 0, int64_t new_v_stride = 0,
                       DecodePlan* plan = nullptr) {
  if (int rc = decode_check(out, q, k_cache, v_cache, k_scales, v_scales, kv_fp8, block_tables,
                            max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, scale, partition_tokens, out_lse,
                            new_k != nullptr))
    return rc;
  if (num_seqs == 0) return PA_OK;
  if (kv_fp8 && init_o) return PA_ERR_UNSUPPORTED;  // no E4M3 cascade suffix pass
  const int mode = decode_mode(partition_tokens);
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;

  DecodeArgs a{};
  a.out = static_cast<__nv_bfloat16*>(out);
  a.q = static_cast<const __nv_bfloat16*>(q);
  a.block_tables = block_tables;
  a.seq_lens = seq_lens;
  a.out_lse = out_lse;
  a.err = d->err;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.num_seqs = num_seqs;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = num_q_heads / num_kv_heads;
  a.scale_log2 = scale * 1.4426950408889634f;
  a.mode = mode;
  a.kv_fp8 = kv_fp8 ? 1 : 0;
  a.k_scales = k_scales;
  a.v_scales = v_scales;
  a.start_blocks = start_blocks;
  a.init_o = init_o;
  a.init_lse = init_lse;
  a.stall_loads = stall_loads;
  a.wait_ns = wait_ns;  // 0: the default limit
  a.new_k = static_cast<const __nv_bfloat16*>(new_k);
  a.new_v = static_cast<const __nv_bfloat16*>(new_v);
  a.new_k_stride = new_k_stride;
  a.new_v_stride = new_v_stride;
  a.k_pool = static_cast<__nv_bfloat16*>(const_cast<void*>(k_cache));
  a.v_pool = static_cast<__nv_bfloat16*>(const_cast<void*>(v_cache));
  int grid = decode_grid(d->num_sms, mode, a.group, kv_fp8);
  if (grid_override > 0) grid = grid_override < d->num_sms ? grid_override : d->num_sms;
  if (mode == kModeSinglePass) {
    a.part_blocks = max_blocks_per_seq;
    a.max_parts = 1;
    if (num_seqs < grid) grid = num_seqs;
  } else if (mode == kModeFixedSplit) {
    a.part_blocks = partition_tokens / block_size;
    a.max_parts = (max_blocks_per_seq + a.part_blocks - 1) / a.part_blocks;
    const size_t need = fixed_workspace_bytes(num_seqs, num_q_heads, head_dim, a.max_parts);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
    const size_t rows = static_cast<size_t>(num_seqs) * num_q_heads * a.max_parts;
    a.part_o = static_cast<float*>(workspace);
    a.part_lse = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                          (rows * head_dim * 4 + 255) / 256 * 256);
    const int64_t units = static_cast<int64_t>(num_seqs) * a.max_parts;
    if (units < grid) grid = static_cast<int>(units);
  } else {
    const size_t need = balanced_workspace_bytes(grid, num_q_heads, head_dim);
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
    a.counters = static_cast<int*>(workspace);
    a.part_o = reinterpret_cast<float*>(static_cast<char*>(workspace) +
                                        (static_cast<size_t>(grid) * 4 + 255) / 256 * 256);
    a.slot_floats = static_cast<int>(balanced_slot_floats(num_q_heads, head_dim));
  }

  CUtensorMap tm_k, tm_v;
  const int elem = kv_fp8 ? 1 : 2;
  if (encode_pool_map(&tm_k, k_cache, num_blocks, num_kv_heads, head_dim, 0, elem) ||
      encode_pool_map(&tm_v, v_cache, num_blocks, num_kv_heads, head_dim, 0, elem))
    return PA_ERR_CUDA;
  if (plan) {
    if (mode != kModeBalanced || kv_fp8 || head_dim != 128) return PA_ERR_UNSUPPORTED;
    plan->a = a;
    plan->tk = tm_k;
    plan->tv = tm_v;
    plan->grid = grid;
    return PA_OK;
  }
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if (launch_decode(a, &tm_k, &tm_v, head_dim, grid, st) != cudaSuccess) return PA_ERR_CUDA;
  if (mode == kModeFixedSplit) {
    MergeArgs m{};
    m.out = a.out;
    m.out_lse = out_lse;
    m.part_o = a.part_o;
    m.part_lse = a.part_lse;
    m.num_parts = nullptr;
    m.seq_lens = seq_lens;
    m.part_blocks = a.part_blocks;
    m.max_blocks = max_blocks_per_seq;
    m.skip_single = 1;
    m.start_blocks = start_blocks;
    m.num_seqs = num_seqs;
    m.num_q_heads = num_q_heads;
    m.head_dim = head_dim;
    m.max_parts = a.max_parts;
    if (launch_merge(m, st) != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

int pa_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
              const int32_t* block_tables, int max_blocks_per_seq, const int32_t* seq_lens,
              int num_seqs, int num_q_heads, int num_kv_heads, int head_dim, int block_size,
              int64_t num_blocks, float scale, int partition_tokens, float* out_lse,
              void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(out, q, k_cache, v_cache, nullptr, nullptr, false, block_tables,
                     max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, scale, partition_tokens, out_lse, workspace,
                     workspace_bytes, stream);
}

int pa_decode_append(void* out, const void* q, const void* key, const void* value,
                     int64_t key_token_stride, int64_t value_token_stride, void* k_cache,
                     void* v_cache, const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                     int head_dim, int block_size, int64_t num_blocks, float scale,
                     int partition_tokens, float* out_lse, void* workspace,
                     size_t workspace_bytes, void* stream) {
  if (num_seqs > 0) {
    const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
    if (!key || !value || !aligned(key, 16) || !aligned(value, 16)) return PA_ERR_INVALID;
    if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 ||
        value_token_stride % 8)
      return PA_ERR_INVALID;
  }
  return decode_impl(out, q, k_cache, v_cache, nullptr, nullptr, false, block_tables,
                     max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, scale, partition_tokens, out_lse, workspace,
                     workspace_bytes, stream, nullptr, nullptr, nullptr, 0, 0, 0, key, value,
                     key_token_stride, value_token_stride);
}

int pa_decode_fp8(void* out, const void* q, const void* k_cache, const void* v_cache,
                  const float* k_scales, const float* v_scales, const int32_t* block_tables,
                  int max_blocks_per_seq, const int32_t* seq_lens, int num_seqs,
                  int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                  int64_t num_blocks, float scale, int partition_tokens, float* out_lse,
                  void* workspace, size_t workspace_bytes, void* stream) {
  return decode_impl(out, q, k_cache, v_cache, k_scales, v_scales, true, block_tables,
                     max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, scale, partition_tokens, out_lse, workspace,
                     workspace_bytes, stream);
}

// Cascade workspace before the decode's: the prefix result (o [S, Hq, 128],
// lse [S, Hq]), the partials of prefix parts 1.. (same shapes, each), and one
// ticket per (group, kv-head subset) -- at most S * Hkv of them.
static size_t round256(size_t b) { return (b + 255) / 256 * 256; }

static size_t cascade_prefix_bytes(int num_seqs, int Hq, int Hkv) {
  const size_t o = round256(static_cast<size_t>(num_seqs) * Hq * 128 * 4);
  const size_t l = round256(static_cast<size_t>(num_seqs) * Hq * 4);
  return (o + l) * kMaxPrefixParts + round256(static_cast<size_t>(num_seqs) * Hkv * 4);
}

size_t pa_cascade_workspace_size(int num_seqs, int num_q_heads, int num_kv_heads, int head_dim,
                                 int max_blocks_per_seq, int block_size, int partition_tokens) {
  if (head_dim != 128 || num_seqs < 0) return 0;
  if (check_shape(num_q_heads, num_kv_heads, head_dim, block_size) != PA_OK) return 0;
  return cascade_prefix_bytes(num_seqs, num_q_heads, num_kv_heads) +
         pa_decode_workspace_size(num_seqs, num_q_heads, num_kv_heads, head_dim,
                                  max_blocks_per_seq, block_size, partition_tokens);
}

int pa_cascade_decode(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* seq_lens, int num_seqs, const int32_t* group_offsets,
                      int num_groups, int max_group_size, const int32_t* prefix_tables,
                      int max_prefix_blocks, const int32_t* shared_blocks, int num_q_heads,
                      int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                      float scale, int partition_tokens, float* out_lse, void* workspace,
                      size_t workspace_bytes, void* stream) {
  if (int rc = check_shape(num_q_heads, num_kv_heads, head_dim, block_size)) return rc;
  if (head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (num_seqs < 0 || num_groups < 0 || max_blocks_per_seq <= 0 || num_blocks <= 0 ||
      max_prefix_blocks < 0)
    return PA_ERR_INVALID;
  if (num_blocks * kBlockSize > (int64_t)INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_INVALID;
  if (num_seqs == 0) return PA_OK;
  if (!group_offsets || !shared_blocks || (max_prefix_blocks > 0 && !prefix_tables) ||
      !aligned(group_offsets, 4) || !aligned(shared_blocks, 4) ||
      (prefix_tables && !aligned(prefix_tables, 4)))
    return PA_ERR_INVALID;
  CascadeArgs c{};
  if (!cascade_shape(num_kv_heads, num_q_heads / num_kv_heads, max_group_size, &c.kv_per_cta,
                     &c.warps_per_kv, &c.stages))
    return PA_ERR_UNSUPPORTED;
  const size_t pre = cascade_prefix_bytes(num_seqs, num_q_heads, num_kv_heads);
  if (!workspace || workspace_bytes < pre || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
  if (!out || !q || !k_cache || !v_cache || !block_tables || !seq_lens) return PA_ERR_INVALID;
  if (!aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16)) return PA_ERR_INVALID;
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  char* wsb = static_cast<char*>(workspace);
  const size_t o_bytes = round256(static_cast<size_t>(num_seqs) * num_q_heads * 128 * 4);
  const size_t l_bytes = round256(static_cast<size_t>(num_seqs) * num_q_heads * 4);
  float* pre_o = reinterpret_cast<float*>(wsb);
  float* pre_lse = reinterpret_cast<float*>(wsb + o_bytes);
  float* part_o = reinterpret_cast<float*>(wsb + o_bytes + l_bytes);
  float* part_lse = reinterpret_cast<float*>(wsb + o_bytes + l_bytes +
                                             (kMaxPrefixParts - 1) * o_bytes);
  int* tickets = reinterpret_cast<int*>(wsb + (o_bytes + l_bytes) * kMaxPrefixParts);
  if (num_groups > 0) {
    c.q = static_cast<const __nv_bfloat16*>(q);
    c.seq_lens = seq_lens;
    c.group_offsets = group_offsets;
    c.prefix_tables = prefix_tables;
    c.shared_blocks = shared_blocks;
    c.pre_o = pre_o;
    c.pre_lse = pre_lse;
    c.err = d->err;
    c.num_blocks = num_blocks;
    c.num_seqs = num_seqs;
    c.max_prefix_blocks = max_prefix_blocks;
    c.num_groups = num_groups;
    c.max_group = max_group_size;
    c.num_q_heads = num_q_heads;
    c.num_kv_heads = num_kv_heads;
    c.group = num_q_heads / num_kv_heads;
    c.scale_log2 = scale * 1.4426950408889634f;
    // too few (group, subset) units to fill the GPU: split each prefix over
    // up to kMaxPrefixParts CTAs
    const int units = num_groups * (num_kv_heads / c.kv_per_cta);
    c.parts = units >= d->num_sms ? 1 : d->num_sms / units;
    c.parts = c.parts < 1 ? 1 : (c.parts > kMaxPrefixParts ? kMaxPrefixParts : c.parts);
    if (static_cast<int64_t>(units) > static_cast<int64_t>(num_seqs) * num_kv_heads)
      c.parts = 1;  // more units than ticket slots: no split
    c.part_o = part_o;
    c.part_lse = part_lse;
    c.tickets = tickets;
    CUtensorMap tk, tv;
    if (encode_pool_map(&tk, k_cache, num_blocks, num_kv_heads, head_dim, -c.kv_per_cta) ||
        encode_pool_map(&tv, v_cache, num_blocks, num_kv_heads, head_dim, -c.kv_per_cta))
      return PA_ERR_CUDA;
    if (launch_cascade_prefix(c, &tk, &tv, static_cast<cudaStream_t>(stream)) != cudaSuccess)
      return PA_ERR_CUDA;
  }
  return decode_impl(out, q, k_cache, v_cache, nullptr, nullptr, false, block_tables,
                     max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, scale, partition_tokens, out_lse,
                     static_cast<char*>(workspace) + pre, workspace_bytes - pre, stream,
                     shared_blocks, pre_o, pre_lse);
}

// Static scratch of pa_decode_noalloc: the balanced split's merge tickets and
// partial slots, for callers that cannot allocate.  In host code the array's
// name is only a host-side stand-in; kernels get its device address, looked
// up once per device below.
static __device__ __align__(256) unsigned char g_noalloc_scratch[PA_NOALLOC_SCRATCH_BYTES];
static std::mutex g_noalloc_mu;
static void* g_noalloc_ptr[pa::kMaxDevices];

int pa_decode_noalloc(void* out, const void* q, const void* k_cache, const void* v_cache,
                      const int32_t* block_tables, int max_blocks_per_seq,
                      const int32_t* seq_lens, int num_seqs, int num_q_heads, int num_kv_heads,
                      int head_dim, int block_size, int64_t num_blocks, float scale,
                      float* out_lse, void* stream) {
  // every argument is checked before the scratch is touched: a rejected call
  // enqueues nothing
  if (int rc = decode_check(out, q, k_cache, v_cache, nullptr, nullptr, false, block_tables,
                            max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads,
                            head_dim, block_size, num_blocks, scale, 0, out_lse))
    return rc;
  if (num_seqs == 0) return PA_OK;
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  const size_t need = balanced_workspace_bytes(d->num_sms, num_q_heads, head_dim);
  if (need > PA_NOALLOC_SCRATCH_BYTES) return PA_ERR_SCRATCH_LIMIT;
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return PA_ERR_CUDA;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_noalloc_mu);
    if (!g_noalloc_ptr[dev]) {
      void* p = nullptr;
      if (cudaGetSymbolAddress(&p, g_noalloc_scratch) != cudaSuccess || p == nullptr)
        return PA_ERR_CUDA;
      g_noalloc_ptr[dev] = p;
    }
    scratch = g_noalloc_ptr[dev];
  }
  // the merge tickets must start at zero (the kernel leaves them zeroed, but a
  // call cut short by an error may not)
  const size_t tickets = (static_cast<size_t>(d->num_sms) * 4 + 255) / 256 * 256;
  if (cudaMemsetAsync(scratch, 0, tickets, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return PA_ERR_CUDA;
  return pa_decode(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, seq_lens, num_seqs,
                   num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, 0, out_lse,
                   scratch, PA_NOALLOC_SCRATCH_BYTES, stream);
}

int pa_merge_partials(void* out, float* out_lse, const float* part_out, const float* part_lse,
                      const int32_t* num_parts, int num_seqs, int num_q_heads, int head_dim,
                      int max_parts, void* stream) {
  if (num_seqs < 0 || num_q_heads <= 0 || max_parts <= 0) return PA_ERR_INVALID;
  if (head_dim != 64 && head_dim != 128) return PA_ERR_UNSUPPORTED;
  if (static_cast<int64_t>(num_seqs) * num_q_heads > INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (num_seqs == 0) return PA_OK;
  if (!out || !part_out || !part_lse || !num_parts) return PA_ERR_INVALID;
  if (!aligned(part_out, 16) || !aligned(part_lse, 4) || !aligned(num_parts, 4) ||
      !aligned(out, 4) || (out_lse && !aligned(out_lse, 4)))
    return PA_ERR_INVALID;
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  MergeArgs m{};
  m.out = static_cast<__nv_bfloat16*>(out);
  m.out_lse = out_lse;
  m.part_o = part_out;
  m.part_lse = part_lse;
  m.num_parts = num_parts;
  m.num_seqs = num_seqs;
  m.num_q_heads = num_q_heads;
  m.head_dim = head_dim;
  m.max_parts = max_parts;
  return launch_merge(m, static_cast<cudaStream_t>(stream)) == cudaSuccess ? PA_OK : PA_ERR_CUDA;
}

// Argument checks of a prefill-chunk call (PA_OK: launch it; done: nothing to do).
// SMs a hybrid step leaves to its chunk by default: about a seventh (22 of
// 152).  On the Sarathi batch (a 512-query chunk next to 128 decodes) this
// hides the chunk's tensor work under the decode's HBM streaming; the fused
// step measured 186.2-186.3 us at 22 SMs, 186.8-187.0 at 24-28 and 187.1 at
// 32.
static int default_chunk_sms(int num_sms) { return (num_sms * 29 + 100) / 200; }

static int prefill_check(const void* out, const void* q, const void* k_cache, const void* v_cache,
                         const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* cu_q_lens, const int32_t* q_start_pos,
                         const int32_t* seq_lens, int num_chunks, int total_q_tokens,
                         int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                         int block_size, int64_t num_blocks, float scale, bool* done) {
  *done = false;
  if (int rc = check_shape(num_q_heads, num_kv_heads, head_dim, block_size)) return rc;
  if (head_dim != 128) return PA_ERR_UNSUPPORTED;
  const int group = num_q_heads / num_kv_heads;
  if (128 % group != 0) return PA_ERR_UNSUPPORTED;
  if (num_chunks < 0 || total_q_tokens < 0 || max_q_len < 0 || max_blocks_per_seq <= 0 ||
      num_blocks <= 0)
    return PA_ERR_INVALID;
  if (num_blocks * kBlockSize > (int64_t)INT32_MAX) return PA_ERR_UNSUPPORTED;
  if (!(scale > 0.f) || !isfinite(scale)) return PA_ERR_INVALID;
  if (num_chunks == 0 || total_q_tokens == 0 || max_q_len == 0) {
    *done = true;
    return PA_OK;
  }
  if (!out || !q || !k_cache || !v_cache || !block_tables || !cu_q_lens || !q_start_pos ||
      !seq_lens)
    return PA_ERR_INVALID;
  if (!aligned(out, 16) || !aligned(q, 16) || !aligned(k_cache, 16) || !aligned(v_cache, 16))
    return PA_ERR_INVALID;
  const int tokens_per_tile = 128 / group;
  const int64_t tiles = static_cast<int64_t>((max_q_len + tokens_per_tile - 1) / tokens_per_tile +
                                             kMaxCluster) * num_chunks * num_kv_heads;
  if (tiles > INT32_MAX) return PA_ERR_UNSUPPORTED;
  return PA_OK;
}

// The chunk launch of pa_prefill_chunk; plan non-null: fill it and launch
// nothing (pa_hybrid_attention).
static int prefill_impl(void* out, const void* q, const void* k_cache, const void* v_cache,
                        const int32_t* block_tables, int max_blocks_per_seq,
                        const int32_t* cu_q_lens, const int32_t* q_start_pos,
                        const int32_t* seq_lens, int num_chunks, int total_q_tokens, int max_q_len,
                        int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                        int64_t num_blocks, float scale, float* out_lse, void* stream,
                        PrefillPlan* plan, int stall_loads = 0, uint64_t wait_ns = 0,
                        const void* new_k = nullptr, const void* new_v = nullptr,
                        int64_t new_k_stride = 0, int64_t new_v_stride = 0) {
  bool done = false;
  if (int rc = prefill_check(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq,
                             cu_q_lens, q_start_pos, seq_lens, num_chunks, total_q_tokens,
                             max_q_len, num_q_heads, num_kv_heads, head_dim, block_size,
                             num_blocks, scale, &done))
    return rc;
  if (done) return PA_OK;
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  const int group = num_q_heads / num_kv_heads;
  PrefillArgs a{};
  a.out = static_cast<__nv_bfloat16*>(out);
  a.block_tables = block_tables;
  a.cu_q_lens = cu_q_lens;
  a.q_start_pos = q_start_pos;
  a.seq_lens = seq_lens;
  a.out_lse = out_lse;
  a.err = d->err;
  a.num_blocks = num_blocks;
  a.max_blocks = max_blocks_per_seq;
  a.num_chunks = num_chunks;
  a.total_q = total_q_tokens;
  a.num_q_heads = num_q_heads;
  a.num_kv_heads = num_kv_heads;
  a.group = group;
  a.stall_loads = stall_loads;
  a.wait_ns = wait_ns;  // 0: the default limit
  a.new_k = static_cast<const __nv_bfloat16*>(new_k);
  a.new_v = static_cast<const __nv_bfloat16*>(new_v);
  a.new_k_stride = new_k_stride;
  a.new_v_stride = new_v_stride;
  a.k_pool = static_cast<__nv_bfloat16*>(const_cast<void*>(k_cache));
  a.v_pool = static_cast<__nv_bfloat16*>(const_cast<void*>(v_cache));
  const int tokens_per_tile = 128 / group;
  a.tiles_per_chunk = (max_q_len + tokens_per_tile - 1) / tokens_per_tile;
  // whole CTA pairs: an odd count gets one tile more, which has no rows
  a.tiles_per_chunk = (a.tiles_per_chunk + kMaxCluster - 1) / kMaxCluster * kMaxCluster;
  a.scale_log2 = scale * 1.4426950408889634f;
  CUtensorMap tm_q, tm_k, tm_v;
  if (encode_q_map(&tm_q, q, total_q_tokens, num_q_heads, head_dim, group, tokens_per_tile) ||
      encode_pool_map(&tm_k, k_cache, num_blocks, num_kv_heads, head_dim, kPoolKeyTile) ||
      encode_pool_map(&tm_v, v_cache, num_blocks, num_kv_heads, head_dim, kPool2D))
    return PA_ERR_CUDA;
  const int64_t tiles = static_cast<int64_t>(a.tiles_per_chunk) * num_chunks * num_kv_heads;
  if (plan) {
    plan->a = a;
    plan->tq = tm_q;
    plan->tk = tm_k;
    plan->tv = tm_v;
    plan->tnk = tm_k;  // not read without new rows
    plan->tnv = tm_v;
    if (new_k && encode_new_row_maps(&plan->tnk, &plan->tnv, new_k, new_v, total_q_tokens,
                                     num_kv_heads, new_k_stride, new_v_stride))
      return PA_ERR_CUDA;
    plan->tiles = static_cast<int>(tiles);
    return PA_OK;
  }
  if (new_k) return PA_ERR_INVALID;  // new rows go through the hybrid launch only
  return launch_prefill(a, &tm_q, &tm_k, &tm_v, static_cast<int>(tiles),
                        static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

int pa_prefill_chunk(void* out, const void* q, const void* k_cache, const void* v_cache,
                     const int32_t* block_tables, int max_blocks_per_seq,
                     const int32_t* cu_q_lens, const int32_t* q_start_pos,
                     const int32_t* seq_lens, int num_chunks, int total_q_tokens, int max_q_len,
                     int num_q_heads, int num_kv_heads, int head_dim, int block_size,
                     int64_t num_blocks, float scale, float* out_lse, void* stream) {
  return prefill_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, cu_q_lens,
                      q_start_pos, seq_lens, num_chunks, total_q_tokens, max_q_len, num_q_heads,
                      num_kv_heads, head_dim, block_size, num_blocks, scale, out_lse, stream,
                      nullptr);
}

size_t pa_hybrid_workspace_size(int num_decode_seqs, int num_q_heads, int num_kv_heads,
                                int head_dim, int max_blocks_per_seq, int block_size) {
  const size_t dec = pa_decode_workspace_size(num_decode_seqs, num_q_heads, num_kv_heads, head_dim,
                                              max_blocks_per_seq, block_size, 0);
  return dec == 0 ? 0 : 256 + dec;
}

int pa_hybrid_attention(void* out_chunk, const void* q_chunk, const int32_t* chunk_block_tables,
                        int chunk_max_blocks, const int32_t* cu_q_lens,
                        const int32_t* q_start_pos, const int32_t* chunk_seq_lens,
                        int num_chunks, int total_q_tokens, int max_q_len, float* chunk_lse,
                        void* out_decode, const void* q_decode,
                        const int32_t* decode_block_tables, int decode_max_blocks,
                        const int32_t* decode_seq_lens, int num_decode_seqs, float* decode_lse,
                        const void* k_cache, const void* v_cache, int num_q_heads,
                        int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                        float scale, int chunk_sms, void* workspace, size_t workspace_bytes,
                        void* stream) {
  bool no_chunk = false;
  if (int rc = prefill_check(out_chunk, q_chunk, k_cache, v_cache, chunk_block_tables,
                             chunk_max_blocks, cu_q_lens, q_start_pos, chunk_seq_lens, num_chunks,
                             total_q_tokens, max_q_len, num_q_heads, num_kv_heads, head_dim,
                             block_size, num_blocks, scale, &no_chunk))
    return rc;
  if (num_decode_seqs < 0 || chunk_sms < 0) return PA_ERR_INVALID;
  if (num_decode_seqs == 0)
    return no_chunk ? PA_OK
                    : prefill_impl(out_chunk, q_chunk, k_cache, v_cache, chunk_block_tables,
                                   chunk_max_blocks, cu_q_lens, q_start_pos, chunk_seq_lens,
                                   num_chunks, total_q_tokens, max_q_len, num_q_heads,
                                   num_kv_heads, head_dim, block_size, num_blocks, scale,
                                   chunk_lse, stream, nullptr);
  const size_t need = pa_hybrid_workspace_size(num_decode_seqs, num_q_heads, num_kv_heads,
                                               head_dim, decode_max_blocks, block_size);
  if (need == 0) return PA_ERR_INVALID;
  if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
  void* dec_ws = static_cast<char*>(workspace) + 256;
  const size_t dec_bytes = workspace_bytes - 256;
  if (no_chunk)
    return decode_impl(out_decode, q_decode, k_cache, v_cache, nullptr, nullptr, false,
                       decode_block_tables, decode_max_blocks, decode_seq_lens, num_decode_seqs,
                       num_q_heads, num_kv_heads, head_dim, block_size, num_blocks, scale, 0,
                       decode_lse, dec_ws, dec_bytes, stream);
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  if (d->num_sms < 4) return PA_ERR_UNSUPPORTED;
  // SMs left to the chunk (default_chunk_sms).  The decode takes an even
  // number of CTAs, so that the launch's clusters of two never mix the roles.
  int cs = chunk_sms > 0 ? chunk_sms : default_chunk_sms(d->num_sms);
  cs = cs < 1 ? 1 : (cs > d->num_sms - 2 ? d->num_sms - 2 : cs);
  const int decode_ctas = (d->num_sms - cs) & ~1;
  // the fused kernel holds the bf16 head_dim-128 decode only; the chunk
  // call's checks above already required head_dim 128
  DecodePlan dp;
  if (int rc = decode_impl(out_decode, q_decode, k_cache, v_cache, nullptr, nullptr, false,
                           decode_block_tables, decode_max_blocks, decode_seq_lens,
                           num_decode_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                           num_blocks, scale, 0, decode_lse, dec_ws, dec_bytes, stream, nullptr,
                           nullptr, nullptr, decode_ctas, 0, 0, nullptr, nullptr, 0, 0, &dp))
    return rc;
  PrefillPlan pp;
  if (int rc = prefill_impl(out_chunk, q_chunk, k_cache, v_cache, chunk_block_tables,
                            chunk_max_blocks, cu_q_lens, q_start_pos, chunk_seq_lens, num_chunks,
                            total_q_tokens, max_q_len, num_q_heads, num_kv_heads, head_dim,
                            block_size, num_blocks, scale, chunk_lse, stream, &pp))
    return rc;
  if (dp.grid != decode_ctas) return PA_ERR_UNSUPPORTED;
  return launch_hybrid(dp.a, &dp.tk, &dp.tv, pp.a, &pp.tq, &pp.tk, &pp.tv, &pp.tnk, &pp.tnv,
                       dp.grid, pp.tiles, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

int pa_hybrid_attention_append(
    void* out_chunk, const void* q_chunk, const void* key_chunk, const void* value_chunk,
    const int32_t* chunk_block_tables, int chunk_max_blocks, const int32_t* cu_q_lens,
    const int32_t* q_start_pos, const int32_t* chunk_seq_lens, int num_chunks,
    int total_q_tokens, int max_q_len, float* chunk_lse, void* out_decode, const void* q_decode,
    const void* key_decode, const void* value_decode, const int32_t* decode_block_tables,
    int decode_max_blocks, const int32_t* decode_seq_lens, int num_decode_seqs, float* decode_lse,
    int64_t key_token_stride, int64_t value_token_stride, void* k_cache, void* v_cache,
    int num_q_heads, int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
    float scale, int chunk_sms, void* workspace, size_t workspace_bytes, void* stream) {
  bool no_chunk = false;
  if (int rc = prefill_check(out_chunk, q_chunk, k_cache, v_cache, chunk_block_tables,
                             chunk_max_blocks, cu_q_lens, q_start_pos, chunk_seq_lens, num_chunks,
                             total_q_tokens, max_q_len, num_q_heads, num_kv_heads, head_dim,
                             block_size, num_blocks, scale, &no_chunk))
    return rc;
  if (num_decode_seqs < 0 || chunk_sms < 0) return PA_ERR_INVALID;
  const int64_t row = static_cast<int64_t>(num_kv_heads) * head_dim;
  if (key_token_stride < row || value_token_stride < row || key_token_stride % 8 ||
      value_token_stride % 8)
    return PA_ERR_INVALID;
  if (!no_chunk && (!key_chunk || !value_chunk || !aligned(key_chunk, 16) ||
                    !aligned(value_chunk, 16)))
    return PA_ERR_INVALID;
  if (num_decode_seqs > 0 && (!key_decode || !value_decode || !aligned(key_decode, 16) ||
                              !aligned(value_decode, 16)))
    return PA_ERR_INVALID;
  if (no_chunk)
    return pa_decode_append(out_decode, q_decode, key_decode, value_decode, key_token_stride,
                            value_token_stride, k_cache, v_cache, decode_block_tables,
                            decode_max_blocks, decode_seq_lens, num_decode_seqs, num_q_heads,
                            num_kv_heads, head_dim, block_size, num_blocks, scale, 0, decode_lse,
                            workspace ? static_cast<char*>(workspace) + 256 : nullptr,
                            workspace_bytes > 256 ? workspace_bytes - 256 : 0, stream);
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  if (d->num_sms < 4) return PA_ERR_UNSUPPORTED;
  PrefillPlan pp;
  if (int rc = prefill_impl(out_chunk, q_chunk, k_cache, v_cache, chunk_block_tables,
                            chunk_max_blocks, cu_q_lens, q_start_pos, chunk_seq_lens, num_chunks,
                            total_q_tokens, max_q_len, num_q_heads, num_kv_heads, head_dim,
                            block_size, num_blocks, scale, chunk_lse, stream, &pp, 0, 0,
                            key_chunk, value_chunk, key_token_stride, value_token_stride))
    return rc;
  DecodePlan dp;
  int decode_ctas = 0;
  if (num_decode_seqs > 0) {
    const size_t need = pa_hybrid_workspace_size(num_decode_seqs, num_q_heads, num_kv_heads,
                                                 head_dim, decode_max_blocks, block_size);
    if (need == 0) return PA_ERR_INVALID;
    if (!workspace || workspace_bytes < need || !aligned(workspace, 256)) return PA_ERR_WORKSPACE;
    // the SMs of the chunk as in pa_hybrid_attention
    int cs = chunk_sms > 0 ? chunk_sms : default_chunk_sms(d->num_sms);
    cs = cs < 1 ? 1 : (cs > d->num_sms - 2 ? d->num_sms - 2 : cs);
    decode_ctas = (d->num_sms - cs) & ~1;
    if (int rc = decode_impl(out_decode, q_decode, k_cache, v_cache, nullptr, nullptr, false,
                             decode_block_tables, decode_max_blocks, decode_seq_lens,
                             num_decode_seqs, num_q_heads, num_kv_heads, head_dim, block_size,
                             num_blocks, scale, 0, decode_lse, static_cast<char*>(workspace) + 256,
                             workspace_bytes - 256, stream, nullptr, nullptr, nullptr,
                             decode_ctas, 0, 0, key_decode, value_decode, key_token_stride,
                             value_token_stride, &dp))
      return rc;
    if (dp.grid != decode_ctas) return PA_ERR_UNSUPPORTED;
  } else {
    // no decodes: every CTA of the launch takes the prefill role
    dp.a = DecodeArgs{};
    dp.tk = pp.tk;
    dp.tv = pp.tv;
  }
  return launch_hybrid(dp.a, &dp.tk, &dp.tv, pp.a, &pp.tq, &pp.tk, &pp.tv, &pp.tnk, &pp.tnv,
                       decode_ctas, pp.tiles, static_cast<cudaStream_t>(stream)) == cudaSuccess
             ? PA_OK
             : PA_ERR_CUDA;
}

int pa_test_decode_stalled(void* out, const void* q, const void* k_cache, const void* v_cache,
                           const int32_t* block_tables, int max_blocks_per_seq,
                           const int32_t* seq_lens, int num_seqs, int num_q_heads,
                           int num_kv_heads, int head_dim, int block_size, int64_t num_blocks,
                           float scale, int partition_tokens, void* workspace,
                           size_t workspace_bytes, unsigned int wait_limit_us, void* stream) {
  if (wait_limit_us == 0 || wait_limit_us > 2000000u) return PA_ERR_INVALID;
  return decode_impl(out, q, k_cache, v_cache, nullptr, nullptr, false, block_tables,
                     max_blocks_per_seq, seq_lens, num_seqs, num_q_heads, num_kv_heads, head_dim,
                     block_size, num_blocks, scale, partition_tokens, nullptr, workspace,
                     workspace_bytes, stream, nullptr, nullptr, nullptr, 0, 1,
                     static_cast<uint64_t>(wait_limit_us) * 1000u);
}

int pa_test_prefill_stalled(void* out, const void* q, const void* k_cache, const void* v_cache,
                            const int32_t* block_tables, int max_blocks_per_seq,
                            const int32_t* cu_q_lens, const int32_t* q_start_pos,
                            const int32_t* seq_lens, int num_chunks, int total_q_tokens,
                            int max_q_len, int num_q_heads, int num_kv_heads, int head_dim,
                            int block_size, int64_t num_blocks, float scale,
                            unsigned int wait_limit_us, void* stream) {
  if (wait_limit_us == 0 || wait_limit_us > 2000000u) return PA_ERR_INVALID;
  return prefill_impl(out, q, k_cache, v_cache, block_tables, max_blocks_per_seq, cu_q_lens,
                      q_start_pos, seq_lens, num_chunks, total_q_tokens, max_q_len, num_q_heads,
                      num_kv_heads, head_dim, block_size, num_blocks, scale, nullptr, stream,
                      nullptr, 1, static_cast<uint64_t>(wait_limit_us) * 1000u);
}

int pa_validate_metadata(const int32_t* block_tables, int max_blocks_per_seq,
                         const int32_t* seq_lens, int num_seqs, const int64_t* slot_mapping,
                         int num_slots, const int32_t* refcount, int64_t num_blocks,
                         int block_size) {
  if (num_seqs < 0 || num_slots < 0 || num_blocks <= 0 || block_size <= 0) return PA_ERR_INVALID;
  if (num_seqs > 0 && !seq_lens) return PA_ERR_INVALID;
  for (int s = 0; s < num_seqs; ++s) {
    const int64_t n = seq_lens[s];
    if (n < 0 || n > static_cast<int64_t>(max_blocks_per_seq) * block_size) return PA_ERR_INVALID;
    if (block_tables) {
      const int64_t nb = (n + block_size - 1) / block_size;
      for (int64_t j = 0; j < nb; ++j) {
        const int64_t b = block_tables[static_cast<int64_t>(s) * max_blocks_per_seq + j];
        if (b < 0 || b >= num_blocks) return PA_ERR_INVALID;
      }
    }
  }
  if (slot_mapping && num_slots > 0) {
    std::unordered_set<int64_t> seen;
    seen.reserve(static_cast<size_t>(num_slots) * 2);
    for (int t = 0; t < num_slots; ++t) {
      const int64_t slot = slot_mapping[t];
      if (slot < 0) continue;
      if (slot >= num_blocks * block_size) return PA_ERR_INVALID;
      if (!seen.insert(slot).second) return PA_ERR_INVALID;
      if (refcount && refcount[slot / block_size] > 1) return PA_ERR_INVALID;
    }
  }
  return PA_OK;
}

int pa_device_error_flags(unsigned int* flags, int reset) {
  if (!flags) return PA_ERR_INVALID;
  DeviceInfo* d;
  if (int rc = current_device_info(&d)) return rc;
  if (cudaDeviceSynchronize() != cudaSuccess) return PA_ERR_CUDA;
  unsigned int v = 0;
  if (cudaMemcpy(&v, d->err, sizeof v, cudaMemcpyDeviceToHost) != cudaSuccess) return PA_ERR_CUDA;
  *flags = v;
  if (reset) {
    const unsigned int z = 0;
    if (cudaMemcpy(d->err, &z, sizeof z, cudaMemcpyHostToDevice) != cudaSuccess) return PA_ERR_CUDA;
  }
  return PA_OK;
}

}  // extern "C"
