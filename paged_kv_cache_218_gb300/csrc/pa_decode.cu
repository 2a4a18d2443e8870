// pa_decode.cu -- the decode launches: the decode kernel (one CTA of
// decode_cta per block, pa_decode_body.cuh) and its launcher.
#include <mutex>

#include "pa_decode_body.cuh"

namespace pa {
namespace dec {
namespace {

template <int D, bool KV8, bool AP>
__global__ void __launch_bounds__(kThreads, 1)
    decode_kernel(const __grid_constant__ CUtensorMap tm_k, const __grid_constant__ CUtensorMap tm_v,
                  const DecodeArgs a) {
  decode_cta<D, KV8, AP>(tm_k, tm_v, a, static_cast<int>(blockIdx.x), static_cast<int>(gridDim.x));
}

}  // namespace
}  // namespace dec

using namespace dec;

size_t balanced_slot_floats(int num_q_heads, int head_dim) {
  const size_t f = static_cast<size_t>(num_q_heads) * (head_dim + 1);
  return (f + 63) / 64 * 64;
}

size_t balanced_workspace_bytes(int grid, int num_q_heads, int head_dim) {
  const size_t counters = (static_cast<size_t>(grid) * 4 + 255) / 256 * 256;
  return counters + static_cast<size_t>(grid) * 2 * balanced_slot_floats(num_q_heads, head_dim) * 4;
}

int decode_grid(int num_sms, int mode, int group, bool kv_fp8) {
  // The balanced bf16 decode with up to 4 q heads per kv head streams fastest
  // from about four fifths of the SMs: fewer block streams in flight contend
  // less in HBM (measured on GB300, 120 of 152 CTAs against all 152: 2-3 %
  // shorter on the Llama-3-8B decode layer, the long-context batch and the
  // hybrid batch's decodes).  Larger groups and E4M3 pools do more arithmetic
  // per byte and use every SM.
  if (mode == kModeBalanced && !kv_fp8 && group <= 4) return max(1, (num_sms * 79 + 50) / 100);
  return num_sms;
}

bool decode_supported(int head_dim, int num_kv_heads, int num_q_heads, int mode, int num_seqs,
                      bool kv_fp8, bool append) {
  if (num_kv_heads > kConsumerWarps) return false;
  if (kv_fp8 && (head_dim != 128 || append)) return false;
  const int pre = mode == kModeBalanced ? balanced_pre_ints(num_seqs) : 0;
  const int wph = warps_per_head(num_kv_heads);
  return make_layout(head_dim, num_kv_heads, num_q_heads, wph, 2, pre, kv_fp8 ? 1 : 2, append)
             .total <= 227 * 1024 - 1024;
}

// Balanced split: a sequence's fixed cost in blocks -- about the time its
// piece takes outside the block loop (query fragments, partial result, merge
// ticket) over the time of one block of streaming.
static int piece_cost(bool kv_fp8) { return kv_fp8 ? 4 : 1; }

size_t decode_smem_bytes(DecodeArgs& a, int head_dim) {
  const int pre = a.mode == kModeBalanced ? balanced_pre_ints(a.num_seqs) : 0;
  const int elem = a.kv_fp8 ? 1 : 2;
  if (a.wait_ns == 0) a.wait_ns = kWaitLimitNs;
  a.warps_per_head = warps_per_head(a.num_kv_heads);
  const bool append = a.new_k != nullptr;
  a.stages = pick_stages(head_dim, a.num_kv_heads, a.num_q_heads, pre, elem, append);
  a.piece_cost = piece_cost(a.kv_fp8 != 0);
  return make_layout(head_dim, a.num_kv_heads, a.num_q_heads, a.warps_per_head, a.stages, pre,
                     elem, append).total +
         1024;
}

cudaError_t launch_decode(DecodeArgs a, const CUtensorMap* tm_k, const CUtensorMap* tm_v,
                          int head_dim, int grid, cudaStream_t stream) {
  const size_t smem = decode_smem_bytes(a, head_dim);
  const bool append = a.new_k != nullptr;
  void (*kern)(const CUtensorMap, const CUtensorMap, const DecodeArgs) =
      a.kv_fp8 ? decode_kernel<128, true, false>
      : append ? (head_dim == 128 ? decode_kernel<128, false, true> : decode_kernel<64, false, true>)
               : (head_dim == 128 ? decode_kernel<128, false, false>
                                  : decode_kernel<64, false, false>);
  // raise the kernel's dynamic shared-memory limit once per device
  static std::mutex mu;
  static int set_for[5][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    int& done = set_for[a.kv_fp8 ? 2 : (head_dim == 128 ? 1 : 0) + (append ? 3 : 0)][dev];
    if (done < static_cast<int>(smem)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               227 * 1024);
      if (e != cudaSuccess) return e;
      done = 227 * 1024;
    }
  }
  // programmatic dependent launch: the CTAs may start while the previous
  // kernel on the stream finishes; they touch no global memory before
  // griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  e = cudaLaunchKernelEx(&cfg, kern, *tm_k, *tm_v, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
