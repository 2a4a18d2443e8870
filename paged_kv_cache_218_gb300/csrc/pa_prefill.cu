// pa_prefill.cu -- the prefill-chunk launch: CTA pairs of prefill_cta
// (pa_prefill_body.cuh), one per two query tiles.
#include <mutex>

#include "pa_prefill_body.cuh"

namespace pa {
namespace pre {
namespace {

template <int kPair>
__global__ void __launch_bounds__(kThreads, 1)
    prefill_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_k,
                   const __grid_constant__ CUtensorMap tm_v, const PrefillArgs a) {
  // no new rows here (a.new_k is null): the new-row maps are not read
  prefill_cta<kPair>(tm_q, tm_k, tm_v, tm_k, tm_v, a, static_cast<int>(blockIdx.x));
}

}  // namespace
}  // namespace pre

using namespace pre;

size_t prefill_smem_bytes() { return Plan<2>::kSmemBytes + 1024; }

cudaError_t launch_prefill(const PrefillArgs& args, const CUtensorMap* tm_q,
                           const CUtensorMap* tm_k, const CUtensorMap* tm_v, int grid_tiles,
                           cudaStream_t stream) {
  PrefillArgs a = args;
  if (a.wait_ns == 0) a.wait_ns = kWaitLimitNs;
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
      e = cudaFuncSetAttribute(prefill_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      set_for[dev] = true;
    }
  }
  // programmatic dependent launch: the CTAs may start while the previous
  // kernel on the stream finishes; they touch no global memory before
  // griddepcontrol.wait.  Clusters of two: the CTA pairs.
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid_tiles);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 2;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  e = cudaLaunchKernelEx(&cfg, prefill_kernel<2>, *tm_q, *tm_k, *tm_v, a);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
