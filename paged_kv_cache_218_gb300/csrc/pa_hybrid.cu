// pa_hybrid.cu -- one launch for a Sarathi hybrid batch ("03 - Engines
// Papers", section 3 Sarathi / Sarathi-Serve: prefill chunks and decodes in
// one step under a token budget; "The LLM inference engine playbook", Theme 1,
// chunked prefill co-scheduled with decodes).
//
// The launch's CTAs take one of two roles by their index: the first
// decode_ctas run the balanced paged decode of the batch's decodes (one CTA
// of decode_cta each, pa_decode_body.cuh), the rest run the chunks' query
// tiles as tcgen05 CTA pairs (prefill_cta<2>, pa_prefill_body.cuh).  The grid
// is launched in clusters of two, which the decode role ignores and which make
// the prefill role's CTAs pairs on the two SMs of a TPC; decode_ctas is even,
// so no cluster mixes the roles.  Blocks are dispatched in index order: the
// decode's CTAs (one per SM: their shared memory leaves room for no other CTA)
// take their SMs first and stream HBM, and the chunk's pairs run on the SMs
// they leave free, on tensor cores the decode does not use.  One launch
// completes when both roles have: the stream's order holds for the kernels
// after it with no hand-shake between the roles.
#include <mutex>

#include "pa_decode_body.cuh"
#include "pa_prefill_body.cuh"

namespace pa {
namespace {

constexpr int kHybridThreads = dec::kThreads > pre::kThreads ? dec::kThreads : pre::kThreads;

// AP: the step's slot scatter is fused in -- the decode role writes (and
// attends in place) each decode's new token, the prefill role writes its
// chunks' new rows and reads the chunks' own keys from them (nk, nv).
template <bool AP>
__global__ void __launch_bounds__(kHybridThreads, 1)
    hybrid_kernel(const __grid_constant__ CUtensorMap dk, const __grid_constant__ CUtensorMap dv,
                  const DecodeArgs d, const __grid_constant__ CUtensorMap pq,
                  const __grid_constant__ CUtensorMap pk, const __grid_constant__ CUtensorMap pv,
                  const __grid_constant__ CUtensorMap nk, const __grid_constant__ CUtensorMap nv,
                  const PrefillArgs p, const int decode_ctas) {
  const int b = static_cast<int>(blockIdx.x);
  if (b < decode_ctas) {
    // the decode role uses its first dec::kThreads threads (its barriers
    // count exactly those)
    if (threadIdx.x < dec::kThreads) dec::decode_cta<128, false, AP>(dk, dv, d, b, decode_ctas);
  } else {
    pre::prefill_cta<2>(pq, pk, pv, nk, nv, p, b - decode_ctas);
  }
}

}  // namespace

cudaError_t launch_hybrid(DecodeArgs d, const CUtensorMap* dk, const CUtensorMap* dv,
                          const PrefillArgs& pargs, const CUtensorMap* pq, const CUtensorMap* pk,
                          const CUtensorMap* pv, const CUtensorMap* nk, const CUtensorMap* nv,
                          int decode_ctas, int prefill_ctas, cudaStream_t stream) {
  // append launches may have no decode CTAs (every CTA a prefill one)
  const bool ap = pargs.new_k != nullptr;
  if ((decode_ctas & 1) || (prefill_ctas & 1) || decode_ctas < 0 || prefill_ctas <= 0 ||
      (decode_ctas == 0 && !ap) || (decode_ctas > 0 && ap != (d.new_k != nullptr)))
    return cudaErrorInvalidValue;
  PrefillArgs p = pargs;
  if (p.wait_ns == 0) p.wait_ns = kWaitLimitNs;
  const size_t dsmem = decode_ctas > 0 ? decode_smem_bytes(d, 128) : 0;
  const size_t psmem = prefill_smem_bytes();
  const size_t smem = dsmem > psmem ? dsmem : psmem;
  static std::mutex mu;
  static bool set_for[2][64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!set_for[ap][dev]) {
      e = cudaFuncSetAttribute(ap ? hybrid_kernel<true> : hybrid_kernel<false>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
      set_for[ap][dev] = true;
    }
  }
  // a programmatic dependent of the kernel before it (the scatter, or the
  // previous step): both roles touch no global memory before
  // griddepcontrol.wait
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(decode_ctas + prefill_ctas);
  cfg.blockDim = dim3(kHybridThreads);
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
  const CUtensorMap* mk = ap ? nk : pk;  // not read without new rows
  const CUtensorMap* mv = ap ? nv : pv;
  e = ap ? cudaLaunchKernelEx(&cfg, hybrid_kernel<true>, *dk, *dv, d, *pq, *pk, *pv, *mk, *mv, p,
                              decode_ctas)
         : cudaLaunchKernelEx(&cfg, hybrid_kernel<false>, *dk, *dv, d, *pq, *pk, *pv, *mk, *mv, p,
                              decode_ctas);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace pa
