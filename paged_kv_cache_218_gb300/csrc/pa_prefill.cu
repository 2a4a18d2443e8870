// pa_prefill.cu -- causal paged prefill chunks on tcgen05 (placeholder until
// the tensor-core kernel lands; reports "not supported").
#include "pa_internal.h"

namespace pa {
size_t prefill_smem_bytes() { return 0; }
cudaError_t launch_prefill(const PrefillArgs&, const CUtensorMap*, const CUtensorMap*,
                           const CUtensorMap*, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
}  // namespace pa
