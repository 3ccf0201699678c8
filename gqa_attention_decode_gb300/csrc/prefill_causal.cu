// prefill_causal.cu -- causal GQA prefill (placeholder until the tcgen05 kernel lands).
#include "kernels.h"

namespace gqa {
cudaError_t prefill_prepare_device() { return cudaSuccess; }
cudaError_t prefill_launch(const PrefillLaunch &, cudaStream_t, PFN_cuTensorMapEncodeTiled_v12000) {
  return cudaErrorNotSupported;
}
}  // namespace gqa
