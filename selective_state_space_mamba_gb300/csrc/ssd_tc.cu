// Tensor-core (tcgen05 / TMEM / TMA) kernels for the bf16 chunk contractions.
#include "ssm_internal.cuh"

namespace ssm {

bool ssd_tc_supported(const SsdDims&) { return false; }

cudaError_t launch_ssd_chunk_state_tc(const void*, const void*, const SsdDims&, const SsdWorkspace&, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_ssd_chunk_scan_tc(const void*, const void*, const void*, const float*, void*, const SsdDims&,
                                     const SsdWorkspace&, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace ssm
