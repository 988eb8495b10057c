// prefill_tc.cu — tensor-core (tcgen05 / TMEM) prefill passes for bf16.
#include "common.cuh"

namespace h2o {

bool prefill_tc_supported(const CacheView &, int) { return false; }

cudaError_t launch_prefill_attn_tc(const CacheView &, const void *, const void *, const void *, void *,
                                   float *, int, cudaStream_t) {
  return cudaErrorNotSupported;
}
cudaError_t launch_prefill_colsum_tc(const CacheView &, const void *, const void *, const float *, float *,
                                     int, cudaStream_t) {
  return cudaErrorNotSupported;
}

}  // namespace h2o
