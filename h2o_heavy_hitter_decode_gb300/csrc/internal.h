// internal.h — host-side launcher interface between the C ABI (api.cu) and
// the kernel translation units.  Not part of the public ABI.
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

namespace h2o {

// Device view of one cache's workspace.
struct CacheView {
  int nh, d, k, kh, kl;
  int dtype;  // 0 fp32, 1 bf16
  void *K, *V;       // [nh][k][d]
  int32_t *pos;      // [nh][k]
  float *score;      // [nh][k]
  float *part;       // [nh][nsplit][2 + d]  split partials (m, l, acc[d])
  float *logits;     // [nh][k + 1]           log2-domain logits of the step
  int *counter;      // [nh]                  split arrival counters (zero between launches)
  int *err;          // [1]                   sticky device error flag
  int nsplit;
};

struct DecodeStep {
  const void *q, *kn, *vn;  // [nh][d]
  void *out;                // [nh][d]
  int32_t *evicted;         // [nh] or nullptr
  int n_valid;              // filled slots before this step
  int p;                    // position of the new token
};

// Decode: one launch per step (split-K + last-arriver combine, score
// update, argmin, in-place write).
cudaError_t launch_decode_step(const CacheView &c, const DecodeStep &s, cudaStream_t st);

// Prefill pass 1 (causal attention -> O, lse) and pass 2 (column sums).
cudaError_t launch_prefill_attn(const CacheView &c, const void *Q, const void *K, const void *V,
                                void *O, float *lse, int L, cudaStream_t st);
cudaError_t launch_prefill_colsum(const CacheView &c, const void *Q, const void *K,
                                  const float *lse, float *colsum, int L, cudaStream_t st);
// Prefill select + gather into the cache slots.
cudaError_t launch_prefill_select(const CacheView &c, const void *K, const void *V,
                                  const float *colsum, int L, cudaStream_t st);

int num_sms_current_device();

}  // namespace h2o
