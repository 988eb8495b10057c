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
  int *done;         // [nh]                  per-head step flags of a persistent decode launch
  int nsplit;
  int n_sink = 0;      // positions 0 .. n_sink-1 are never evicted (pinned attention sinks)
  int score_mode = 0;  // 0: rank by accumulated score; 1: by score / queries that attended
  // fp8 cache (inputs bf16): K, V hold e4m3 codes [nh][k][d] and each row has
  // one fp32 scale, Ksc / Vsc [nh][k]; a row reads back as code * scale.
  int kv_fp8 = 0;
  float *Ksc = nullptr, *Vsc = nullptr;
};

struct DecodeStep {
  const void *q, *kn, *vn;  // [nh][d] in the input type (bf16 or fp32)
  void *out;                // [nh][d]
  int32_t *evicted;         // [nh] or nullptr
  int n_valid;              // filled slots before this step
  int p;                    // position of the new token
};

// Decode: one launch per step (split-K + last-arriver combine, score
// update, argmin, in-place write).
cudaError_t launch_decode_step(const CacheView &c, const DecodeStep &s, cudaStream_t st);
// Persistent multi-step decode: one cooperative grid runs `nsteps` steps
// (all (head, split) CTAs resident; per-head release/acquire step flags in
// `done`, zeroed by the launcher).  decode_persistent_fits says whether the
// grid can be co-resident on the current device.
bool decode_persistent_fits(const CacheView &c);
cudaError_t launch_decode_persistent(const CacheView &c, const DecodeStep &s, int nsteps, int *done,
                                     cudaStream_t st);
// Multi-step decode with one thread-block cluster per head (c.nsplit CTAs,
// at most 8): scores/tags/logits in shared memory, DSMEM pushes completing on
// the receivers' mbarriers; no global scratch.
bool decode_cluster_supported(const CacheView &c);
// CTAs per head (cluster size, 1..8) of the cluster form for nh heads of k
// slots on `sms` SMs.
int decode_cluster_size(int nh, int k, int sms);
cudaError_t launch_decode_cluster(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st);
// The cluster form with each step's eviction decision taken while the next
// step's attention pass runs (decode_pipe.cu); same cluster size and layout.
bool decode_pipe_supported(const CacheView &c);
int decode_pipe_cluster_size(const CacheView &c, int sms);  // CTAs per head of the pipelined form
cudaError_t launch_decode_pipe(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st);
// Split count of the decode launch for nh heads of k slots on `sms` SMs
// (fixes the size of the split-partial scratch).
int decode_splits(int nh, int k, int sms);

// Prefill pass 1 (causal attention -> O, lse) and pass 2 (column sums).
cudaError_t launch_prefill_attn(const CacheView &c, const void *Q, const void *K, const void *V,
                                void *O, float *lse, int L, cudaStream_t st);
cudaError_t launch_prefill_colsum(const CacheView &c, const void *Q, const void *K,
                                  const float *lse, float *colsum, int L, cudaStream_t st);
// Prefill select + gather into the cache slots.
cudaError_t launch_prefill_select(const CacheView &c, const void *K, const void *V,
                                  const float *colsum, int L, cudaStream_t st);

int num_sms_current_device();

// cudaFuncGetAttributes of a library kernel on the current device.
cudaError_t kernel_attributes(cudaFuncAttributes *a);

}  // namespace h2o
