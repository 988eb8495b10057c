// probe.cu — a read-bandwidth kernel for measuring the memory roof the decode
// runs against: when a K/V cache fits in L2 (129 MB on GB300), the decode
// steps read it from L2, whose bandwidth no library kernel reports.  Not part
// of the method; the bench calls it beside the timed job.
#include "../../include/h2o.h"
#include "common.cuh"

namespace h2o {
namespace {

constexpr int kProbeThreads = 512;
constexpr int kProbeUnroll = 8;

// Every thread reads 16-byte words of the buffer through L2 (ld.global.cg),
// kProbeUnroll loads in flight, `reps` sweeps; the XOR of what it read goes
// to `sink` only in the impossible case it matches a key, so the loads stay.
__global__ void __launch_bounds__(kProbeThreads) read_probe(const uint4 *__restrict__ buf, size_t n16, int reps,
                                                            uint32_t *sink) {
  const size_t stride = (size_t)gridDim.x * blockDim.x;
  uint32_t acc = 0u;
  for (int r = 0; r < reps; ++r) {
    size_t i = (size_t)blockIdx.x * blockDim.x + threadIdx.x;
    for (; i + (kProbeUnroll - 1) * stride < n16; i += kProbeUnroll * stride) {
      uint4 v[kProbeUnroll];
#pragma unroll
      for (int u = 0; u < kProbeUnroll; ++u) v[u] = ld_cg16(buf + i + u * stride);
#pragma unroll
      for (int u = 0; u < kProbeUnroll; ++u) acc ^= v[u].x ^ v[u].y ^ v[u].z ^ v[u].w;
    }
    for (; i < n16; i += stride) {
      const uint4 v = ld_cg16(buf + i);
      acc ^= v.x ^ v.y ^ v.z ^ v.w;
    }
  }
  if (acc == 0x9e3779b9u) sink[0] = acc;
}

}  // namespace
}  // namespace h2o

extern "C" h2o_status h2o_probe_read(const void *buf, size_t bytes, int reps, uint32_t *sink, void *cuda_stream) {
  if (!buf || !sink || reps < 1 || bytes < 16 || (bytes & 15) || ((uintptr_t)buf & 15)) return H2O_EINVAL;
  const int sms = h2o::num_sms_current_device();
  if (sms <= 0) return H2O_ECUDA;
  h2o::read_probe<<<4 * sms, h2o::kProbeThreads, 0, (cudaStream_t)cuda_stream>>>((const uint4 *)buf, bytes / 16,
                                                                                reps, sink);
  return cudaGetLastError() == cudaSuccess ? H2O_OK : H2O_ECUDA;
}
