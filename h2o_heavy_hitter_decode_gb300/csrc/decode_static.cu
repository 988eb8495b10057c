// decode_static.cu — h2o_decode_step_static: the decode step with its scratch
// in a fixed device array instead of caller-provided workspace.
//
// For callers that cannot allocate device memory (see include/h2o.h).  The
// kernel is the regular decode kernel (decode.cu); only where its scratch
// lives differs.  Nothing here calls cudaMalloc, cudaFree or any allocating
// library routine.
#include <cuda.h>

#include <mutex>

#include "../../include/h2o.h"
#include "internal.h"

namespace {

constexpr size_t kScratchBytes = H2O_STATIC_SCRATCH_BYTES;
constexpr size_t kAlign = 256;
constexpr int kMaxDevices = 256;

// Split partials, logits, arrival counters and the flag of one call.  Shared by
// every call in the process; device code could name it directly, host code
// only through the address looked up per device below.
static __device__ __align__(256) unsigned char g_scratch[kScratchBytes];

std::mutex g_setup_mu;
void *g_scratch_addr[kMaxDevices];  // device address of g_scratch, per device
CUcontext g_scratch_ctx[kMaxDevices];  // the context that address belongs to

// The calling thread's current context (null if it cannot be read): the
// array's address is looked up again when a device is used under another
// context than the one it was looked up in (each context loads the library's
// module separately).
CUcontext current_context() {
  using Fn = CUresult (*)(CUcontext *);
  static Fn fn = nullptr;
  static bool tried = false;
  if (!tried) {  // under g_setup_mu
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuCtxGetCurrent", &p, 4000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (Fn)p;
  }
  CUcontext ctx = nullptr;
  if (!fn || fn(&ctx) != CUDA_SUCCESS) return nullptr;
  return ctx;
}

size_t up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool a16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

}  // namespace

extern "C" h2o_status h2o_decode_step_static(int B, int H, int d, int k_heavy, int k_local, h2o_dtype dtype,
                                             void *K, void *V, int32_t *pos, float *score, int n_valid,
                                             int64_t position, const void *q_t, const void *k_t,
                                             const void *v_t, void *out, int32_t *evicted,
                                             void *cuda_stream) {
  if (B < 1 || H < 1 || k_heavy < 0 || k_local < 0) return H2O_EINVAL;
  if ((int64_t)B * H > (1LL << 24)) return H2O_EINVAL;
  const int64_t k64 = (int64_t)k_heavy + k_local;
  if (k64 < 1 || k64 > (1 << 24)) return H2O_EINVAL;
  if (dtype != H2O_F32 && dtype != H2O_BF16) return H2O_EINVAL;
  if (d != 64 && d != 128) return H2O_EUNSUPPORTED;
  if (!K || !V || !pos || !score || !q_t || !k_t || !v_t || !out) return H2O_EINVAL;
  if (!a16(K) || !a16(V) || !a16(q_t) || !a16(k_t) || !a16(v_t) || !a16(out) || ((uintptr_t)pos & 3u) ||
      ((uintptr_t)score & 3u) || ((uintptr_t)evicted & 3u))
    return H2O_EINVAL;
  const int k = (int)k64, nh = B * H;
  if (n_valid < 0 || n_valid > k || position < 0 || position >= 0x7fffffffLL) return H2O_EINVAL;

  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return H2O_ECUDA;
  if (dev < 0 || dev >= kMaxDevices) return H2O_EUNSUPPORTED;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || sms <= 0)
    return H2O_ECUDA;
  const int ns = h2o::decode_splits(nh, k, sms);

  // Carve the fixed array like a cache workspace's scratch sections.
  const size_t off_part = 0;
  const size_t off_logits = up(off_part + (size_t)nh * ns * (2 + d) * sizeof(float));
  const size_t off_counter = up(off_logits + (size_t)nh * (k + 1) * sizeof(float));
  const size_t off_err = off_counter + (size_t)nh * sizeof(int);
  const size_t need = up(off_err + sizeof(int));
  if (need > kScratchBytes) return H2O_EINVAL;  // shape too large for the fixed scratch

  void *base = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_setup_mu);
    // cudaGetDevice above made the runtime's context for `dev` current.
    const CUcontext ctx = current_context();
    if (!g_scratch_addr[dev] || ctx != g_scratch_ctx[dev]) {
      void *p = nullptr;
      if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || !p) return H2O_ECUDA;
      g_scratch_addr[dev] = p;
      g_scratch_ctx[dev] = ctx;
    }
    base = g_scratch_addr[dev];
  }
  char *s = (char *)base;
  cudaStream_t st = (cudaStream_t)cuda_stream;

  h2o::CacheView c;
  c.nh = nh; c.d = d; c.k = k; c.kh = k_heavy; c.kl = k_local;
  c.dtype = dtype == H2O_BF16 ? 1 : 0;
  c.K = K; c.V = V; c.pos = pos; c.score = score;
  c.part = (float *)(s + off_part);
  c.logits = (float *)(s + off_logits);
  c.counter = (int *)(s + off_counter);
  c.err = (int *)(s + off_err);
  c.done = nullptr;  // single steps only
  c.nsplit = ns;

  // The arrival counters (and the flag right after them) must start at zero;
  // a previous call may have been cut short, so clear them every time.
  if (cudaMemsetAsync(c.counter, 0, off_err + sizeof(int) - off_counter, st) != cudaSuccess) return H2O_ECUDA;

  h2o::DecodeStep step;
  step.q = q_t; step.kn = k_t; step.vn = v_t; step.out = out;
  step.evicted = evicted;
  step.n_valid = n_valid;
  step.p = (int)position;
  if (h2o::launch_decode_step(c, step, st) != cudaSuccess) return H2O_ECUDA;
  return H2O_OK;
}
