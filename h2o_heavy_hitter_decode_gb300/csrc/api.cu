// api.cu — the C ABI declared in include/h2o.h.
//
// Host-side bookkeeping only: argument checks, the workspace carve-up, the
// per-cache counters (next position, filled slots) and the launch sequence.
// Every step of the method runs in the kernels of decode.cu, prefill_*.cu and
// select.cu.
#include <cstdint>
#include <cstdlib>
#include <cstring>
#include <new>
#include <vector>

#include "../../include/h2o.h"
#include "internal.h"

namespace h2o {
cudaError_t launch_prefill_attn_simt(const CacheView &c, const void *Q, const void *K, const void *V,
                                     void *O, float *lse, int L, cudaStream_t st);
cudaError_t launch_prefill_colsum_simt(const CacheView &c, const void *Q, const void *K, const float *lse,
                                       float *colsum, int L, cudaStream_t st);
bool prefill_tc_supported(const CacheView &c, int L);
cudaError_t launch_prefill_attn_tc(const CacheView &c, const void *Q, const void *K, const void *V,
                                   void *O, float *lse, int L, cudaStream_t st);
cudaError_t launch_prefill_colsum_tc(const CacheView &c, const void *Q, const void *K, const float *lse,
                                     float *colsum, int L, cudaStream_t st);
}  // namespace h2o

using namespace h2o;

struct h2o_cache {
  int B, H, d, kh, kl, k, nh;
  h2o_dtype dtype;
  int esize;  // bytes per input / output element
  int ssize;  // bytes per stored K/V element (1 for an fp8 cache)
  int64_t next_pos;
  int n_valid;
  bool prefilled;
  std::vector<char> row_done;  // batch rows prefilled so far (h2o_prefill_rows)
  int rows_done = 0;
  int prefill_L = 0;           // prompt length shared by every row
  cudaStream_t stream;
  int device;
  CacheView view;
  int decode_form = 0;  // h2o_set_decode_form
  int form_used = 0;    // form of the last decode call
  // phase timing (h2o_profile_enable / h2o_profile_read)
  bool profiling = false;
  struct Mark {
    int phase;
    int64_t launches;
    cudaEvent_t a, b;
  };
  std::vector<Mark> marks;
};

namespace {

thread_local int g_last_cuda = 0;

constexpr size_t kAlign = 256;
constexpr int64_t kMaxPos = 0x7fffffffLL;  // positions are int32 tags

size_t align_up(size_t x) { return (x + kAlign - 1) & ~(kAlign - 1); }

bool shape_ok(int B, int H, int d, int kh, int kl, h2o_dtype dt) {
  if (B < 1 || H < 1 || kh < 0 || kl < 0) return false;
  if ((int64_t)kh + kl < 1 || (int64_t)kh + kl > (1 << 24)) return false;
  if ((int64_t)B * H > (1LL << 24)) return false;
  if (dt != H2O_F32 && dt != H2O_BF16 && dt != H2O_BF16_FP8KV) return false;
  return d >= 1;
}

bool d_supported(int d) { return d == 64 || d == 128; }

int choose_nsplit(int nh, int k, int sms) { return h2o::decode_splits(nh, k, sms); }

struct Layout {
  size_t K, V, pos, score, Ksc, Vsc, part, logits, counter, done, err, total;
};

int input_size(h2o_dtype dt) { return dt == H2O_F32 ? 4 : 2; }
int stored_size(h2o_dtype dt) { return dt == H2O_F32 ? 4 : dt == H2O_BF16 ? 2 : 1; }

Layout layout(int nh, int k, int d, h2o_dtype dt, int nsplit) {
  Layout l;
  const int ssize = stored_size(dt);
  const size_t scales = dt == H2O_BF16_FP8KV ? (size_t)nh * k * sizeof(float) : 0;
  size_t o = 0;
  l.K = o;       o = align_up(o + (size_t)nh * k * d * ssize);
  l.V = o;       o = align_up(o + (size_t)nh * k * d * ssize);
  l.pos = o;     o = align_up(o + (size_t)nh * k * sizeof(int32_t));
  l.score = o;   o = align_up(o + (size_t)nh * k * sizeof(float));
  l.Ksc = o;     o = align_up(o + scales);
  l.Vsc = o;     o = align_up(o + scales);
  l.part = o;    o = align_up(o + (size_t)nh * nsplit * (2 + d) * sizeof(float));
  l.logits = o;  o = align_up(o + (size_t)nh * (k + 1) * sizeof(float));
  l.counter = o; o = align_up(o + (size_t)nh * sizeof(int));
  l.done = o;    o = align_up(o + (size_t)nh * sizeof(int));
  l.err = o;     o = align_up(o + sizeof(int));
  l.total = o;
  return l;
}

h2o_status cuda_fail(cudaError_t e) {
  g_last_cuda = (int)e;
  return H2O_ECUDA;
}

bool aligned16(const void *p) { return ((uintptr_t)p & 15u) == 0; }

// Brackets one phase with events on the cache's stream when profiling is on.
struct PhaseTimer {
  h2o_cache *c;
  h2o_cache::Mark m{};
  bool on = false;
  PhaseTimer(h2o_cache *c_, int phase, int64_t launches) : c(c_) {
    if (!c->profiling) return;
    m.phase = phase;
    m.launches = launches;
    if (cudaEventCreate(&m.a) != cudaSuccess) return;
    if (cudaEventCreate(&m.b) != cudaSuccess) {
      cudaEventDestroy(m.a);
      return;
    }
    on = cudaEventRecord(m.a, c->stream) == cudaSuccess;
  }
  void done() {
    if (!on) return;
    cudaEventRecord(m.b, c->stream);
    c->marks.push_back(m);
    on = false;
  }
  ~PhaseTimer() {
    if (on) {  // error path: nothing to keep
      cudaEventDestroy(m.a);
      cudaEventDestroy(m.b);
    }
  }
};

}  // namespace

namespace h2o {
int num_sms_current_device() {
  int dev = 0, sms = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  return sms;
}
}  // namespace h2o

extern "C" {

size_t h2o_cache_workspace_bytes(int B, int H, int d, int k_heavy, int k_local, h2o_dtype dtype) {
  if (!shape_ok(B, H, d, k_heavy, k_local, dtype) || !d_supported(d)) return 0;
  const int sms = num_sms_current_device();
  if (sms <= 0) return 0;
  const int nh = B * H, k = k_heavy + k_local;
  return layout(nh, k, d, dtype, choose_nsplit(nh, k, sms)).total;
}

h2o_status h2o_cache_create(int B, int H, int d, int k_heavy, int k_local, h2o_dtype dtype,
                            void *workspace, void *cuda_stream, h2o_cache_t *out) {
  if (!out) return H2O_EINVAL;
  *out = nullptr;
  if (!shape_ok(B, H, d, k_heavy, k_local, dtype)) return H2O_EINVAL;
  if (!d_supported(d)) return H2O_EUNSUPPORTED;
  if (!workspace || ((uintptr_t)workspace & (kAlign - 1))) return H2O_EINVAL;
  const int sms = num_sms_current_device();
  if (sms <= 0) return cuda_fail(cudaGetLastError());
  h2o_cache *c = new (std::nothrow) h2o_cache();
  if (!c) return H2O_ENOMEM;
  c->B = B; c->H = H; c->d = d; c->kh = k_heavy; c->kl = k_local;
  c->k = k_heavy + k_local; c->nh = B * H; c->dtype = dtype;
  c->esize = input_size(dtype);
  c->ssize = stored_size(dtype);
  c->next_pos = 0; c->n_valid = 0; c->prefilled = false;
  c->stream = (cudaStream_t)cuda_stream;
  cudaGetDevice(&c->device);
  const int ns = choose_nsplit(c->nh, c->k, sms);
  const Layout l = layout(c->nh, c->k, d, dtype, ns);
  char *w = (char *)workspace;
  CacheView &v = c->view;
  v.nh = c->nh; v.d = d; v.k = c->k; v.kh = k_heavy; v.kl = k_local;
  v.dtype = dtype == H2O_F32 ? 0 : 1;  // input type: fp32 or bf16
  v.kv_fp8 = dtype == H2O_BF16_FP8KV ? 1 : 0;
  if (v.kv_fp8) {
    v.Ksc = (float *)(w + l.Ksc);
    v.Vsc = (float *)(w + l.Vsc);
  }
  v.K = w + l.K; v.V = w + l.V;
  v.pos = (int32_t *)(w + l.pos); v.score = (float *)(w + l.score);
  v.part = (float *)(w + l.part); v.logits = (float *)(w + l.logits);
  v.counter = (int *)(w + l.counter); v.err = (int *)(w + l.err);
  v.done = (int *)(w + l.done);
  v.nsplit = ns;
  // Empty slots: pos = -1 (all bits set), score = 0, counters and flag 0.
  cudaError_t e = cudaMemsetAsync(v.pos, 0xff, (size_t)c->nh * c->k * sizeof(int32_t), c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(v.score, 0, (size_t)c->nh * c->k * sizeof(float), c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(v.counter, 0, (size_t)c->nh * sizeof(int), c->stream);
  if (e == cudaSuccess) e = cudaMemsetAsync(v.err, 0, sizeof(int), c->stream);
  if (e == cudaSuccess && v.kv_fp8)
    e = cudaMemsetAsync(v.Ksc, 0, (l.Vsc - l.Ksc) * 2, c->stream);  // both scale arrays
  if (e != cudaSuccess) {
    delete c;
    return cuda_fail(e);
  }
  *out = c;
  return H2O_OK;
}

h2o_status h2o_cache_destroy(h2o_cache_t c) {
  if (c) {
    for (auto &m : c->marks) {
      cudaEventDestroy(m.a);
      cudaEventDestroy(m.b);
    }
  }
  delete c;
  return H2O_OK;
}

h2o_status h2o_profile_enable(h2o_cache_t c, int on) {
  if (!c) return H2O_EINVAL;
  c->profiling = on != 0;
  return H2O_OK;
}

h2o_status h2o_profile_read(h2o_cache_t c, double *ms, int64_t *launches) {
  if (!c) return H2O_EINVAL;
  double acc[4] = {0, 0, 0, 0};
  int64_t cnt[4] = {0, 0, 0, 0};
  h2o_status st = H2O_OK;
  for (auto &m : c->marks) {
    float t = 0.f;
    cudaError_t e = cudaEventSynchronize(m.b);
    if (e == cudaSuccess) e = cudaEventElapsedTime(&t, m.a, m.b);
    if (e != cudaSuccess && st == H2O_OK) st = cuda_fail(e);
    acc[m.phase] += t;
    cnt[m.phase] += m.launches;
    cudaEventDestroy(m.a);
    cudaEventDestroy(m.b);
  }
  c->marks.clear();
  for (int i = 0; i < 4; ++i) {
    if (ms) ms[i] = acc[i];
    if (launches) launches[i] = cnt[i];
  }
  return st;
}

h2o_status h2o_set_stream(h2o_cache_t c, void *s) {
  if (!c) return H2O_EINVAL;
  c->stream = (cudaStream_t)s;
  return H2O_OK;
}

h2o_status h2o_prefill(h2o_cache_t c, const void *Q, const void *K, const void *V, int L, void *O,
                       float *lse, float *colsum) {
  if (!c) return H2O_EINVAL;
  return h2o_prefill_rows(c, 0, c->B, Q, K, V, L, O, lse, colsum);
}

h2o_status h2o_prefill_rows(h2o_cache_t c, int b0, int nb, const void *Q, const void *K, const void *V, int L,
                            void *O, float *lse, float *colsum) {
  if (!c || !Q || !K || !V || !lse || !colsum) return H2O_EINVAL;
  if (L < 1 || (int64_t)L >= kMaxPos) return H2O_EINVAL;
  if (b0 < 0 || nb < 1 || b0 > c->B - nb) return H2O_EINVAL;
  if (!aligned16(Q) || !aligned16(K) || !aligned16(V) || (O && !aligned16(O)) || !aligned16(lse) ||
      !aligned16(colsum))
    return H2O_EINVAL;
  if (c->prefilled) return H2O_ESTATE;
  if (c->rows_done > 0 && L != c->prefill_L) return H2O_EINVAL;  // one prompt length per cache
  if ((int)c->row_done.size() != c->B) c->row_done.assign((size_t)c->B, 0);
  for (int b = b0; b < b0 + nb; ++b)
    if (c->row_done[(size_t)b]) return H2O_ESTATE;  // a row is prefilled once
  // The rows' heads are a contiguous block of the slot-major workspace.
  CacheView v = c->view;
  const size_t hoff = (size_t)b0 * c->H, slots = hoff * c->k;
  v.nh = nb * c->H;
  v.K = (char *)v.K + slots * c->d * c->ssize;
  v.V = (char *)v.V + slots * c->d * c->ssize;
  v.pos += slots;
  v.score += slots;
  if (v.kv_fp8) {
    v.Ksc += slots;
    v.Vsc += slots;
  }
  cudaError_t e;
  const bool tc = prefill_tc_supported(v, L);
  {
    PhaseTimer pt(c, 0, 1);
    e = tc ? launch_prefill_attn_tc(v, Q, K, V, O, lse, L, c->stream)
           : launch_prefill_attn_simt(v, Q, K, V, O, lse, L, c->stream);
    if (e != cudaSuccess) return cuda_fail(e);
    pt.done();
  }
  {
    PhaseTimer pt(c, 1, 1);
    e = tc ? launch_prefill_colsum_tc(v, Q, K, lse, colsum, L, c->stream)
           : launch_prefill_colsum_simt(v, Q, K, lse, colsum, L, c->stream);
    if (e != cudaSuccess) return cuda_fail(e);
    pt.done();
  }
  {
    PhaseTimer pt(c, 2, 1);
    e = launch_prefill_select(v, K, V, colsum, L, c->stream);
    if (e != cudaSuccess) return cuda_fail(e);
    pt.done();
  }
  for (int b = b0; b < b0 + nb; ++b) c->row_done[(size_t)b] = 1;
  c->rows_done += nb;
  c->prefill_L = L;
  if (c->rows_done == c->B) {  // every row has its initial cache: decode may start
    c->next_pos = L;
    c->n_valid = L < c->k ? L : c->k;
    c->prefilled = true;
  }
  return H2O_OK;
}

h2o_status h2o_decode_steps(h2o_cache_t c, int n, const void *q, const void *k, const void *v, void *out,
                            int32_t *evicted) {
  if (!c || n < 0) return H2O_EINVAL;
  if (n == 0) return H2O_OK;
  if (!q || !k || !v || !out) return H2O_EINVAL;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || ((uintptr_t)evicted & 3u))
    return H2O_EINVAL;
  if (!c->prefilled) return H2O_ESTATE;
  if (c->next_pos + n > kMaxPos) return H2O_EINVAL;
  const size_t step = (size_t)c->nh * c->d * c->esize;
  CacheView vc = c->view;  // cluster form: one cluster of <= 8 CTAs per head
  vc.nsplit = decode_cluster_size(c->nh, c->k, num_sms_current_device());
  const int form = c->decode_form;
  const bool cluster_ok = n >= 2 && decode_cluster_supported(vc);
  CacheView vp = vc;  // pipelined form: its own cluster size
  vp.nsplit = decode_pipe_cluster_size(c->view, num_sms_current_device());
  const bool pipe_ok = n >= 2 && decode_pipe_supported(vp);
  const bool coop_ok = n >= 2 && (form == 0 || form == 2) && decode_persistent_fits(c->view);
  bool use_cluster = false, use_pipe = false, use_coop = false;
  if (form == 4) {
    use_pipe = pipe_ok;
  } else if (form == 3) {
    use_cluster = cluster_ok;
  } else if (form == 2) {
    use_coop = coop_ok;
  } else if (form == 0) {
    // Automatic: the pipelined cluster form for bf16 and fp32 caches, the
    // cluster form for an fp8 cache, else the cooperative grid, else one
    // launch per step.  Measured on GB300, us per decode step (cluster /
    // pipelined): 8K prompt 90.1 / 73.5, OPT-30B 69.3 / 57.8, OPT-6.7B
    // 7.33 / 6.24, long stream 2.51 / 2.40; with an fp8 cache 8K prompt
    // 108.2 / 154.2, OPT-30B 97.3 / 133.6 (the pipelined kernel's lane-group
    // fp8 instance runs fewer CTAs per SM).
    if (pipe_ok && !c->view.kv_fp8)
      use_pipe = true;
    else if (cluster_ok)
      use_cluster = true;
    else if (coop_ok)
      use_coop = true;
  }
  if (n >= 2 && ((form == 4 && !use_pipe) || (form == 3 && !use_cluster) || (form == 2 && !use_coop)))
    return H2O_EUNSUPPORTED;
  PhaseTimer pt(c, 3, use_cluster || use_pipe ? 1 : use_coop ? (n + 16383) / 16384 : n);
  c->form_used = use_pipe ? 4 : use_cluster ? 3 : use_coop ? 2 : 1;
  if (use_cluster || use_pipe) {
    DecodeStep s;
    s.q = q;
    s.kn = k;
    s.vn = v;
    s.out = out;
    s.evicted = evicted;
    s.n_valid = c->n_valid;
    s.p = (int)c->next_pos;
    cudaError_t e = use_pipe ? launch_decode_pipe(vp, s, n, c->stream) : launch_decode_cluster(vc, s, n, c->stream);
    if (e != cudaSuccess) return cuda_fail(e);
    c->next_pos += n;
    c->n_valid = (int)((int64_t)c->n_valid + n < c->k ? c->n_valid + n : c->k);
    pt.done();
    return H2O_OK;
  }
  if (use_coop) {
    // One cooperative launch per chunk of steps (bounded launch length).
    constexpr int kChunk = 16384;
    for (int i0 = 0; i0 < n; i0 += kChunk) {
      const int m = n - i0 < kChunk ? n - i0 : kChunk;
      DecodeStep s;
      s.q = (const char *)q + i0 * step;
      s.kn = (const char *)k + i0 * step;
      s.vn = (const char *)v + i0 * step;
      s.out = (char *)out + i0 * step;
      s.evicted = evicted ? evicted + (size_t)i0 * c->nh : nullptr;
      s.n_valid = c->n_valid;
      s.p = (int)c->next_pos;
      cudaError_t e = launch_decode_persistent(c->view, s, m, c->view.done, c->stream);
      if (e != cudaSuccess) return cuda_fail(e);
      c->next_pos += m;
      c->n_valid = (int)((int64_t)c->n_valid + m < c->k ? c->n_valid + m : c->k);
    }
    pt.done();
    return H2O_OK;
  }
  for (int i = 0; i < n; ++i) {
    DecodeStep s;
    s.q = (const char *)q + i * step;
    s.kn = (const char *)k + i * step;
    s.vn = (const char *)v + i * step;
    s.out = (char *)out + i * step;
    s.evicted = evicted ? evicted + (size_t)i * c->nh : nullptr;
    s.n_valid = c->n_valid;
    s.p = (int)c->next_pos;
    cudaError_t e = launch_decode_step(c->view, s, c->stream);
    if (e != cudaSuccess) return cuda_fail(e);
    c->next_pos += 1;
    if (c->n_valid < c->k) c->n_valid += 1;
  }
  pt.done();
  return H2O_OK;
}

h2o_status h2o_decode_step(h2o_cache_t c, const void *q, const void *k, const void *v, void *out) {
  return h2o_decode_steps(c, 1, q, k, v, out, nullptr);
}

h2o_status h2o_set_decode_form(h2o_cache_t c, int form) {
  if (!c || form < 0 || form > 4) return H2O_EINVAL;
  c->decode_form = form;
  return H2O_OK;
}

h2o_status h2o_cache_set_policy(h2o_cache_t c, int n_sink, int score_mode) {
  if (!c || n_sink < 0 || n_sink > c->kh || (score_mode != 0 && score_mode != 1)) return H2O_EINVAL;
  c->view.n_sink = n_sink;
  c->view.score_mode = score_mode;
  return H2O_OK;
}

h2o_status h2o_cache_get_policy(h2o_cache_t c, int *n_sink, int *score_mode) {
  if (!c) return H2O_EINVAL;
  if (n_sink) *n_sink = c->view.n_sink;
  if (score_mode) *score_mode = c->view.score_mode;
  return H2O_OK;
}

h2o_status h2o_decode_form_used(h2o_cache_t c, int *form) {
  if (!c || !form) return H2O_EINVAL;
  *form = c->form_used;
  return H2O_OK;
}

h2o_status h2o_cache_export(h2o_cache_t c, int32_t *pos, float *score, void *K, void *V, int64_t *next_pos,
                            int *n_valid) {
  if (!c) return H2O_EINVAL;
  const CacheView &v = c->view;
  const size_t slots = (size_t)c->nh * c->k;
  cudaError_t e = cudaSuccess;
  if (pos) e = cudaMemcpyAsync(pos, v.pos, slots * sizeof(int32_t), cudaMemcpyDefault, c->stream);
  if (e == cudaSuccess && score)
    e = cudaMemcpyAsync(score, v.score, slots * sizeof(float), cudaMemcpyDefault, c->stream);
  if (e == cudaSuccess && K) e = cudaMemcpyAsync(K, v.K, slots * c->d * c->ssize, cudaMemcpyDefault, c->stream);
  if (e == cudaSuccess && V) e = cudaMemcpyAsync(V, v.V, slots * c->d * c->ssize, cudaMemcpyDefault, c->stream);
  if (e != cudaSuccess) return cuda_fail(e);
  if (next_pos) *next_pos = c->next_pos;
  if (n_valid) *n_valid = c->n_valid;
  return H2O_OK;
}

h2o_status h2o_cache_import(h2o_cache_t c, const int32_t *pos, const float *score, const void *K,
                            const void *V, int64_t next_pos, int n_valid) {
  if (!c || !pos || !score || !K || !V) return H2O_EINVAL;
  if (next_pos < 0 || next_pos >= kMaxPos || n_valid < 0 || n_valid > c->k) return H2O_EINVAL;
  const CacheView &v = c->view;
  const size_t slots = (size_t)c->nh * c->k;
  cudaError_t e = cudaMemcpyAsync(v.pos, pos, slots * sizeof(int32_t), cudaMemcpyDefault, c->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(v.score, score, slots * sizeof(float), cudaMemcpyDefault, c->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(v.K, K, slots * c->d * c->ssize, cudaMemcpyDefault, c->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(v.V, V, slots * c->d * c->ssize, cudaMemcpyDefault, c->stream);
  if (e != cudaSuccess) return cuda_fail(e);
  c->next_pos = next_pos;
  c->n_valid = n_valid;
  c->prefilled = true;
  return H2O_OK;
}

h2o_status h2o_cache_export_scales(h2o_cache_t c, float *Ksc, float *Vsc) {
  if (!c) return H2O_EINVAL;
  if (!c->view.kv_fp8) return H2O_EUNSUPPORTED;
  const size_t bytes = (size_t)c->nh * c->k * sizeof(float);
  cudaError_t e = cudaSuccess;
  if (Ksc) e = cudaMemcpyAsync(Ksc, c->view.Ksc, bytes, cudaMemcpyDefault, c->stream);
  if (e == cudaSuccess && Vsc) e = cudaMemcpyAsync(Vsc, c->view.Vsc, bytes, cudaMemcpyDefault, c->stream);
  return e == cudaSuccess ? H2O_OK : cuda_fail(e);
}

h2o_status h2o_cache_import_scales(h2o_cache_t c, const float *Ksc, const float *Vsc) {
  if (!c || !Ksc || !Vsc) return H2O_EINVAL;
  if (!c->view.kv_fp8) return H2O_EUNSUPPORTED;
  const size_t bytes = (size_t)c->nh * c->k * sizeof(float);
  cudaError_t e = cudaMemcpyAsync(c->view.Ksc, Ksc, bytes, cudaMemcpyDefault, c->stream);
  if (e == cudaSuccess) e = cudaMemcpyAsync(c->view.Vsc, Vsc, bytes, cudaMemcpyDefault, c->stream);
  return e == cudaSuccess ? H2O_OK : cuda_fail(e);
}

h2o_status h2o_cache_info(h2o_cache_t c, int *B, int *H, int *d, int *k_heavy, int *k_local, int *dtype,
                          int64_t *next_pos, int *n_valid, int *n_split) {
  if (!c) return H2O_EINVAL;
  if (B) *B = c->B;
  if (H) *H = c->H;
  if (d) *d = c->d;
  if (k_heavy) *k_heavy = c->kh;
  if (k_local) *k_local = c->kl;
  if (dtype) *dtype = (int)c->dtype;
  if (next_pos) *next_pos = c->next_pos;
  if (n_valid) *n_valid = c->n_valid;
  if (n_split) *n_split = c->view.nsplit;
  return H2O_OK;
}

h2o_status h2o_get_error(h2o_cache_t c) {
  if (!c) return H2O_EINVAL;
  int flag = 0;
  cudaError_t e = cudaMemcpyAsync(&flag, c->view.err, sizeof(int), cudaMemcpyDeviceToHost, c->stream);
  if (e == cudaSuccess) e = cudaStreamSynchronize(c->stream);
  if (e != cudaSuccess) return cuda_fail(e);
  return flag ? H2O_EDEVICE : H2O_OK;
}

const char *h2o_status_str(h2o_status s) {
  switch (s) {
    case H2O_OK: return "ok";
    case H2O_EINVAL: return "invalid argument";
    case H2O_ESTATE: return "invalid state";
    case H2O_ECUDA: return "CUDA error";
    case H2O_ENOMEM: return "out of host memory";
    case H2O_EDEVICE: return "device-side inconsistency";
    case H2O_EUNSUPPORTED: return "unsupported shape";
  }
  return "unknown status";
}

int h2o_last_cuda_error(void) { return g_last_cuda; }

int h2o_build_arch(void) { return 1030; }

h2o_status h2o_kernel_arch(int *ptx_version, int *binary_version) {
  cudaFuncAttributes a;
  const cudaError_t e = kernel_attributes(&a);
  if (e != cudaSuccess) return cuda_fail(e);
  if (ptx_version) *ptx_version = a.ptxVersion;
  if (binary_version) *binary_version = a.binaryVersion;
  return H2O_OK;
}

}  // extern "C"
