// select.cu — prefill selection of the initial cache set and the gather of
// the kept K/V rows into the slots (one CTA per head).
//
// H2O summary page, "Algorithm / figure walkthrough" step 1 together with the
// local/heavy split of "The mechanism": if the prompt fits (L <= k) every
// position is kept; otherwise the k_local newest positions are kept plus the
// k_heavy largest column sums among positions 0 .. L-k_local-1, equal sums
// resolved in favour of the higher position.  Policy variants ("Limitations":
// attention-sink streaming, the old-token bias of summed scores): positions
// below n_sink are always kept and take n_sink of the heavy slots; score_mode
// 1 ranks position j by colsum_j / (L - j), its mean weight over the prompt
// queries that attended to it.
//
// Ranking keys are non-negative floats, so their bit patterns order like the
// values.  A 4-pass radix select (8-bit digits, per-warp shared histograms)
// finds the threshold pattern and how many of the equal-to-threshold
// positions to keep; a block-wide ballot scan then assigns slots in ascending
// position order, and the CTA copies the kept rows with 16-byte accesses (an
// fp8 cache quantises each kept row instead: one warp per row, one scale per
// row).
#include "common.cuh"

namespace h2o {
namespace {

constexpr int kThreads = 512;
constexpr int kWarps = kThreads / 32;

// T: input type of the prompt K/V; S: type of the stored cache rows.
template <typename T, typename S, int D>
__global__ void __launch_bounds__(kThreads) select_gather(const CacheView c, const T *__restrict__ K,
                                                          const T *__restrict__ V,
                                                          const float *__restrict__ colsum, int L) {
  constexpr int EPL = VecN<T>::N, CH = D / EPL;
  __shared__ unsigned hist[kWarps][256];
  __shared__ unsigned s_tot[256];
  __shared__ unsigned s_digit, s_need, s_eq;
  __shared__ int s_weq[kWarps], s_wkeep[kWarps];

  const int h = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int k = c.k, kh = c.kh, kl = c.kl;
  const float *cs = colsum + (size_t)h * L;
  int32_t *posh = c.pos + (size_t)h * k;
  float *sch = c.score + (size_t)h * k;
  const bool keep_all = L <= k;
  const int nc = keep_all ? L : L - kl;  // heavy-hitter candidates n_sink .. nc-1
  const int ns = c.n_sink, mode = c.score_mode;
  const bool by_score = !keep_all && kh > ns;
  auto rank_of = [&](int j) -> uint32_t {
    const float v = cs[j];
    return __float_as_uint(mode ? __fdiv_rn(v, (float)(L - j)) : v);
  };

  uint32_t thr = 0;
  int need = 0, eq_total = 0;
  if (by_score) {
    uint32_t prefix = 0, pmask = 0;
    unsigned want = (unsigned)(kh - ns);
    for (int shift = 24; shift >= 0; shift -= 8) {
      for (int b = tid; b < kWarps * 256; b += kThreads) (&hist[0][0])[b] = 0u;
      __syncthreads();
      for (int j = ns + tid; j < nc; j += kThreads) {
        const uint32_t key = rank_of(j);
        if ((key & pmask) == prefix) atomicAdd(&hist[warp][(key >> shift) & 255u], 1u);
      }
      __syncthreads();
      for (int b = tid; b < 256; b += kThreads) {
        unsigned t = 0;
#pragma unroll
        for (int w = 0; w < kWarps; ++w) t += hist[w][b];
        s_tot[b] = t;
      }
      __syncthreads();
      if (tid == 0) {
        unsigned cum = 0;
        int b = 255;
        for (; b > 0; --b) {
          if (cum + s_tot[b] >= want) break;
          cum += s_tot[b];
        }
        s_digit = (unsigned)b;
        s_need = want - cum;
        s_eq = s_tot[b];
      }
      __syncthreads();
      prefix |= s_digit << shift;
      pmask |= 255u << shift;
      want = s_need;
      __syncthreads();
    }
    thr = prefix;
    need = (int)want;     // equal-to-threshold positions to keep (the highest ones)
    eq_total = (int)s_eq;  // equal-to-threshold positions in all
  }

  int run_eq = 0, run_keep = 0;
  const unsigned lt = (1u << lane) - 1u;
  for (int base = 0; base < L; base += kThreads) {
    const int j = base + tid;
    const bool in = j < L;
    const float v = in ? cs[j] : 0.f;
    const uint32_t key = in ? rank_of(j) : 0u;
    bool keep = false, eq = false;
    if (in) {
      if (keep_all || j >= nc || j < ns) keep = true;
      else if (by_score) {
        if (key > thr) keep = true;
        else if (key == thr) eq = true;
      }
    }
    const unsigned beq = __ballot_sync(0xffffffffu, eq);
    if (lane == 0) s_weq[warp] = __popc(beq);
    __syncthreads();
    int eq_rank = run_eq + __popc(beq & lt) + 1;  // 1-based rank among equals, ascending position
    int eq_chunk = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) eq_rank += s_weq[w];
      eq_chunk += s_weq[w];
    }
    if (eq) keep = eq_rank > eq_total - need;
    const unsigned bk = __ballot_sync(0xffffffffu, keep);
    if (lane == 0) s_wkeep[warp] = __popc(bk);
    __syncthreads();
    int slot = run_keep + __popc(bk & lt);
    int keep_chunk = 0;
    for (int w = 0; w < kWarps; ++w) {
      if (w < warp) slot += s_wkeep[w];
      keep_chunk += s_wkeep[w];
    }
    if (keep && slot < k) {
      posh[slot] = j;
      sch[slot] = v;
    }
    run_eq += eq_chunk;
    run_keep += keep_chunk;
    __syncthreads();
  }
  const int n = min(run_keep, k);
  if (run_keep != (keep_all ? L : k) && tid == 0) atomicOr(c.err, 2);
  for (int s = n + tid; s < k; s += kThreads) {
    posh[s] = -1;
    sch[s] = 0.f;
  }
  __syncthreads();

  const size_t hb = (size_t)h * L * D;
  if constexpr (is_fp8<S>()) {
    constexpr int PER = D / 32;  // lane L quantises elements L*PER ..
    for (int s = warp; s < k; s += kWarps) {
      const bool live = s < n;
      const int j = live ? posh[s] : 0;
      float xk[PER], xv[PER], sk, sv;
#pragma unroll
      for (int q = 0; q < PER; ++q) {
        xk[q] = live ? to_f32<T>(K[hb + (size_t)j * D + lane * PER + q]) : 0.f;
        xv[q] = live ? to_f32<T>(V[hb + (size_t)j * D + lane * PER + q]) : 0.f;
      }
      const uint32_t ck = quant_row_e4m3<PER>(xk, sk), cv = quant_row_e4m3<PER>(xv, sv);
      const size_t slot = (size_t)h * k + s;
      store_codes<PER>((uint8_t *)c.K + slot * D, lane, ck);
      store_codes<PER>((uint8_t *)c.V + slot * D, lane, cv);
      if (lane == 0) {
        c.Ksc[slot] = sk;
        c.Vsc[slot] = sv;
      }
    }
    return;
  }
  uint4 *Kc = (uint4 *)((T *)c.K + (size_t)h * k * D);
  uint4 *Vc = (uint4 *)((T *)c.V + (size_t)h * k * D);
  for (int idx = tid; idx < k * CH; idx += kThreads) {
    const int s = idx / CH, cc = idx % CH;
    uint4 kv = make_uint4(0u, 0u, 0u, 0u), vv = kv;
    if (s < n) {
      const int j = posh[s];
      kv = *(const uint4 *)(K + hb + (size_t)j * D + cc * EPL);
      vv = *(const uint4 *)(V + hb + (size_t)j * D + cc * EPL);
    }
    Kc[(size_t)s * CH + cc] = kv;
    Vc[(size_t)s * CH + cc] = vv;
  }
}

template <typename T, typename S, int D>
cudaError_t select_t(const CacheView &c, const void *K, const void *V, const float *colsum, int L,
                     cudaStream_t st) {
  select_gather<T, S, D><<<c.nh, kThreads, 0, st>>>(c, (const T *)K, (const T *)V, colsum, L);
  return cudaGetLastError();
}

}  // namespace

// Attributes of one kernel of this library as the runtime loaded it on the
// current device (binaryVersion 103 = an sm_103 cubin, not JIT-compiled PTX).
cudaError_t kernel_attributes(cudaFuncAttributes *a) {
  return cudaFuncGetAttributes(a, select_gather<__nv_bfloat16, __nv_bfloat16, 128>);
}

cudaError_t launch_prefill_select(const CacheView &c, const void *K, const void *V, const float *colsum,
                                  int L, cudaStream_t st) {
  if (c.dtype == 1 && c.kv_fp8) {
    if (c.d == 128) return select_t<__nv_bfloat16, e4m3, 128>(c, K, V, colsum, L, st);
    if (c.d == 64) return select_t<__nv_bfloat16, e4m3, 64>(c, K, V, colsum, L, st);
  } else if (c.dtype == 1) {
    if (c.d == 128) return select_t<__nv_bfloat16, __nv_bfloat16, 128>(c, K, V, colsum, L, st);
    if (c.d == 64) return select_t<__nv_bfloat16, __nv_bfloat16, 64>(c, K, V, colsum, L, st);
  } else if (!c.kv_fp8) {
    if (c.d == 128) return select_t<float, float, 128>(c, K, V, colsum, L, st);
    if (c.d == 64) return select_t<float, float, 64>(c, K, V, colsum, L, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace h2o
