// decode.cu — one H2O decode step for every (batch, head) in ONE launch.
//
// H2O summary page, "Algorithm / figure walkthrough" steps 2-4 and "The
// mechanism": the new query attends over the cached entries plus itself, each
// entry's softmax weight is added to its accumulated score F_score, and when
// the cache is full the lowest-scoring entry outside the k_local newest
// positions is evicted; the new token's K/V are written into the freed slot.
//
// Layout: slot-major cache, K/V [head][slot][d], pos/score [head][slot].
// Grid: nsplit CTAs per head, each owning a contiguous range of slots (the new
// token is virtual row n_valid).  Each CTA streams its K rows (16-byte
// coalesced loads, LPR lanes per row), keeps the log2-domain logits in shared
// memory and in a per-head global row, then streams its V rows and writes a
// partial (max m, sum l, acc[d]).  The last CTA of a head to arrive (atomic
// ticket, no spinning) combines the partials into the output, turns every
// logit into its exact weight exp2(s - M) / L, adds it to the score, finds the
// (score, position) argmin among eligible slots with warp shuffles, and
// writes the new token in place.  Every other CTA of that head has finished
// reading K/V before it took its ticket, so the in-place write cannot race.
#include <climits>

#include "common.cuh"

namespace h2o {
namespace {

constexpr int kThreads = 128;
constexpr int kWarps = kThreads / 32;
constexpr int kMaxSplit = 64;
constexpr int kUnroll = 4;

template <typename T, int D> struct Geo {
  static constexpr int EPL = VecN<T>::N;  // elements per lane per 16-byte load
  static constexpr int LPR = D / EPL;     // lanes per row
  static constexpr int RPW = 32 / LPR;    // rows per warp per pass
  static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row must map onto a warp");
};

struct Args {
  CacheView c;
  DecodeStep s;
  int chunk;     // slot rows per split
  float qscale;  // log2(e) / sqrt(d)
};

template <typename T, int D>
__global__ void __launch_bounds__(kThreads) decode_step_kernel(const Args a) {
  using G = Geo<T, D>;
  constexpr int EPL = G::EPL, LPR = G::LPR, RPW = G::RPW;
  constexpr int STRIDE = kWarps * RPW;  // rows covered by the CTA per pass
  extern __shared__ float s_lg[];       // [chunk] logits of this split
  __shared__ float s_red[kWarps], s_lsum[kWarps];
  __shared__ float s_acc[kWarps][D];
  __shared__ float s_fac[kMaxSplit];
  __shared__ float s_ML[2];
  __shared__ ArgMin s_am[kWarps];
  __shared__ int s_flag;

  const CacheView &c = a.c;
  const int nsplit = c.nsplit;
  const int split = blockIdx.x % nsplit;
  const int h = blockIdx.x / nsplit;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  const int n = a.s.n_valid;
  const int R = n + 1;  // cached entries plus the new token
  const int r0 = split * a.chunk;
  const int r1 = min(R, r0 + a.chunk);
  const size_t hk = (size_t)h * c.k;
  const T *Kc = (const T *)c.K + hk * D;
  const T *Vc = (const T *)c.V + hk * D;
  const T *kn = (const T *)a.s.kn + (size_t)h * D;
  const T *vn = (const T *)a.s.vn + (size_t)h * D;
  float *lg = c.logits + (size_t)h * (c.k + 1);
  float *part = c.part + ((size_t)h * nsplit + split) * (2 + D);

  float qv[EPL];
  Unpack<T>::run(ld_nc16((const T *)a.s.q + (size_t)h * D + sub * EPL), qv);
#pragma unroll
  for (int e = 0; e < EPL; ++e) qv[e] *= a.qscale;

  // ---- pass over K: logits (log2 units) and the split max
  float mloc = -INFINITY;
  for (int base = r0 + warp * RPW; base < r1; base += STRIDE * kUnroll) {
    uint4 raw[kUnroll];
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int r = base + u * STRIDE + grp;
      raw[u] = make_uint4(0u, 0u, 0u, 0u);
      if (r < r1) raw[u] = ld_nc16((r < n ? Kc + (size_t)r * D : kn) + sub * EPL);
    }
#pragma unroll
    for (int u = 0; u < kUnroll; ++u) {
      const int r = base + u * STRIDE + grp;
      float x[EPL];
      Unpack<T>::run(raw[u], x);
      float s = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) s = fmaf(qv[e], x[e], s);
#pragma unroll
      for (int o = LPR / 2; o; o >>= 1) s += __shfl_xor_sync(0xffffffffu, s, o);
      if (r < r1) {
        mloc = fmaxf(mloc, s);
        if (sub == 0) {
          s_lg[r - r0] = s;
          lg[r] = s;
        }
      }
    }
  }
  mloc = warp_max(mloc);
  if (lane == 0) s_red[warp] = mloc;
  __syncthreads();
  float M = s_red[0];
#pragma unroll
  for (int w = 1; w < kWarps; ++w) M = fmaxf(M, s_red[w]);

  // ---- pass over V: p = 2^(s - M), l = sum p, acc = sum p v
  float acc[EPL];
#pragma unroll
  for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
  float lsum = 0.f;
  if (r0 < r1) {
    for (int base = r0 + warp * RPW; base < r1; base += STRIDE * kUnroll) {
      uint4 raw[kUnroll];
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int r = base + u * STRIDE + grp;
        raw[u] = make_uint4(0u, 0u, 0u, 0u);
        if (r < r1) raw[u] = ld_nc16((r < n ? Vc + (size_t)r * D : vn) + sub * EPL);
      }
#pragma unroll
      for (int u = 0; u < kUnroll; ++u) {
        const int r = base + u * STRIDE + grp;
        if (r < r1) {
          const float p = exp2f(s_lg[r - r0] - M);
          lsum += p;
          float x[EPL];
          Unpack<T>::run(raw[u], x);
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = fmaf(p, x[e], acc[e]);
        }
      }
    }
  }
#pragma unroll
  for (int o = LPR; o < 32; o <<= 1) {
    lsum += __shfl_xor_sync(0xffffffffu, lsum, o);
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
  }
  if (grp == 0) {
#pragma unroll
    for (int e = 0; e < EPL; ++e) s_acc[warp][sub * EPL + e] = acc[e];
  }
  if (lane == 0) s_lsum[warp] = lsum;
  __syncthreads();
  for (int col = tid; col < D; col += kThreads) {
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) t += s_acc[w][col];
    part[2 + col] = t;
  }
  if (tid == 0) {
    float l = 0.f;
#pragma unroll
    for (int w = 0; w < kWarps; ++w) l += s_lsum[w];
    part[0] = M;  // -inf for an empty split
    part[1] = l;
  }

  // ---- last arriver of this head finishes the step
  __threadfence();
  __syncthreads();
  if (tid == 0) s_flag = (atomicAdd(&c.counter[h], 1) == nsplit - 1);
  __syncthreads();
  if (!s_flag) return;
  __threadfence();

  const float *ph = c.part + (size_t)h * nsplit * (2 + D);
  if (warp == 0) {
    float mv = -INFINITY;
    for (int s = lane; s < nsplit; s += 32) mv = fmaxf(mv, __ldcg(ph + (size_t)s * (2 + D)));
    mv = warp_max(mv);
    float lv = 0.f;
    for (int s = lane; s < nsplit; s += 32) {
      const float ms = __ldcg(ph + (size_t)s * (2 + D));
      const float f = (ms == -INFINITY) ? 0.f : exp2f(ms - mv);
      s_fac[s] = f;
      lv = fmaf(f, __ldcg(ph + (size_t)s * (2 + D) + 1), lv);
    }
    lv = warp_sum(lv);
    if (lane == 0) {
      s_ML[0] = mv;
      s_ML[1] = lv;
      c.counter[h] = 0;  // ready for the next launch
    }
  }
  __syncthreads();
  const float Mg = s_ML[0];
  const float invL = 1.f / s_ML[1];
  T *out = (T *)a.s.out + (size_t)h * D;
  for (int col = tid; col < D; col += kThreads) {
    float o = 0.f;
    for (int s = 0; s < nsplit; ++s) o = fmaf(s_fac[s], __ldcg(ph + (size_t)s * (2 + D) + 2 + col), o);
    out[col] = from_f32<T>(o * invL);
  }

  // exact weights into the scores; argmin over entries outside the local block
  int32_t *posh = c.pos + hk;
  float *sch = c.score + hk;
  const int p = a.s.p;
  const long long lim = (long long)p - c.kl;  // eligible iff pos <= p - k_local
  ArgMin best{INFINITY, INT_MAX, -2};
  for (int j = tid; j < n; j += kThreads) {
    const float w = exp2f(__ldcg(lg + j) - Mg) * invL;
    const float sc = sch[j] + w;
    sch[j] = sc;
    const int pj = posh[j];
    if ((long long)pj <= lim) {
      const ArgMin cand{sc, pj, j};
      if (am_less(cand, best)) best = cand;
    }
  }
  const float w_new = exp2f(__ldcg(lg + n) - Mg) * invL;
  if (tid == 0 && c.kl == 0) {
    const ArgMin cand{w_new, p, -1};
    if (am_less(cand, best)) best = cand;
  }
  best = warp_argmin(best);
  if (lane == 0) s_am[warp] = best;
  __syncthreads();
  if (tid == 0) {
    ArgMin b = s_am[0];
#pragma unroll
    for (int w = 1; w < kWarps; ++w)
      if (am_less(s_am[w], b)) b = s_am[w];
    int e = -1, ev = -1;
    if (n < c.k) {
      e = n;  // |S| < k: admit into the next free slot
    } else if (b.slot == -2) {
      atomicOr(c.err, 1);  // no eviction candidate: state was inconsistent
    } else if (b.slot == -1) {
      ev = p;  // the new token itself scores lowest (k_local = 0)
    } else {
      e = b.slot;
      ev = posh[e];
    }
    if (e >= 0) {
      posh[e] = p;
      sch[e] = w_new;
    }
    if (a.s.evicted) a.s.evicted[h] = ev;
    s_flag = e;
  }
  __syncthreads();
  const int e = s_flag;
  if (e >= 0) {
    uint4 *Kw = (uint4 *)((T *)c.K + (hk + e) * D);
    uint4 *Vw = (uint4 *)((T *)c.V + (hk + e) * D);
    for (int i = tid; i < D / EPL; i += kThreads) {
      Kw[i] = ld_nc16(kn + i * EPL);
      Vw[i] = ld_nc16(vn + i * EPL);
    }
  }
}

template <typename T, int D>
cudaError_t launch_t(const CacheView &c, const DecodeStep &s, cudaStream_t st) {
  Args a;
  a.c = c;
  a.s = s;
  const int R = s.n_valid + 1;
  a.chunk = (R + c.nsplit - 1) / c.nsplit;
  a.qscale = kLog2e / sqrtf((float)D);
  const size_t smem = (size_t)a.chunk * sizeof(float);
  if (smem > 48 * 1024) {
    cudaError_t e = cudaFuncSetAttribute(decode_step_kernel<T, D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem);
    if (e != cudaSuccess) return e;
  }
  decode_step_kernel<T, D><<<dim3((unsigned)(c.nsplit * c.nh)), kThreads, smem, st>>>(a);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_decode_step(const CacheView &c, const DecodeStep &s, cudaStream_t st) {
  if (c.nsplit < 1 || c.nsplit > kMaxSplit) return cudaErrorInvalidValue;
  if (c.dtype == 1) {
    if (c.d == 128) return launch_t<__nv_bfloat16, 128>(c, s, st);
    if (c.d == 64) return launch_t<__nv_bfloat16, 64>(c, s, st);
  } else {
    if (c.d == 128) return launch_t<float, 128>(c, s, st);
    if (c.d == 64) return launch_t<float, 64>(c, s, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace h2o
