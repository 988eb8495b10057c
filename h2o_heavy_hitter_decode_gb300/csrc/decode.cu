// decode.cu — H2O decode steps for every (batch, head).
//
// H2O summary page, "Algorithm / figure walkthrough" steps 2-4 and "The
// mechanism": the new query attends over the cached entries plus itself, each
// entry's softmax weight is added to its accumulated score F_score, and when
// the cache is full the lowest-scoring entry outside the k_local newest
// positions is evicted; the new token's K/V are written into the freed slot.
//
// Layout: slot-major cache, K/V [head][slot][d], pos/score [head][slot], so
// the slots a CTA owns are one contiguous byte range of K and one of V.
//
// One CTA per (head, split).  A producer warp streams the split's K and V
// rows as contiguous 4 KB slabs (cp.async.bulk into a 3-stage shared-memory
// ring, mbarrier-tracked); four consumer warps read the slabs with 16-byte
// conflict-free shared loads (LPR lanes per row), keep a per-warp online
// softmax (one rescale per slab), and write the log2-domain logits to a
// per-head global row.  The warps merge into the split's partial (max m, sum
// l, acc[d]).  The last CTA of a head to arrive (atomic ticket, no spinning)
// combines the partials into the output, turns every logit into its exact
// weight exp2(s - M) / L, adds it to the score, finds the (score, position)
// argmin among eligible slots with warp shuffles, and writes the new token in
// place.  Every other CTA of that head has finished reading K/V before it took
// its ticket, so the in-place write cannot race.
//
// An fp8 cache (S = e4m3) streams 1-byte codes: each K logit is scaled by its
// row's K scale and each V row enters the accumulator with weight times its V
// scale; the new token's row is quantised (one scale per row) when written.
//
// Two launch forms share this body:
//  * per step: one grid per step, chained with programmatic dependent launch;
//  * persistent: one cooperative grid (all CTAs resident) runs many steps.
//    Heads are independent, so there is no grid-wide barrier: before loading
//    step s a CTA's producer waits (bounded spin, acquire) until its head's
//    step s-1 is published (release by that step's last arriver).  Tails of
//    one head overlap with the streaming of others and no launch gaps remain.
#include <climits>
#include <cmath>

#include "common.cuh"
#include "sm100.cuh"

namespace h2o {
namespace {

using namespace sm100;

constexpr int kConsumers = 4;                    // consumer warps
constexpr int kConsumerThreads = 32 * kConsumers;
constexpr int kThreads = kConsumerThreads + 32;  // + one producer warp
constexpr int kMaxSplit = 64;
constexpr int kStages = 3;
constexpr int kStageBytes = 4096;                // per operand (K or V) per stage
constexpr int kSmemBytes = kStages * 2 * kStageBytes;
constexpr uint32_t kDoneSpinLimit = 1u << 24;    // polls of a head's step flag

template <typename S, int D> struct Geo {
  static constexpr int EPL = Lane<S>::VB / (int)sizeof(S);  // elements per lane per load
  static constexpr int LPR = D / EPL;             // lanes per row
  static constexpr int RPW = 32 / LPR;            // rows per warp per pass
  static constexpr int ROWB = D * (int)sizeof(S); // bytes per slot row
  static constexpr int TR = kStageBytes / ROWB;   // rows per slab
  static constexpr int ITER = TR / (kConsumers * RPW);
  static_assert(LPR >= 1 && LPR <= 32 && 32 % LPR == 0, "row must map onto a warp");
  static_assert(ITER >= 1 && TR % (kConsumers * RPW) == 0, "slab must split evenly over warps");
};

struct Args {
  CacheView c;
  DecodeStep s;      // pointers of the first step; step i adds i * nh * d elements
  int nsteps;        // steps this launch runs
  float qscale;      // log2(e) / sqrt(d)
  int *done;         // [nh] steps published per head (persistent form), zeroed before launch
};

// Named barrier over the consumer warps only (the producer may be waiting on
// its head's step flag meanwhile).
__device__ __forceinline__ void consumers_sync() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

__device__ __forceinline__ int ld_acquire(const int *p) {
  int v;
  asm volatile("ld.acquire.gpu.global.b32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
__device__ __forceinline__ void st_release(int *p, int v) {
  asm volatile("st.release.gpu.global.b32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
__device__ __forceinline__ void fence_proxy_async_global() {
  asm volatile("fence.proxy.async.global;" ::: "memory");
}

// T: type of the step inputs and outputs; S: type of the stored K/V rows.
template <typename T, typename S, int D, bool kPersistent>
__global__ void __launch_bounds__(kThreads) decode_kernel(const Args a) {
  using G = Geo<S, D>;
  constexpr bool kFp8 = is_fp8<S>();
  constexpr int EPL = G::EPL, LPR = G::LPR, RPW = G::RPW, ROWB = G::ROWB, TR = G::TR, ITER = G::ITER;
  extern __shared__ __align__(128) uint8_t s_ring[];  // [kStages][K | V][kStageBytes]
  __shared__ uint64_t s_full[kStages], s_empty[kStages];
  __shared__ uint64_t s_go;  // one phase per step: the producer saw the head's previous step published
  __shared__ float s_m[kConsumers], s_l[kConsumers];
  __shared__ float s_acc[kConsumers][D];
  __shared__ float s_fac[kMaxSplit];
  __shared__ float s_ML[2];
  __shared__ ArgMin s_am[kConsumers];
  __shared__ int s_flag, s_abort;

  if (!kPersistent) {
    // Programmatic dependent launch: wait for the previous step's grid and its
    // memory before any global access, then let the next step's grid be
    // scheduled behind this one.
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
  }

  const CacheView &c = a.c;
  const int nsplit = c.nsplit;
  const int split = blockIdx.x % nsplit;
  const int h = blockIdx.x / nsplit;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  const size_t hk = (size_t)h * c.k;
  const size_t step_elems = (size_t)c.nh * D;
  float *lg = c.logits + (size_t)h * (c.k + 1);
  float *part = c.part + ((size_t)h * nsplit + split) * (2 + D);
  const float *ph = c.part + (size_t)h * nsplit * (2 + D);
  int32_t *posh = c.pos + hk;
  float *sch = c.score + hk;

  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kConsumers);
    }
    mbar_init(&s_go, 1);
    s_abort = 0;
    fence_mbar_init();
  }
  __syncthreads();

  int g = 0;  // slabs streamed so far by this CTA (ring position), kept in step by both roles
  for (int step = 0; step < a.nsteps; ++step) {
    const int n = min(a.s.n_valid + step, c.k);  // filled slots before this step
    const int p = a.s.p + step;                   // position of the new token
    const int R = n + 1;                          // cached entries plus the new token (virtual row n)
    const int chunk = (R + nsplit - 1) / nsplit;
    const int r0 = split * chunk;
    const int r1 = min(R, r0 + chunk);
    const int nrows = max(0, min(r1, n) - r0);    // cache rows of this split: [r0, r0 + nrows)
    const int nst = (nrows + TR - 1) / TR;        // slabs
    const bool has_new = (r0 <= n && n < r1);
    const uint8_t *Kc = (const uint8_t *)c.K + (hk + r0) * ROWB;
    const uint8_t *Vc = (const uint8_t *)c.V + (hk + r0) * ROWB;
    const T *kn = (const T *)a.s.kn + step * step_elems + (size_t)h * D;
    const T *vn = (const T *)a.s.vn + step * step_elems + (size_t)h * D;

    if (warp == kConsumers) {
      // ------------------------------------------------------------ producer
      if (lane == 0) {
        bool ok = true;
        if (kPersistent && step > 0) {  // the head's previous step must be published
          uint32_t it = 0;
          while (ld_acquire(a.done + h) < step) {
            if (++it > kDoneSpinLimit || *(volatile int *)&s_abort) {
              ok = false;
              break;
            }
            __nanosleep(64);
          }
          fence_proxy_async_global();  // its generic writes, before our bulk reads
        }
        // Consumers write this step's logits and partials only after this
        // point, i.e. after the previous step's last arriver has read them.
        if (ok) mbar_arrive(&s_go);
        int issued = 0;
        for (; ok && issued < nst; ++issued) {
          const int gi = g + issued, st = gi % kStages;
          if (gi >= kStages && !(ok = mbar_wait_backoff(&s_empty[st], ((gi / kStages) - 1) & 1))) break;
          const uint32_t bytes = (uint32_t)(min(TR, nrows - issued * TR) * ROWB);
          mbar_expect_tx(&s_full[st], 2 * bytes);
          bulk_load(s_ring + st * 2 * kStageBytes, Kc + (size_t)issued * TR * ROWB, bytes, &s_full[st]);
          bulk_load(s_ring + st * 2 * kStageBytes + kStageBytes, Vc + (size_t)issued * TR * ROWB, bytes,
                    &s_full[st]);
        }
        if (!ok) {  // flag, and let copies already issued land before the CTA exits
          s_abort = 1;
          atomicOr(c.err, 1);
          for (int j = max(0, issued - kStages); j < issued; ++j)
            mbar_wait(&s_full[(g + j) % kStages], ((g + j) / kStages) & 1);
        }
      }
      g += nst;
      if (__any_sync(0xffffffffu, lane == 0 && *(volatile int *)&s_abort)) break;
      continue;
    }

    // -------------------------------------------------------------- consumers
    // A lane group (LPR lanes) takes ITER rows per slab: K dot products from
    // packed q, one transposed reduction, one exp2 per lane for the row it
    // ends up holding, broadcast back for the V rows.
    const T *qrow = (const T *)a.s.q + step * step_elems + (size_t)h * D + sub * EPL;
    QLane<S, EPL> qk;
    qk.load(qrow, a.qscale);
    constexpr int LPI = LPR / ITER;  // lanes holding one reduced row
    const int myit = sub / LPI;
    float m = -INFINITY, l = 0.f, acc[EPL];
#pragma unroll
    for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
    bool ok = __all_sync(0xffffffffu, mbar_wait(&s_go, step & 1));
    for (int i = 0; ok && i < nst; ++i, ++g) {
      const int st = g % kStages;
      const int rows = min(TR, nrows - i * TR);
      const int rm = warp * RPW + grp + myit * kConsumers * RPW;
      const bool valid = rm < rows;
      float kscm = 1.f, vsc[ITER];  // row scales of an fp8 cache (read before the slab wait)
      if (kFp8) {
        kscm = valid ? __ldcg(c.Ksc + hk + r0 + (size_t)i * TR + rm) : 0.f;
#pragma unroll
        for (int it = 0; it < ITER; ++it) {
          const int r = warp * RPW + grp + it * kConsumers * RPW;
          vsc[it] = (r < rows) ? __ldcg(c.Vsc + hk + r0 + (size_t)i * TR + r) : 0.f;
        }
      }
      if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[st], (g / kStages) & 1)))) break;
      const uint8_t *ks = s_ring + st * 2 * kStageBytes;
      const uint8_t *vs = ks + kStageBytes;
      float x[ITER];
#pragma unroll
      for (int it = 0; it < ITER; ++it) {
        const int r = warp * RPW + grp + it * kConsumers * RPW;
        x[it] = qk.dot(ks + (r < rows ? r : 0) * ROWB + sub * Lane<S>::VB);
      }
      float lgt = xreduce<ITER, LPR>(x, sub) * qk.scale;
      if (kFp8) lgt *= kscm;
      lgt = valid ? lgt : -INFINITY;
      if (valid && sub % LPI == 0) lg[r0 + i * TR + rm] = lgt;
      float wmax = lgt;  // over the warp's rows of this slab
#pragma unroll
      for (int o = LPI; o < 32; o <<= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
      if (wmax > m) {  // warp-uniform: rescale only when the running max grows
        const float sc = ex2(m - wmax);
        l *= sc;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] *= sc;
        m = wmax;
      }
      const float prm = valid ? ex2(lgt - m) : 0.f;
#pragma unroll
      for (int it = 0; it < ITER; ++it) {
        const int r = warp * RPW + grp + it * kConsumers * RPW;
        const float pr = __shfl_sync(0xffffffffu, prm, grp * LPR + it * LPI);
        if (r < rows) {
          l += pr;
          const float pv = kFp8 ? pr * vsc[it] : pr;
          float vx[EPL];
          unpack_lane<S>(vs + r * ROWB + sub * Lane<S>::VB, vx);
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pv, vx[e], acc[e]);
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_empty[st]);
    }
    // Warp-uniform and, through s_abort, CTA-consistent: a failed wait stops
    // every consumer warp at the same step.
    if (!ok && lane == 0) {
      s_abort = 1;
      atomicOr(c.err, 1);
    }
    consumers_sync();
    if (*(volatile int *)&s_abort) break;
    if (has_new && warp == 0) {  // the new token, straight from the step inputs
      float qv[EPL], kx[EPL];
      load_f32_nc<T, EPL>(qrow, qv);
      load_f32_nc<T, EPL>(kn + sub * EPL, kx);
      float dot = 0.f;
#pragma unroll
      for (int e = 0; e < EPL; ++e) dot = fmaf(qv[e], kx[e], dot);
#pragma unroll
      for (int o = LPR / 2; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
      dot *= a.qscale;
      if (lane == 0) lg[n] = dot;
      const float mn = fmaxf(m, dot);
      const float sc = ex2(m - mn);
      l *= sc;
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] *= sc;
      m = mn;
      if (grp == 0) {
        const float pr = ex2(dot - m);
        l += pr;
        float vx[EPL];
        load_f32_nc<T, EPL>(vn + sub * EPL, vx);
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pr, vx[e], acc[e]);
      }
    }
#pragma unroll
    for (int o = LPR; o < 32; o <<= 1) {
      l += __shfl_xor_sync(0xffffffffu, l, o);
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
    }
    if (grp == 0) {
#pragma unroll
      for (int e = 0; e < EPL; ++e) s_acc[warp][sub * EPL + e] = acc[e];
    }
    if (lane == 0) {
      s_m[warp] = m;
      s_l[warp] = l;
    }
    consumers_sync();

    // ---- split partial: merge the consumer warps
    {
      float M = s_m[0];
#pragma unroll
      for (int w = 1; w < kConsumers; ++w) M = fmaxf(M, s_m[w]);
      float f[kConsumers];
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) f[w] = (s_m[w] == -INFINITY) ? 0.f : exp2f(s_m[w] - M);
      for (int col = tid; col < D; col += kConsumerThreads) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) t = fmaf(f[w], s_acc[w][col], t);
        part[2 + col] = t;
      }
      if (tid == 0) {
        float lsum = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) lsum = fmaf(f[w], s_l[w], lsum);
        part[0] = M;  // -inf for an empty split
        part[1] = lsum;
      }
    }

    // ---- the last arriver of this head finishes the step
    __threadfence();
    consumers_sync();
    if (tid == 0) s_flag = (atomicAdd(&c.counter[h], 1) == nsplit - 1);
    consumers_sync();
    if (s_flag) {
      __threadfence();
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
          c.counter[h] = 0;  // ready for the next step
        }
      }
      consumers_sync();
      const float Mg = s_ML[0];
      const float invL = 1.f / s_ML[1];
      T *out = (T *)a.s.out + step * step_elems + (size_t)h * D;
      for (int col = tid; col < D; col += kConsumerThreads) {
        float o = 0.f;
        for (int s = 0; s < nsplit; ++s) o = fmaf(s_fac[s], __ldcg(ph + (size_t)s * (2 + D) + 2 + col), o);
        out[col] = from_f32<T>(o * invL);
      }

      // exact weights into the scores; argmin over entries outside the local block
      // (eligible iff n_sink <= pos <= p - k_local)
      const long long lim = (long long)p - c.kl;
      ArgMin best{INFINITY, INT_MAX, -2};
      for (int j = tid; j < n; j += kConsumerThreads) {
        const float w = exp2f(__ldcg(lg + j) - Mg) * invL;
        const float sc = sch[j] + w;
        sch[j] = sc;
        const int pj = posh[j];
        if ((long long)pj <= lim && pj >= c.n_sink) {
          const ArgMin cand{rank_key(sc, p, pj, c.score_mode), pj, j};
          if (am_less(cand, best)) best = cand;
        }
      }
      const float w_new = exp2f(__ldcg(lg + n) - Mg) * invL;
      if (tid == 0 && c.kl == 0 && p >= c.n_sink) {
        const ArgMin cand{w_new, p, -1};  // attended by one query: its mean is its weight
        if (am_less(cand, best)) best = cand;
      }
      best = warp_argmin(best);
      if (lane == 0) s_am[warp] = best;
      consumers_sync();
      if (tid == 0) {
        ArgMin b = s_am[0];
#pragma unroll
        for (int w = 1; w < kConsumers; ++w)
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
        if (a.s.evicted) a.s.evicted[(size_t)step * c.nh + h] = ev;
        s_flag = e;
      }
      consumers_sync();
      const int e = s_flag;
      if (e >= 0 && kFp8) {
        if (warp == 0) {  // quantise the new row: one scale per row, lane L codes elements L*PER..
          constexpr int PER = D / 32;
          float xk[PER], xv[PER], sk, sv;
#pragma unroll
          for (int j = 0; j < PER; ++j) {
            xk[j] = to_f32<T>(kn[lane * PER + j]);
            xv[j] = to_f32<T>(vn[lane * PER + j]);
          }
          const uint32_t ck = quant_row_e4m3<PER>(xk, sk), cv = quant_row_e4m3<PER>(xv, sv);
          store_codes<PER>((uint8_t *)c.K + (hk + e) * ROWB, lane, ck);
          store_codes<PER>((uint8_t *)c.V + (hk + e) * ROWB, lane, cv);
          if (lane == 0) {
            c.Ksc[hk + e] = sk;
            c.Vsc[hk + e] = sv;
          }
        }
      } else if (e >= 0) {
        uint4 *Kw = (uint4 *)((S *)c.K + (hk + e) * D);
        uint4 *Vw = (uint4 *)((S *)c.V + (hk + e) * D);
        for (int i = tid; i < D / EPL; i += kConsumerThreads) {
          Kw[i] = ld_nc16(kn + i * EPL);
          Vw[i] = ld_nc16(vn + i * EPL);
        }
      }
      if (kPersistent) {
        __threadfence();
        fence_proxy_async_global();
        consumers_sync();
        if (tid == 0) st_release(a.done + h, step + 1);  // publish: head h finished this step
      }
    }
    consumers_sync();  // shared partial buffers are rewritten next step
  }
  __syncthreads();
}

template <typename T, typename S, int D, bool P>
cudaError_t set_smem_attr() {
  // The shared-memory opt-in is per device; remember it per device ordinal.
  static bool done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess && dev >= 0 && dev < 64 && done[dev]) return cudaSuccess;
  cudaError_t e = cudaFuncSetAttribute(decode_kernel<T, S, D, P>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                       kSmemBytes);
  if (e == cudaSuccess && dev >= 0 && dev < 64) done[dev] = true;
  return e;
}

template <typename T, typename S, int D>
cudaError_t launch_step_t(const CacheView &c, const DecodeStep &s, cudaStream_t st) {
  Args a{c, s, 1, kLog2e / sqrtf((float)D), nullptr};
  cudaError_t e = set_smem_attr<T, S, D, false>();
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(c.nsplit * c.nh));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<T, S, D, false>, a);
}

template <typename T, typename S, int D>
bool persistent_fits_t(const CacheView &c) {
  int dev = 0, sms = 0, per_sm = 0, coop = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&coop, cudaDevAttrCooperativeLaunch, dev) != cudaSuccess || !coop) return false;
  if (set_smem_attr<T, S, D, true>() != cudaSuccess) return false;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_kernel<T, S, D, true>, kThreads, kSmemBytes) !=
      cudaSuccess)
    return false;
  return (long long)c.nsplit * c.nh <= (long long)per_sm * sms;
}

template <typename T, typename S, int D>
cudaError_t launch_persistent_t(const CacheView &c, const DecodeStep &s, int nsteps, int *done, cudaStream_t st) {
  Args a{c, s, nsteps, kLog2e / sqrtf((float)D), done};
  cudaError_t e = set_smem_attr<T, S, D, true>();
  if (e != cudaSuccess) return e;
  e = cudaMemsetAsync(done, 0, (size_t)c.nh * sizeof(int), st);
  if (e != cudaSuccess) return e;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(c.nsplit * c.nh));
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // every CTA resident: cross-CTA waits cannot deadlock
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_kernel<T, S, D, true>, a);
}

}  // namespace

// Splits per head.  A CTA needs ~27 KB of shared memory, so eight fit on an
// SM.  Fewer heads than resident CTA slots: split so one wave covers the GPU
// (>= 32 rows per split).  More heads: pick the smallest split count whose last
// wave is at least 90 % full (up to 8), else the best-filled one.
int decode_splits(int nh, int k, int sms) {
  const int rows = k + 1;
  const int slots = 8 * (sms > 0 ? sms : 1);
  int max_ns = (rows + 31) / 32;
  if (max_ns > kMaxSplit) max_ns = kMaxSplit;
  if (max_ns < 1) max_ns = 1;
  if (nh < slots) {
    int ns = slots / nh;
    return ns < 1 ? 1 : (ns > max_ns ? max_ns : ns);
  }
  int best = 1;
  double best_eff = 0.0;
  for (int ns = 1; ns <= 8 && ns <= max_ns; ++ns) {
    const double waves = (double)ns * nh / slots;
    const double eff = waves / std::ceil(waves);
    if (eff >= 0.9) return ns;
    if (eff > best_eff + 1e-9) {
      best_eff = eff;
      best = ns;
    }
  }
  return best;
}

#define H2O_DISPATCH(FN, ...)                                                      \
  do {                                                                            \
    if (c.dtype == 1 && c.kv_fp8) {                                               \
      if (c.d == 128) return FN<__nv_bfloat16, e4m3, 128>(__VA_ARGS__);           \
      if (c.d == 64) return FN<__nv_bfloat16, e4m3, 64>(__VA_ARGS__);             \
    } else if (c.dtype == 1) {                                                    \
      if (c.d == 128) return FN<__nv_bfloat16, __nv_bfloat16, 128>(__VA_ARGS__);  \
      if (c.d == 64) return FN<__nv_bfloat16, __nv_bfloat16, 64>(__VA_ARGS__);    \
    } else if (!c.kv_fp8) {                                                       \
      if (c.d == 128) return FN<float, float, 128>(__VA_ARGS__);                  \
      if (c.d == 64) return FN<float, float, 64>(__VA_ARGS__);                    \
    }                                                                             \
  } while (0)

cudaError_t launch_decode_step(const CacheView &c, const DecodeStep &s, cudaStream_t st) {
  if (c.nsplit < 1 || c.nsplit > kMaxSplit) return cudaErrorInvalidValue;
  H2O_DISPATCH(launch_step_t, c, s, st);
  return cudaErrorInvalidValue;
}

bool decode_persistent_fits(const CacheView &c) {
  if (c.nsplit < 1 || c.nsplit > kMaxSplit) return false;
  H2O_DISPATCH(persistent_fits_t, c);
  return false;
}

cudaError_t launch_decode_persistent(const CacheView &c, const DecodeStep &s, int nsteps, int *done,
                                     cudaStream_t st) {
  if (c.nsplit < 1 || c.nsplit > kMaxSplit || nsteps < 1 || !done) return cudaErrorInvalidValue;
  H2O_DISPATCH(launch_persistent_t, c, s, nsteps, done, st);
  return cudaErrorInvalidValue;
}

}  // namespace h2o
