// decode_pipe.cu — many H2O decode steps in one launch, one thread-block
// cluster per (batch, head), with each step's eviction decision taken while
// the next step's attention pass runs.
//
// Method: H2O summary page, "Algorithm / figure walkthrough" steps 2-4 (the
// same computation as decode.cu and decode_cluster.cu): attend over the cache
// plus the new token, add each exact weight to its entry's accumulated score,
// evict the lowest (score, position) outside the k_local newest positions,
// write the new token in place.
//
// Slot ownership, the slab ring and the two DSMEM exchanges of a step are
// those of decode_cluster.cu; the order of the work differs.  Step t attends
// over the cache state S_t, which differs from S_{t-1} in one slot at most
// (Definition 4.3 of the explainer page: at most one change per step).  So:
//   * the consumer warps run step t's attention pass (logits, per-warp online
//     softmax) over the rows of S_{t-1}: the slabs carry every decision up to
//     step t-3, and the slot that step t-2 changed is read from that
//     decision's pending copy of its new row;
//   * meanwhile one warp (the protocol warp) finishes step t-1: (m, l)
//     exchange, exact weights into the scores, argmin, candidate exchange,
//     decision; a producer warp feeds the slab ring and writes decisions
//     back to the cache rows;
//   * when the consumers hand over step t's partial (m, l, acc), the protocol
//     warp applies decision t-1 to it: it removes the evicted row's term (its
//     logit at step t is in the step's logit buffer; its V row was saved at
//     the decision) and adds the admitted token's row, then adds the step's
//     new token (rank 0) and runs step t's exchanges.
// Removing a term is exact up to rounding when it is at most half of the
// CTA's partial mass.  When it is more (the entry evicted as the least
// attended takes most of the next query's attention in this CTA), the CTA's
// partial is recomputed from the step's stored logits and the V rows.
// Decisions reach the cache rows in HBM three steps late: the producer warp
// writes decision u's row only after every slab of step u+1 has landed (those
// must still see the old row) and before it issues the first slab of step
// u+3.  A CTA whose rows stay resident in shared memory writes a decision's
// row to its resident copy and to HBM during the next step, after that
// step's exchange push (nothing in the launch reads the HBM rows, and the
// consumers read the slot from the pending copy until then).
// All waits are bounded (error flag, drain, exit); clusters never wait on one
// another.
#include <cooperative_groups.h>

#include <climits>

#include "common.cuh"
#include "sm100.cuh"

namespace cg = cooperative_groups;

namespace h2o {
namespace {

using namespace sm100;

constexpr int kShortChunk = 256;                                 // <= : two consumer warps, else four
constexpr int threads_for(int nc) { return 32 * nc + 64; }        // + the protocol and producer warps
constexpr int kMaxCluster = 8;
constexpr int stage_bytes(bool wide) { return 4096; }  // 4 KB per operand (16 bf16 rows of 128 in the wide layout)
constexpr int ring_bytes(int stages, bool wide = false) { return stages * 2 * stage_bytes(wide); }
constexpr int kResidentMaxBytes = 96 * 1024;
constexpr int kBufs = 3;  // step-input and pending-row buffers (steps t, t-1, t-2 in use)

template <typename S, int D, int NC, bool W> struct Geo {
  static constexpr int EPL = Lane<S>::VB / (int)sizeof(S);
  static constexpr int LPR = D / EPL;
  static constexpr int RPW = 32 / LPR;
  static constexpr int ROWB = D * (int)sizeof(S);
  static constexpr int SB = stage_bytes(W);
  static constexpr int TR = SB / ROWB;
  static constexpr int ITER = W ? 1 : TR / (NC * RPW);
  static_assert(W ? (TR == 16 && ROWB == 256) : (ITER >= 1 && TR % (NC * RPW) == 0),
                "slab must split evenly over warps (wide: 32 bf16 rows of 128)");
};

struct PArgs {
  CacheView c;
  DecodeStep s;  // first step; step i adds i * nh * d elements to q/k/v/out, i * nh to evicted
  int nsteps;
  int chunk;     // slots per CTA
  float qscale;  // log2(e) / sqrt(d)
};

// Elements lane*N .. lane*N+N-1 of a stored row (bf16, fp32 or e4m3 codes,
// unscaled) as floats.
template <typename S, int N> __device__ __forceinline__ void row_part(const void *row, int lane, float *x) {
  if constexpr (std::is_same<S, float>::value) {
    const float *p = (const float *)row + lane * N;
#pragma unroll
    for (int i = 0; i < N; ++i) x[i] = p[i];
  } else if constexpr (std::is_same<S, __nv_bfloat16>::value) {
    const uint32_t *p = (const uint32_t *)row + lane * (N / 2);
#pragma unroll
    for (int i = 0; i < N / 2; ++i) {
      const uint32_t w = p[i];
      x[2 * i] = bf16lo(w);
      x[2 * i + 1] = bf16hi(w);
    }
  } else {
    static_assert(N == 2 || N == 4, "a lane holds 2 or 4 codes");
    const uint8_t *p = (const uint8_t *)row + lane * N;
    if constexpr (N == 4) {
      e4m3x4_to_f32(*(const uint32_t *)p, x);
    } else {
      const __half2_raw h = __nv_cvt_fp8x2_to_halfraw2((__nv_fp8x2_storage_t)(*(const uint16_t *)p), __NV_E4M3);
      x[0] = __half2float(__ushort_as_half(h.x));
      x[1] = __half2float(__ushort_as_half(h.y));
    }
  }
}

// Warp maximum of a float by one integer min/max reduction: the bit
// pattern, with the magnitude bits of negative values flipped, orders like
// the value (-inf lowest; no NaN arrives here).
__device__ __forceinline__ float warp_max_ordered(float v) {
  const int i = __float_as_int(v);
  const int k = __reduce_max_sync(0xffffffffu, i >= 0 ? i : i ^ 0x7fffffff);
  return __int_as_float(k >= 0 ? k : k ^ 0x7fffffff);
}

// Warp copy of `bytes` (a multiple of 64) from src to dst, 4-byte words.
__device__ __forceinline__ void warp_copy(void *dst, const void *src, int bytes, int lane) {
  for (int o = lane * 4; o < bytes; o += 128) *(uint32_t *)((uint8_t *)dst + o) = *(const uint32_t *)((const uint8_t *)src + o);
}

// T: type of the step inputs and outputs; S: type of the stored K/V rows;
// NC: consumer warps; W: wide-row layout (bf16 rows of 128).
template <typename T, typename S, int D, bool kResident, int kStages, int NC, bool W>
__global__ void __launch_bounds__(threads_for(NC), W ? 5 : (NC == 2 ? 7 : 5))
    decode_pipe_kernel(const PArgs a) {
  constexpr int kThreads = threads_for(NC);
  using G = Geo<S, D, NC, W>;
  constexpr int SB = G::SB;
  constexpr bool kFp8 = is_fp8<S>();
  constexpr int EPL = G::EPL, LPR = G::LPR, RPW = G::RPW, ROWB = G::ROWB, TR = G::TR, ITER = G::ITER;
  constexpr int CPL = D / 32;  // dimensions per lane in the protocol warp
  static_assert(!kFp8 || CPL == 2 || CPL == 4, "fp8 rows of 64 or 128");
  constexpr uint32_t FULL = 0xffffffffu;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(1024) uint8_t smem[];
  // Full barriers: one per ring stage, or (wide layout) one per stage and
  // consumer warp, so that every full barrier is waited on by one consumer
  // warp only, in order.
  constexpr int kFullBars = W ? kStages * NC : kStages;
  __shared__ uint64_t s_full[kFullBars], s_empty[kStages];
  __shared__ uint64_t s_inbar[kBufs];  // step inputs landed
  __shared__ uint64_t s_part[2];       // a step's consumer partials (NC arrivals)
  __shared__ uint64_t s_dec[4];        // decision of step u made (phase u / 4 of s_dec[u % 4])
  __shared__ uint64_t s_oldv;          // evicted V row saved (one phase per decision)
  __shared__ __align__(8) uint64_t s_bml, s_bacc[2], s_bcand;  // acc values of step u complete on s_bacc[u & 1]
  __shared__ __align__(16) T s_in[kBufs][3][D];  // q, k_t, v_t of step u in buffer u % 3
  __shared__ float s_wm[2][NC], s_wl[2][NC];
  __shared__ __align__(16) float s_wacc[2][NC][D];
  __shared__ __align__(16) uint4 s_mlx[kMaxCluster];    // every rank's (m, l, new-token logit)
  __shared__ __align__(16) uint4 s_candx[kMaxCluster];  // every rank's candidate
  // Pending decision of step u (buffer u % 3): the slot it wrote in this CTA
  // (-1: none here), whether it replaced a filled slot, and the new row as
  // stored (K then V; e4m3 codes and their scales for an fp8 cache).
  __shared__ int s_pslot[kBufs], s_pevict[kBufs];
  __shared__ float s_pksc[kBufs], s_pvsc[kBufs];
  __shared__ __align__(16) uint8_t s_pend[kBufs][2][ROWB];
  __shared__ __align__(16) uint8_t s_oldrow[ROWB];  // the evicted slot's V row (streaming form)
  __shared__ int s_tp, s_pw;  // decisions made; decisions written back to the cache rows in HBM
  __shared__ int s_abort;

  const CacheView &c = a.c;
  const int P = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int h = blockIdx.x / P;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  const int chunk = a.chunk;
  const int s0 = rank * chunk;
  const int own = max(0, min(c.k, s0 + chunk) - s0);
  // Output row: rank 0 writes it from every rank's acc row, except in the
  // wide-row layout, where each rank writes D/P of its dimensions from every
  // rank's acc values there (a smaller exchange buffer: the shared memory
  // goes to the ring and a fifth CTA per SM; on the short per-step chains of
  // resident and lane-group shapes the extra exchange wait costs more).
  constexpr bool kSplitOut = W && !kResident;
  const int DPR = kSplitOut ? D / P : D;  // output dimensions per writing rank (P divides D)
  const size_t hk = (size_t)h * c.k;
  const size_t step_elems = (size_t)c.nh * D;

  // dynamic shared memory: [ring or resident K|V][score][pos][score
  // compensation][logits of two steps] (+ [K scale][V scale])[output
  // exchange of two steps: every rank's acc row, 2 x P x D (read on rank
  // 0), or every rank's values of this CTA's D/P dimensions, 2 x D (wide
  // rows)]
  uint8_t *kv = smem;
  const int kv_bytes = kResident ? 2 * chunk * ROWB : ring_bytes(kStages, W);
  float *sc = (float *)(smem + kv_bytes);
  int *ps = (int *)(sc + chunk);
  float *cm = (float *)(ps + chunk);
  float *lgb = cm + chunk;  // logits of step u at lgb + (u & 1) * chunk
  float *ksc = lgb + 2 * chunk;
  float *vsc = ksc + chunk;
  float *accx = (float *)(smem + ((kv_bytes + (kFp8 ? 7 : 5) * chunk * 4 + 15) & ~15));

  // Rows of this CTA filled in the cache state after u decisions of this call.
  auto rows_after = [&](int u) -> int {
    const long long n = min((long long)a.s.n_valid + u, (long long)c.k);
    return (int)max(0LL, min((long long)own, n - s0));
  };

  if (tid == 0) {
    for (int i = 0; i < kFullBars; ++i) mbar_init(&s_full[i], 1);
    for (int i = 0; i < kStages; ++i) mbar_init(&s_empty[i], W ? 1 : NC);
    for (int i = 0; i < kBufs; ++i) {
      mbar_init(&s_inbar[i], 1);
      s_pslot[i] = -1;
      s_pevict[i] = 0;
    }
    mbar_init(&s_part[0], NC);
    mbar_init(&s_part[1], NC);
    for (int i = 0; i < 4; ++i) mbar_init(&s_dec[i], 1);
    mbar_init(&s_oldv, 1);
    mbar_init(&s_bml, 1);
    mbar_init(&s_bacc[0], 1);
    mbar_init(&s_bacc[1], 1);
    mbar_init(&s_bcand, 1);
    s_abort = 0;
    s_tp = 0;
    s_pw = 0;
    fence_mbar_init();
  }
  for (int j = tid; j < own; j += kThreads) {
    sc[j] = c.score[hk + s0 + j];
    cm[j] = 0.f;
    ps[j] = c.pos[hk + s0 + j];
    if (kFp8) {
      ksc[j] = c.Ksc[hk + s0 + j];
      vsc[j] = c.Vsc[hk + s0 + j];
    }
  }
  __syncthreads();
  if (kResident) {  // all owned rows, once
    if (tid == 0 && own > 0) {
      mbar_expect_tx(&s_full[0], 2u * own * ROWB);
      bulk_load(kv, (const uint8_t *)c.K + (hk + s0) * ROWB, own * ROWB, &s_full[0]);
      bulk_load(kv + chunk * ROWB, (const uint8_t *)c.V + (hk + s0) * ROWB, own * ROWB, &s_full[0]);
    }
    if (own > 0 && !__all_sync(FULL, mbar_wait(&s_full[0], 0)) && lane == 0) s_abort = 1;
  }
  // The step inputs (q, k_t, v_t rows) go to buffer u % 3, three steps ahead.
  auto fetch_inputs = [&](int u) {
    const size_t off = (size_t)u * step_elems + (size_t)h * D;
    uint64_t *bar = &s_inbar[u % kBufs];
    mbar_expect_tx(bar, 3 * D * (int)sizeof(T));
    bulk_load(s_in[u % kBufs][0], (const T *)a.s.q + off, D * sizeof(T), bar);
    bulk_load(s_in[u % kBufs][1], (const T *)a.s.kn + off, D * sizeof(T), bar);
    bulk_load(s_in[u % kBufs][2], (const T *)a.s.vn + off, D * sizeof(T), bar);
  };
  if (tid == 32 * NC)
    for (int u = 0; u < kBufs && u < a.nsteps; ++u) fetch_inputs(u);
  __syncthreads();
  // The exchange barriers must be initialised in every CTA before any peer
  // pushes into them.
  cluster.sync();

  if (warp < NC) {
    // =================================================================
    // Consumers: step t's attention pass over the rows of S_{t-1}, with the
    // slot of decision t-2 read from that decision's pending row.
    int g = 0;  // ring position of the step's first slab
    for (int t = 0; t < a.nsteps; ++t) {
      if (*(volatile int *)&s_abort) break;
      bool ok = __all_sync(FULL, mbar_wait(&s_inbar[t % kBufs], (t / kBufs) & 1));
      int pe = -1;  // row of this CTA that decision t-2 wrote (patched from its pending copy)
      const uint8_t *pk = nullptr, *pv = nullptr;
      float pks = 0.f, pvs = 0.f;
      if (ok && t >= 2) {
        ok = __all_sync(FULL, mbar_wait(&s_dec[(t - 2) & 3], ((t - 2) >> 2) & 1));
        const int q2 = (t - 2) % kBufs;
        pe = s_pslot[q2];
        pk = s_pend[q2][0];
        pv = s_pend[q2][1];
        if (kFp8) {
          pks = s_pksc[q2];
          pvs = s_pvsc[q2];
        }
      }
      if (!ok) {
        if (lane == 0) {
          s_abort = 1;
          atomicOr(c.err, 1);
        }
        break;
      }
      const T *in_q = s_in[t % kBufs][0];
      float *lg = lgb + (t & 1) * chunk;
      const int rows_t = rows_after(t > 0 ? t - 1 : 0);
      const int nslab = (rows_t + TR - 1) / TR;
      float *wacc = s_wacc[t & 1][warp];
      if constexpr (W) {
        // Wide rows: one warp per 16-row slab (layout below).  The
        // slab at ring position x goes to warp x mod NC whatever its step:
        // consumer warps are not in step with one another, and each full
        // barrier (x mod (stages * NC)) must be waited on by one warp only,
        // in order, so that no wait can be satisfied by an earlier phase.
        // Two lanes per row: lane i takes row i % 16 of a 16-row slab and
        // its dimensions 64 * (i / 16) .. +63 (eight 16-byte chunks walked in
        // an order rotated by the row, q rotated the same way); one shuffle
        // adds the two halves.  V: lane i owns output dimensions 4i .. 4i+3.
        const int vr = lane & 15, hh = lane >> 4;
        uint32_t qr[8][4];
#pragma unroll
        for (int cch = 0; cch < 8; ++cch) {
          const uint4 u = *(const uint4 *)(in_q + hh * 64 + (((cch + vr) & 7) << 3));
          qr[cch][0] = u.x; qr[cch][1] = u.y; qr[cch][2] = u.z; qr[cch][3] = u.w;
        }
        // two accumulator sets (even and odd rows) halve the dependent chain
        // of the V rows' FMAs
        float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f}, acc2[4] = {0.f, 0.f, 0.f, 0.f};
        for (int i = (warp + NC - g % NC) % NC; i < nslab; i += NC) {
          const int gi = g + i;
          const int st = gi % kStages;
          const uint8_t *ks, *vs;
          if (kResident) {
            ks = kv + (size_t)i * TR * ROWB;
            vs = kv + (size_t)chunk * ROWB + (size_t)i * TR * ROWB;
          } else {
            if (!(ok = __all_sync(FULL, mbar_wait(&s_full[gi % kFullBars], (gi / kFullBars) & 1)))) break;
            ks = kv + st * 2 * SB;
            vs = ks + SB;
          }
          const int rows = min(TR, rows_t - i * TR);
          const int plane = pe - i * TR;                  // patched row of this slab, if in [0, rows)
          const bool pin = (unsigned)plane < (unsigned)rows;  // warp-uniform
          const bool valid = vr < rows;
          const uint8_t *krow = ((pin && vr == plane) ? pk : ks + (valid ? vr : 0) * ROWB) + hh * 128;
          float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
          for (int cch = 0; cch < 8; ++cch) {
            const uint4 kc = *(const uint4 *)(krow + (((cch + vr) & 7) << 4));
            float dd = d4[cch & 3];
            dd = fma2_bf16(qr[cch][0], kc.x, dd);
            dd = fma2_bf16(qr[cch][1], kc.y, dd);
            dd = fma2_bf16(qr[cch][2], kc.z, dd);
            dd = fma2_bf16(qr[cch][3], kc.w, dd);
            d4[cch & 3] = dd;
          }
          float lgt = (d4[0] + d4[1]) + (d4[2] + d4[3]);
          lgt = (lgt + __shfl_xor_sync(FULL, lgt, 16)) * a.qscale;
          lgt = valid ? lgt : -INFINITY;
          if (valid && hh == 0) lg[i * TR + vr] = lgt;
          const float wmax = warp_max_ordered(lgt);
          if (wmax > m) {
            const float sc_ = ex2(m - wmax);
            l *= sc_;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              acc[u] *= sc_;
              acc2[u] *= sc_;
            }
            m = wmax;
          }
          const float pr = valid ? ex2(lgt - m) : 0.f;
          if (hh == 0) l += pr;  // each row once
          const float pwv = (pin && vr == plane) ? 0.f : pr;  // the patched row's V comes from its pending copy
          const uint8_t *vcol = vs + lane * 8;
          auto vrow = [&](int r) {
            const float w = __shfl_sync(FULL, pwv, r);
            const uint2 v = *(const uint2 *)(vcol + r * ROWB);
            float *ac = (r & 1) ? acc2 : acc;
            fma_pair(ac[0], ac[1], w, bf16lo(v.x), bf16hi(v.x));
            fma_pair(ac[2], ac[3], w, bf16lo(v.y), bf16hi(v.y));
          };
          if (rows == TR) {
#pragma unroll
            for (int r = 0; r < TR; ++r) vrow(r);
          } else {
            for (int r = 0; r < rows; ++r) vrow(r);
          }
          if (pin) {
            const float w = __shfl_sync(FULL, pr, plane);
            const uint2 v = *(const uint2 *)(pv + lane * 8);
            fma_pair(acc[0], acc[1], w, bf16lo(v.x), bf16hi(v.x));
            fma_pair(acc[2], acc[3], w, bf16lo(v.y), bf16hi(v.y));
          }
          if (!kResident) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[st]);
          }
        }
        l = warp_sum(l);
#pragma unroll
        for (int u = 0; u < 4; ++u) wacc[4 * lane + u] = acc[u] + acc2[u];
        if (lane == 0) {
          s_wm[t & 1][warp] = m;
          s_wl[t & 1][warp] = l;
        }
      } else {
        // Lane groups: LPR lanes per row, ITER rows per lane group per slab,
        // one transposed reduction, one exp2 per lane.
        QLane<S, EPL> qk;
        qk.load(in_q + sub * EPL, a.qscale);
        constexpr int LPI = LPR / ITER;
        float m = -INFINITY, l = 0.f, acc[EPL];
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
        const int myit = sub / LPI;
        int st = g % kStages, ph = (g / kStages) & 1;
        for (int i = 0; i < nslab; ++i) {
          const uint8_t *ks, *vs;
          if (kResident) {
            ks = kv + (size_t)i * TR * ROWB;
            vs = kv + (size_t)chunk * ROWB + (size_t)i * TR * ROWB;
          } else {
            if (!(ok = __all_sync(FULL, mbar_wait(&s_full[st], ph)))) break;
            ks = kv + st * 2 * SB;
            vs = ks + SB;
          }
          const int rows = min(TR, rows_t - i * TR);
          const int plane = pe - i * TR;
          auto slab = [&](auto full_tag) {
            constexpr bool kFull = decltype(full_tag)::value;
            float x[ITER];
#pragma unroll
            for (int it = 0; it < ITER; ++it) {
              const int r = warp * RPW + grp + it * NC * RPW;
              const int rr = (kFull || r < rows) ? r : 0;
              const uint8_t *kp = (rr == plane) ? pk : ks + rr * ROWB;
              x[it] = qk.dot(kp + sub * Lane<S>::VB);
            }
            const int rm = warp * RPW + grp + myit * NC * RPW;
            const bool valid = kFull || rm < rows;
            float lgt = xreduce<ITER, LPR>(x, sub) * qk.scale;
            if (kFp8) lgt *= valid ? (rm == plane ? pks : ksc[i * TR + rm]) : 0.f;
            lgt = valid ? lgt : -INFINITY;
            if (valid && sub % LPI == 0) lg[i * TR + rm] = lgt;
            const float wmax = warp_max_ordered(lgt);  // over the warp's rows of this slab
            if (wmax > m) {
              const float sc_ = ex2(m - wmax);
              l *= sc_;
#pragma unroll
              for (int e = 0; e < EPL; ++e) acc[e] *= sc_;
              m = wmax;
            }
            const float prm = valid ? ex2(lgt - m) : 0.f;
            if (sub % LPI == 0) l += prm;
#pragma unroll
            for (int it = 0; it < ITER; ++it) {
              const int r = warp * RPW + grp + it * NC * RPW;
              const float pr = __shfl_sync(FULL, prm, grp * LPR + it * LPI);
              if (kFull || r < rows) {
                const bool patched = r == plane;
                const float pvw = kFp8 ? pr * (patched ? pvs : vsc[i * TR + r]) : pr;
                float vx[EPL];
                unpack_lane<S>((patched ? pv : vs + r * ROWB) + sub * Lane<S>::VB, vx);
#pragma unroll
                for (int e = 0; e < EPL; e += 2) fma_pair(acc[e], acc[e + 1], pvw, vx[e], vx[e + 1]);
              }
            }
          };
          if (rows == TR)
            slab(std::true_type{});
          else
            slab(std::false_type{});
          if (!kResident) {
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_empty[st]);
            if (++st == kStages) {
              st = 0;
              ph ^= 1;
            }
          }
        }
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) l += __shfl_xor_sync(FULL, l, o);
#pragma unroll
        for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] += __shfl_xor_sync(FULL, acc[e], o);
        }
        if (grp == 0) {
#pragma unroll
          for (int e = 0; e < EPL; ++e) wacc[sub * EPL + e] = acc[e];
        }
        if (lane == 0) {
          s_wm[t & 1][warp] = m;
          s_wl[t & 1][warp] = l;
        }
      }
      if (!ok) {
        if (lane == 0) {
          s_abort = 1;
          atomicOr(c.err, 1);
        }
        break;
      }
      g += kResident ? 0 : nslab;
      __syncwarp();
      if (lane == 0) mbar_arrive(&s_part[t & 1]);
    }
  } else if (warp == NC) {
    // =================================================================
    // Protocol warp: every step's exchanges and decision.
    int tp = 0;  // decisions made
    bool failed = false;
    auto wait_bar = [&](uint64_t *bar, uint32_t par) -> bool { return __all_sync(FULL, mbar_wait(bar, par)); };
    // log2-domain logit of a step's new token against its own query
    auto new_logit = [&](const T *qq, const T *kk) -> float {
      float qv[CPL], kx[CPL];
      row_part<T, CPL>(qq, lane, qv);
      row_part<T, CPL>(kk, lane, kx);
      float dot = 0.f;
#pragma unroll
      for (int u = 0; u < CPL; ++u) dot = fmaf(qv[u], kx[u], dot);
      return warp_sum(dot) * a.qscale;
    };
    float lg_next = 0.f;  // rank 0: the next step's new-token logit

    for (int t = 0; t < a.nsteps && !failed; ++t) {
      if (*(volatile int *)&s_abort) {
        failed = true;
        break;
      }
      if (lane == 0) {  // bytes this CTA receives during step t's exchanges
        mbar_expect_tx(&s_bml, P * 16);
        mbar_expect_tx(&s_bcand, P * 16);
        if (kSplitOut)
          mbar_expect_tx(&s_bacc[t & 1], D * 4);  // every rank's values of this CTA's D/P dimensions
        else if (rank == 0)
          mbar_expect_tx(&s_bacc[t & 1], P * D * 4);
      }
      const int q = t % kBufs;
      if (!wait_bar(&s_inbar[q], (t / kBufs) & 1) || !wait_bar(&s_part[t & 1], (t >> 1) & 1)) {
        failed = true;
        break;
      }
      const T *in_q = s_in[q][0], *in_k = s_in[q][1], *in_v = s_in[q][2];
      float *lg = lgb + (t & 1) * chunk;
      const int p = a.s.p + t;
      // ---- merge the consumer warps' partials
      float M = s_wm[t & 1][0];
#pragma unroll
      for (int w = 1; w < NC; ++w) M = fmaxf(M, s_wm[t & 1][w]);
      float l = 0.f, acc[CPL];
#pragma unroll
      for (int u = 0; u < CPL; ++u) acc[u] = 0.f;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float f = (s_wm[t & 1][w] == -INFINITY) ? 0.f : exp2f(s_wm[t & 1][w] - M);
        l = fmaf(f, s_wl[t & 1][w], l);
#pragma unroll
        for (int u = 0; u < CPL; ++u) acc[u] = fmaf(f, s_wacc[t & 1][w][lane * CPL + u], acc[u]);
      }
      // ---- decision t-1 applied to this step's partial
      if (t >= 1) {
        const int q1 = (t - 1) % kBufs;
        const int j = s_pslot[q1];
        if (j >= 0) {
          if (s_pevict[q1]) {  // slot j held a row this step's pass has counted
            const uint8_t *orow;
            if (kResident) {
              orow = kv + (size_t)chunk * ROWB + (size_t)j * ROWB;
            } else {
              if (!wait_bar(&s_oldv, (t - 1) & 1)) {
                failed = true;
                break;
              }
              orow = s_oldrow;
            }
            const float po = (M == -INFINITY) ? 0.f : exp2f(lg[j] - M);
            if (po <= 0.5f * l) {
              float vo[CPL];
              row_part<S, CPL>(orow, lane, vo);
              const float wv = kFp8 ? po * vsc[j] : po;
              l -= po;
#pragma unroll
              for (int u = 0; u < CPL; ++u) acc[u] = fmaf(-wv, vo[u], acc[u]);
            } else {
              // The evicted row holds more than half of the partial mass:
              // recompute the partial over the other rows of S_{t-1}.
              const int nr = rows_after(t - 1);
              float mx = -INFINITY;
              for (int r = lane; r < nr; r += 32)
                if (r != j) mx = fmaxf(mx, lg[r]);
              mx = warp_max(mx);
              float ls = 0.f;
              for (int r = lane; r < nr; r += 32)
                if (r != j && mx != -INFINITY) ls += exp2f(lg[r] - mx);
              l = warp_sum(ls);
#pragma unroll
              for (int u = 0; u < CPL; ++u) acc[u] = 0.f;
              const int q2 = (t - 2) % kBufs;
              const int pj2 = t >= 2 ? s_pslot[q2] : -1;
              for (int r = 0; r < nr && mx != -INFINITY; ++r) {
                if (r == j) continue;
                const float w = exp2f(lg[r] - mx) * (kFp8 ? vsc[r] : 1.f);
                const void *vrow;
                if (kResident)
                  vrow = kv + (size_t)chunk * ROWB + (size_t)r * ROWB;
                else if (r == pj2)
                  vrow = s_pend[q2][1];
                else
                  vrow = (const uint8_t *)c.V + (hk + s0 + r) * (size_t)ROWB;
                float vx[CPL];
                row_part<S, CPL>(vrow, lane, vx);
#pragma unroll
                for (int u = 0; u < CPL; ++u) acc[u] = fmaf(w, vx[u], acc[u]);
              }
              M = mx;
            }
          }
          __syncwarp();
          if (kFp8 && lane == 0) {
            ksc[j] = s_pksc[q1];
            vsc[j] = s_pvsc[q1];
          }
          // the admitted token's row, as stored, attended by this step's query
          float qv[CPL], kx[CPL], vx[CPL];
          row_part<T, CPL>(in_q, lane, qv);
          row_part<S, CPL>(s_pend[q1][0], lane, kx);
          float dot = 0.f;
#pragma unroll
          for (int u = 0; u < CPL; ++u) dot = fmaf(qv[u], kx[u], dot);
          dot = warp_sum(dot) * a.qscale * (kFp8 ? s_pksc[q1] : 1.f);
          const float mn = fmaxf(M, dot);
          const float scl = (M == -INFINITY) ? 0.f : exp2f(M - mn);
          const float pn = exp2f(dot - mn);
          l = fmaf(l, scl, pn);
          row_part<S, CPL>(s_pend[q1][1], lane, vx);
          const float wn = kFp8 ? pn * s_pvsc[q1] : pn;
#pragma unroll
          for (int u = 0; u < CPL; ++u) acc[u] = fmaf(wn, vx[u], acc[u] * scl);
          M = mn;
          __syncwarp();
          if (lane == 0) lg[j] = dot;
        }
      }
      // ---- rank 0: the step's new token, from the step inputs (its logit
      // taken in advance while the previous step waited for candidates)
      float lgnew = 0.f;
      if (rank == 0) {
        float vx[CPL];
        lgnew = t == 0 ? new_logit(in_q, in_k) : lg_next;
        const float mn = fmaxf(M, lgnew);
        const float scl = (M == -INFINITY) ? 0.f : exp2f(M - mn);
        const float pn = exp2f(lgnew - mn);
        l = fmaf(l, scl, pn);
        row_part<T, CPL>(in_v, lane, vx);
#pragma unroll
        for (int u = 0; u < CPL; ++u) acc[u] = fmaf(pn, vx[u], acc[u] * scl);
        M = mn;
      }
      // ---- exchange 1: (m, l, new-token logit) to every rank; the acc row to
      // rank 0, or each group of D/P dimensions to the rank that writes them
      {
        const int dim = lane * CPL, dst_rank = kSplitOut ? dim / DPR : 0;
        const uint32_t dst = mapa(&accx[((t & 1) * P + rank) * DPR + dim % DPR], dst_rank),
                       bar0 = mapa(&s_bacc[t & 1], dst_rank);
        if constexpr (CPL == 4) {
          st_async_v4(dst, make_uint4(__float_as_uint(acc[0]), __float_as_uint(acc[1]), __float_as_uint(acc[2]),
                                      __float_as_uint(acc[3])),
                      bar0);
        } else {
          st_async_b64(dst, ((uint64_t)__float_as_uint(acc[1]) << 32) | __float_as_uint(acc[0]), bar0);
        }
        if (lane < P)
          st_async_v4(mapa(&s_mlx[rank], lane),
                      make_uint4(__float_as_uint(M), __float_as_uint(l), __float_as_uint(lgnew), 0u),
                      mapa(&s_bml, lane));
      }
      if (kResident && t >= 1 && s_pslot[(t - 1) % kBufs] >= 0) {
        // Decision t-1's row into the resident copy and the cache rows in
        // HBM, off the exchange's path: the consumers read slot j from the
        // pending copy until decision t is made, and nothing in this launch
        // reads the rows in HBM.
        const int q1 = (t - 1) % kBufs, j = s_pslot[q1];
        warp_copy(kv + (size_t)j * ROWB, s_pend[q1][0], ROWB, lane);
        warp_copy(kv + (size_t)chunk * ROWB + (size_t)j * ROWB, s_pend[q1][1], ROWB, lane);
        const size_t off = (hk + s0 + j) * (size_t)ROWB;
        warp_copy((uint8_t *)c.K + off, s_pend[q1][0], ROWB, lane);
        warp_copy((uint8_t *)c.V + off, s_pend[q1][1], ROWB, lane);
        __syncwarp();
      }
      if (!wait_bar(&s_bml, t & 1)) {
        failed = true;
        break;
      }
      float mr = -INFINITY, lr = 0.f;
      if (lane < P) {
        mr = __uint_as_float(s_mlx[lane].x);
        lr = __uint_as_float(s_mlx[lane].y);
      }
      // lanes 0..P-1 (P <= 8) hold the ranks' values: three butterfly levels
      // reduce them in lanes 0..7, lane 0 gives the result to the warp
      float Mg = mr;
#pragma unroll
      for (int o = kMaxCluster / 2; o; o >>= 1) Mg = fmaxf(Mg, __shfl_xor_sync(FULL, Mg, o));
      const float fr = (mr == -INFINITY) ? 0.f : exp2f(mr - Mg);
      float Lg = fr * lr;
#pragma unroll
      for (int o = kMaxCluster / 2; o; o >>= 1) Lg += __shfl_xor_sync(FULL, Lg, o);
      Mg = __shfl_sync(FULL, Mg, 0);
      const float invL = 1.f / __shfl_sync(FULL, Lg, 0);
      // ---- exact weights into the scores of S_t; local argmin
      const int nr = rows_after(t);
      const long long lim = (long long)p - c.kl;
      ArgMin best{INFINITY, INT_MAX, -2};
      // four entries per lane at a time, all loaded before any is stored
      for (int j0 = lane; j0 < nr; j0 += 128) {
        float lv[4], sv[4], cv[4];
        int pv[4];
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + 32 * u;
          if (j < nr) {
            lv[u] = lg[j];
            sv[u] = sc[j];
            cv[u] = cm[j];
            pv[u] = ps[j];
          }
        }
#pragma unroll
        for (int u = 0; u < 4; ++u) {
          const int j = j0 + 32 * u;
          if (j < nr) {
            kahan_add(sv[u], cv[u], exp2f(lv[u] - Mg) * invL);
            sc[j] = sv[u];
            cm[j] = cv[u];
            if ((long long)pv[u] <= lim && pv[u] >= c.n_sink) {
              const ArgMin cand{rank_key(sv[u], p, pv[u], c.score_mode), pv[u], s0 + j};
              if (am_less(cand, best)) best = cand;
            }
          }
        }
      }
      const float w_new = exp2f(__uint_as_float(s_mlx[0].z) - Mg) * invL;
      if (rank == 0 && lane == 0 && c.kl == 0 && p >= c.n_sink) {
        const ArgMin cand{w_new, p, -1};
        if (am_less(cand, best)) best = cand;
      }
      best = warp_argmin(best);
      if (lane < P)
        st_async_v4(mapa(&s_candx[rank], lane),
                    make_uint4(__float_as_uint(best.s), (uint32_t)best.p, (uint32_t)best.slot, 0u),
                    mapa(&s_bcand, lane));
      if (kSplitOut) {
        // This CTA's dimensions of the step's output row, off the path to the
        // decision: step t's values sit in buffer t & 1, which the ranks
        // refill only with step t+2's, after this CTA's candidate of step t+1.
        if (!wait_bar(&s_bacc[t & 1], (t >> 1) & 1)) {
          failed = true;
          break;
        }
        const float *ax = accx + (t & 1) * P * DPR;
        T *out = (T *)a.s.out + (size_t)t * step_elems + (size_t)h * D + rank * DPR;
        for (int d0 = 0; d0 < DPR; d0 += 32) {
          float o = 0.f;
          for (int r = 0; r < P; ++r) {
            const float f = __shfl_sync(FULL, fr, r);
            if (d0 + lane < DPR && f != 0.f) o = fmaf(f, ax[r * DPR + d0 + lane], o);
          }
          if (d0 + lane < DPR) out[d0 + lane] = from_f32<T>(o * invL);
        }
      } else if (rank == 0) {
        // The step's output row, off the path to the decision: the acc rows
        // of step t sit in buffer t & 1, which the ranks refill only with
        // step t+2's rows, after this CTA's candidate of step t+1.
        if (!wait_bar(&s_bacc[t & 1], (t >> 1) & 1)) {
          failed = true;
          break;
        }
        const float *ax = accx + (t & 1) * P * D;
        float o[CPL];
#pragma unroll
        for (int u = 0; u < CPL; ++u) o[u] = 0.f;
        for (int r = 0; r < P; ++r) {
          const float f = __shfl_sync(FULL, fr, r);
          if (f != 0.f) {
#pragma unroll
            for (int u = 0; u < CPL; ++u) o[u] = fmaf(f, ax[r * D + lane * CPL + u], o[u]);
          }
        }
        T *out = (T *)a.s.out + (size_t)t * step_elems + (size_t)h * D;
#pragma unroll
        for (int u = 0; u < CPL; ++u) out[lane * CPL + u] = from_f32<T>(o[u] * invL);
      }
      if (rank == 0 && t + 1 < a.nsteps) {  // the next step's new-token logit, while candidates travel
        const int qn = (t + 1) % kBufs;
        if (!wait_bar(&s_inbar[qn], ((t + 1) / kBufs) & 1)) {
          failed = true;
          break;
        }
        lg_next = new_logit(s_in[qn][0], s_in[qn][1]);
      }
      if (!wait_bar(&s_bcand, t & 1)) {
        failed = true;
        break;
      }
      // ---- the decision (identical in every CTA)
      ArgMin b{INFINITY, INT_MAX, -2};
      if (lane < P) {
        const uint4 cv = s_candx[lane];
        b = ArgMin{__uint_as_float(cv.x), (int)cv.y, (int)cv.z};
      }
      b = warp_argmin(b);
      const int n = (int)min((long long)a.s.n_valid + t, (long long)c.k);
      int e = -1, ev = -1;
      if (n < c.k) {
        e = n;  // |S| < k: admit into the next free slot
      } else if (b.slot == -2) {
        if (lane == 0 && rank == 0) atomicOr(c.err, 1);  // no eviction candidate: inconsistent state
      } else if (b.slot == -1) {
        ev = p;  // the new token itself scores lowest (k_local = 0)
      } else {
        e = b.slot;
        ev = b.p;
      }
      if (lane == 0 && rank == 0 && a.s.evicted) a.s.evicted[(size_t)t * c.nh + h] = ev;
      // pending buffer q is free once decision t-3 is in the cache rows
      if (!kResident) {
        for (uint32_t i = 0; *(volatile int *)&s_pw <= t - 3; ++i) {
          if (i >= kSpinLimit || *(volatile int *)&s_abort) {
            failed = true;
            break;
          }
          __nanosleep(32);
        }
        if (failed) break;
        __threadfence_block();
      }
      const bool mine = e >= s0 && e < s0 + own;
      const int j = e - s0;
      const int q1 = (t - 1) % kBufs, q2 = (t - 2) % kBufs;
      const int pj1 = t >= 1 ? s_pslot[q1] : -1, pj2 = t >= 2 ? s_pslot[q2] : -1;
      __syncwarp();
      if (mine) {
        if (lane == 0) {
          ps[j] = p;
          sc[j] = w_new;
          cm[j] = 0.f;
          s_pslot[q] = j;
          s_pevict[q] = n >= c.k;
        }
        if constexpr (kFp8) {
          constexpr int PER = D / 32;
          float xk[PER], xv[PER], sk, sv;
          row_part<T, PER>(in_k, lane, xk);
          row_part<T, PER>(in_v, lane, xv);
          store_codes<PER>(s_pend[q][0], lane, quant_row_e4m3<PER>(xk, sk));
          store_codes<PER>(s_pend[q][1], lane, quant_row_e4m3<PER>(xv, sv));
          if (lane == 0) {
            s_pksc[q] = sk;
            s_pvsc[q] = sv;
          }
        } else {
          warp_copy(s_pend[q][0], in_k, ROWB, lane);
          warp_copy(s_pend[q][1], in_v, ROWB, lane);
        }
        __syncwarp();
        if (kResident) {
          // the row goes to the resident copy and HBM during the next step
        } else if (n >= c.k) {
          // The row S_t holds in slot j (its V is needed when decision t is
          // applied to step t+1): the pending copy of decision t-1 or t-2 if
          // one of them wrote slot j, else the cache row in HBM.
          if (j == pj1 || j == pj2) {
            warp_copy(s_oldrow, s_pend[j == pj1 ? q1 : q2][1], ROWB, lane);
            __syncwarp();
            if (lane == 0) mbar_arrive(&s_oldv);
          } else if (lane == 0) {
            mbar_expect_tx(&s_oldv, ROWB);
            bulk_load(s_oldrow, (const uint8_t *)c.V + (hk + e) * (size_t)ROWB, ROWB, &s_oldv);
          }
        } else if (lane == 0) {
          mbar_arrive(&s_oldv);
        }
      } else {
        if (lane == 0) {
          s_pslot[q] = -1;
          s_pevict[q] = 0;
          if (!kResident) mbar_arrive(&s_oldv);
        }
      }
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(&s_dec[t & 3]);
        __threadfence_block();
        *(volatile int *)&s_tp = t + 1;
        if (t + kBufs < a.nsteps) fetch_inputs(t + kBufs);  // buffer q: step t is done with it
      }
      tp = t + 1;
    }
    if (failed && lane == 0) {
      s_abort = 1;
      atomicOr(c.err, 1);
    }
    if (tp > 0 && !failed) {  // the last decision (no next step applies it)
      const int q = (tp - 1) % kBufs, j = s_pslot[q];
      if (j >= 0) {
        if (kFp8 && lane == 0) {
          ksc[j] = s_pksc[q];
          vsc[j] = s_pvsc[q];
        }
        if (kResident) {
          const size_t off = (hk + s0 + j) * (size_t)ROWB;
          warp_copy((uint8_t *)c.K + off, s_pend[q][0], ROWB, lane);
          warp_copy((uint8_t *)c.V + off, s_pend[q][1], ROWB, lane);
        }
      }
    }
    // inputs fetched for steps that never ran (an aborted call) must land too
    if (lane == 0)
      for (int u = tp; u < a.nsteps && u < tp + kBufs; ++u) mbar_wait(&s_inbar[u % kBufs], (u / kBufs) & 1);
  } else if (!kResident) {
    // =================================================================
    // Producer warp (streaming form): the slabs of every step, in ring
    // order (lane 0 issues), and each decision's row written back to the
    // cache rows in HBM (the whole warp).
    bool ok = true;
    int gp = 0, pw = 0;
    int gfirst[4] = {0, 0, 0, 0};  // ring position of the first slab of steps u-3 .. u (index u % 4)
    // Bounded wait for `target` decisions made.
    auto wait_decisions = [&](int target) -> bool {
      for (uint32_t i = 0; i < kSpinLimit; ++i) {
        if (*(volatile int *)&s_tp >= target) {
          __threadfence_block();
          return true;
        }
        if (*(volatile int *)&s_abort) return false;
        __nanosleep(64);
      }
      return false;
    };
    auto write_back = [&](int u) {
      const int q = u % kBufs;
      const int j = s_pslot[q];
      if (j >= 0) {
        const size_t off = (hk + s0 + j) * (size_t)ROWB;
        warp_copy((uint8_t *)c.K + off, s_pend[q][0], ROWB, lane);
        warp_copy((uint8_t *)c.V + off, s_pend[q][1], ROWB, lane);
        asm volatile("fence.proxy.async.global;" ::: "memory");  // before later bulk reads of the row
      }
      __syncwarp();
      pw = u + 1;
      __threadfence_block();
      if (lane == 0) *(volatile int *)&s_pw = pw;
    };
    for (int u = 0; u < a.nsteps && ok; ++u) {
      if (*(volatile int *)&s_abort) break;
      if (u >= 3) {
        // Step u's slabs carry decisions up to u-3 and none after.  Decision
        // u-3 is written back once step u-2's partial has taken the saved
        // copy of the row it replaced (decision u-2 made) and every slab of
        // step u-2 (the last step that reads its old row from a slab) has
        // landed.
        ok = wait_decisions(u - 1);
        for (int x = max(gfirst[(u - 2) & 3], gp - kStages); ok && x < gfirst[(u - 1) & 3]; ++x)
          ok = __all_sync(FULL, mbar_wait(&s_full[x % kFullBars], (x / kFullBars) & 1));
        if (!ok) break;
        write_back(u - 3);
      }
      gfirst[u & 3] = gp;
      const int rows = rows_after(u > 0 ? u - 1 : 0);
      const int nst = (rows + TR - 1) / TR;
      for (int i = 0; i < nst && ok; ++i) {
        const int st = gp % kStages;
        if (gp >= kStages) ok = __all_sync(FULL, mbar_wait_backoff(&s_empty[st], ((gp / kStages) - 1) & 1));
        if (ok && lane == 0) {
          const uint32_t bytes = (uint32_t)(min(TR, rows - i * TR) * ROWB);
          const size_t off = (hk + s0 + (size_t)i * TR) * ROWB;
          uint64_t *fb = &s_full[gp % kFullBars];
          mbar_expect_tx(fb, 2 * bytes);
          bulk_load(kv + st * 2 * SB, (const uint8_t *)c.K + off, bytes, fb);
          bulk_load(kv + st * 2 * SB + SB, (const uint8_t *)c.V + off, bytes, fb);
        }
        if (ok) ++gp;
      }
    }
    // Every issued slab lands before the CTA exits; the last decisions go to
    // the cache rows once they are made and the last saved V row (a bulk
    // read of the row being replaced) has arrived.
    bool drained = true;
    for (int x = max(0, gp - kStages); x < gp; ++x)
      drained = drained && __all_sync(FULL, mbar_wait(&s_full[x % kFullBars], (x / kFullBars) & 1));
    if (ok && drained && wait_decisions(a.nsteps)) {
      if (__all_sync(FULL, mbar_wait(&s_oldv, (a.nsteps - 1) & 1)))
        for (int u = pw; u < a.nsteps; ++u) write_back(u);
      else
        drained = false;
    }
    if ((!ok || !drained) && lane == 0) {
      s_abort = 1;
      atomicOr(c.err, 1);
    }
  }
  __syncthreads();
  // write back the owned scores and tags; no CTA leaves while a peer could
  // still push into its shared memory
  for (int j = tid; j < own; j += kThreads) {
    c.score[hk + s0 + j] = sc[j] - cm[j];  // the compensated sum, rounded once
    c.pos[hk + s0 + j] = ps[j];
    if (kFp8) {
      c.Ksc[hk + s0 + j] = ksc[j];
      c.Vsc[hk + s0 + j] = vsc[j];
    }
  }
  cluster.sync();
}

// Per-slot shared-memory words beside K/V: score, tag, compensation, two
// logits (+ two scales for an fp8 cache).
template <typename S> constexpr int slot_words() { return is_fp8<S>() ? 7 : 5; }

template <typename S, int D> constexpr int row_bytes() { return D * (int)sizeof(S); }

template <typename S, int D, bool R, int St, bool W = false>
int smem_bytes(int chunk, int P) {
  const int base = (R ? 2 * chunk * row_bytes<S, D>() : ring_bytes(St, W)) + slot_words<S>() * chunk * 4;
  return ((base + 15) & ~15) + 2 * (W && !R ? 1 : P) * D * 4;  // + the output exchange buffer of two steps
}

int chunk_of(const CacheView &c) { return (c.k + c.nsplit - 1) / c.nsplit; }

template <typename T, typename S, int D, bool R, int St, int NC, bool W = false>
cudaError_t launch_t(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st) {
  const int P = c.nsplit;
  PArgs a{c, s, nsteps, chunk_of(c), kLog2e / sqrtf((float)D)};
  const int smem = smem_bytes<S, D, R, St, W>(a.chunk, P);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  static bool attr_done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_pipe_kernel<T, S, D, R, St, NC, W>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
    if (e != cudaSuccess) return e;
    if (dev >= 0 && dev < 64) attr_done[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(c.nh * P));
  cfg.blockDim = dim3(threads_for(NC));
  cfg.dynamicSmemBytes = (size_t)smem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = (unsigned)P;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_pipe_kernel<T, S, D, R, St, NC, W>, a);
}

template <typename T, typename S, int D, bool R, int St, int NC, bool W = false>
bool all_resident(const CacheView &c, int chunk) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return false;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return false;
  const int smem = smem_bytes<S, D, R, St, W>(chunk, c.nsplit);
  if (smem > 200 * 1024) return false;
  if (cudaFuncSetAttribute(decode_pipe_kernel<T, S, D, R, St, NC, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           200 * 1024) != cudaSuccess)
    return false;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_pipe_kernel<T, S, D, R, St, NC, W>,
                                                    threads_for(NC), smem) != cudaSuccess)
    return false;
  return per_sm > 0 && (long long)c.nh * c.nsplit <= (long long)per_sm * sms;
}

template <typename T, typename S, int D> constexpr bool wide_rows() {
  return std::is_same<T, __nv_bfloat16>::value && std::is_same<S, __nv_bfloat16>::value && D == 128;
}

// Rows resident in shared memory when they fit and the grid is
// co-resident; the wide-row layout (four stages of 16-row slabs) for bf16
// rows of 128 and at least 64 slots per CTA; else lane groups with a
// three-stage ring, or two stages when that makes the grid co-resident.
template <typename T, typename S, int D, int NC>
cudaError_t dispatch_nc(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st) {
  const int chunk = chunk_of(c);
  if (2 * chunk * row_bytes<S, D>() <= kResidentMaxBytes && all_resident<T, S, D, true, 1, NC>(c, chunk))
    return launch_t<T, S, D, true, 1, NC>(c, s, nsteps, st);
  if constexpr (wide_rows<T, S, D>()) {
    if (chunk >= 64)
      return launch_t<T, S, D, false, 4, NC, true>(c, s, nsteps, st);
  }
  if (!all_resident<T, S, D, false, 3, NC>(c, chunk) && all_resident<T, S, D, false, 2, NC>(c, chunk))
    return launch_t<T, S, D, false, 2, NC>(c, s, nsteps, st);
  return launch_t<T, S, D, false, 3, NC>(c, s, nsteps, st);
}

template <typename T, typename S, int D>
cudaError_t dispatch_t(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st) {
  return chunk_of(c) > kShortChunk ? dispatch_nc<T, S, D, 4>(c, s, nsteps, st)
                                   : dispatch_nc<T, S, D, 2>(c, s, nsteps, st);
}

}  // namespace

// Cluster size of the pipelined form.  Shapes that take the wide-row layout
// (bf16 rows of 128, no fp8): the smallest power of two that leaves each CTA
// at most 256 slots, doubled (up to 8) while the doubled grid still fits one
// wave of five CTAs per SM.  Other shapes: the cluster form's rule.
// Measured on GB300 (us per decode step): OPT-6.7B shape (256 heads,
// k = 512) wide rows with clusters of 2: 6.50, lane groups with clusters of
// 4 (the cluster form's rule): 6.91, wide rows with clusters of 4: 7.51.
int decode_pipe_cluster_size(const CacheView &c, int sms) {
  if (!(c.dtype == 1 && !c.kv_fp8 && c.d == 128)) return decode_cluster_size(c.nh, c.k, sms);
  int P = 1;
  while (P < kMaxCluster && (c.k + P - 1) / P > kShortChunk) P *= 2;
  if ((c.k + P - 1) / P < 64) return decode_cluster_size(c.nh, c.k, sms);  // lane groups (or resident rows)
  const long long wave = 5LL * (sms > 0 ? sms : 1);
  while (P < kMaxCluster && (long long)c.nh * P * 2 <= wave) P *= 2;
  return P;
}

bool decode_pipe_supported(const CacheView &c) {
  if (c.nsplit < 1 || c.nsplit > kMaxCluster) return false;
  if (!(c.d == 64 || c.d == 128)) return false;
  const int chunk = (c.k + c.nsplit - 1) / c.nsplit;
  const int row = c.d * (c.kv_fp8 ? 1 : c.dtype == 1 ? 2 : 4);
  const int kv = (2 * chunk * row <= kResidentMaxBytes) ? 2 * chunk * row : ring_bytes(3);
  return kv + (c.kv_fp8 ? 7 : 5) * chunk * 4 + 16 + 2 * c.nsplit * c.d * 4 <= 200 * 1024;
}

cudaError_t launch_decode_pipe(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st) {
  if (!decode_pipe_supported(c) || nsteps < 1) return cudaErrorInvalidValue;
  if (c.dtype == 1 && c.kv_fp8) {
    if (c.d == 128) return dispatch_t<__nv_bfloat16, e4m3, 128>(c, s, nsteps, st);
    if (c.d == 64) return dispatch_t<__nv_bfloat16, e4m3, 64>(c, s, nsteps, st);
  } else if (c.dtype == 1) {
    if (c.d == 128) return dispatch_t<__nv_bfloat16, __nv_bfloat16, 128>(c, s, nsteps, st);
    if (c.d == 64) return dispatch_t<__nv_bfloat16, __nv_bfloat16, 64>(c, s, nsteps, st);
  } else if (!c.kv_fp8) {
    if (c.d == 128) return dispatch_t<float, float, 128>(c, s, nsteps, st);
    if (c.d == 64) return dispatch_t<float, float, 64>(c, s, nsteps, st);
  }
  return cudaErrorInvalidValue;
}

}  // namespace h2o
