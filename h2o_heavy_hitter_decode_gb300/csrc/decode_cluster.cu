// decode_cluster.cu — many H2O decode steps in one launch, one thread-block
// cluster per (batch, head).
//
// Same method as decode.cu (H2O summary page, "Algorithm / figure
// walkthrough" steps 2-4): attend over the cache plus the new token, add each
// exact weight to its entry's accumulated score, evict the lowest (score,
// position) outside the k_local newest positions, write the new token in place.
//
// Layout of the work: the cluster's P CTAs split the head's k slots into
// fixed ranges of `chunk` slots; CTA r owns slots [r*chunk, (r+1)*chunk).
// Scores, position tags and the step's logits of its slots live in the CTA's
// shared memory for the whole launch (read at the start, written back at the
// end); within the launch each score is a compensated (Kahan) sum of its
// weights, folded into the stored fp32 score at the end, so a score that
// collects millions of small weights over a long stream stays accurate; K/V rows are streamed from HBM each step (4 KB cp.async.bulk slabs in
// a 2- or 3-stage ring fed by a producer warp, which also issues the next
// step's first slabs while the cluster exchanges partials) or, when a CTA's
// rows fit and the grid is co-resident, loaded once and kept in shared
// memory.  Per step:
//   1. consumer warps: K dot products from packed q, a transposed reduction
//      per lane group, per-warp online softmax -> the CTA's (m, l, acc[d])
//      (rank 0 also takes the new token);
//   2. each CTA pushes (m, l) (and rank 0 its new-token logit) to every rank
//      and its acc row to rank 0 with st.async stores that complete on the
//      receiver's mbarrier; every CTA derives the global (M, L), and rank
//      0's producer warp merges the acc rows into the output row while its
//      consumer warps go on with step 3;
//   3. every CTA turns its logits into exact weights exp2(s - M) / L, adds
//      them to its scores, takes its local (key, position) argmin over
//      eligible slots and pushes it to every rank;
//   4. every CTA reduces the P candidates to the same decision (admit /
//      evict / drop the new token);
//   5. the owner of the chosen slot writes the new token's K/V row (HBM, its
//      resident copy, and the next step's slab if it was already loaded) and
//      its position tag and score.
// An fp8 cache (S = e4m3) streams 1-byte codes; the owned rows' K and V
// scales stay in shared memory beside the scores, each logit is scaled by its
// K scale and each V row weighted by its V scale, and the owner quantises the
// new token's row (one scale per row) when it writes it.
// All synchronisation is a CTA barrier or an mbarrier (bounded waits; the
// cluster barrier only at the start and the end); there is no global atomic,
// fence round trip or spin between CTAs, and clusters never wait on one
// another.
#include <cooperative_groups.h>

#include <climits>

#include "common.cuh"
#include "sm100.cuh"

namespace cg = cooperative_groups;

namespace h2o {
namespace {

using namespace sm100;

// Consumer warps per CTA (NC, a template argument): two when a CTA owns at
// most kShortChunk slots — each warp takes more rows per slab (the per-slab
// wait, reduction and arrive spread over more rows) and fewer warps run the
// per-step code — and four for longer per-CTA streams, which need more loads
// in flight per CTA (both measured on GB300).
constexpr int kShortChunk = 256;
constexpr int threads_for(int nc) { return 32 * nc + 32; }  // + one producer warp
constexpr int kMaxCluster = 8;
// Bytes per operand per slab: 4 KB for the lane-group layout; 8 KB (32 rows)
// for the wide-row layout (W), where one warp takes a whole slab.
constexpr int stage_bytes(bool wide) { return wide ? 8192 : 4096; }
constexpr int ring_bytes(int stages, bool wide = false) { return stages * 2 * stage_bytes(wide); }
constexpr int kResidentMaxBytes = 96 * 1024;  // K+V rows of one CTA kept in shared memory

template <typename S, int D, int NC, bool W = false> struct Geo {
  static constexpr int EPL = Lane<S>::VB / (int)sizeof(S);  // elements per lane per load
  static constexpr int LPR = D / EPL;
  static constexpr int RPW = 32 / LPR;
  static constexpr int ROWB = D * (int)sizeof(S);
  static constexpr int SB = stage_bytes(W);
  static constexpr int TR = SB / ROWB;  // rows per slab
  static constexpr int ITER = W ? 1 : TR / (NC * RPW);
  static_assert(W ? (TR == 32 && ROWB == 256) : (ITER >= 1 && TR % (NC * RPW) == 0),
                "slab must split evenly over warps (wide: 32 bf16 rows of 128)");
};

struct CArgs {
  CacheView c;
  DecodeStep s;  // first step; step i adds i * nh * d elements to q/k/v/out, i * nh to evicted
  int nsteps;
  int chunk;     // slots per CTA
  float qscale;  // log2(e) / sqrt(d)
};

template <int NC> __device__ __forceinline__ void consumers_sync() {
  asm volatile("bar.sync 1, %0;" ::"n"(32 * NC) : "memory");
}

// T: type of the step inputs and outputs; S: type of the stored K/V rows;
// NC: consumer warps; W: wide-row layout (bf16 rows of 128, see the consumer
// loop).
template <typename T, typename S, int D, bool kResident, int kStages, int NC, bool W>
__global__ void __launch_bounds__(threads_for(NC), W ? (kStages == 2 ? 5 : 4) : 7)
    decode_cluster_kernel(const CArgs a) {
  constexpr int kConsumers = NC, kConsumerThreads = 32 * NC, kThreads = threads_for(NC);
  using G = Geo<S, D, NC, W>;
  constexpr int SB = G::SB;
  constexpr bool kFp8 = is_fp8<S>();
  constexpr int EPL = G::EPL, LPR = G::LPR, RPW = G::RPW, ROWB = G::ROWB, TR = G::TR, ITER = G::ITER;
  cg::cluster_group cluster = cg::this_cluster();
  extern __shared__ __align__(1024) uint8_t smem[];
  // Full barriers: one per ring stage, or (wide layout) one per stage and
  // consumer warp: slab g signals s_full[g % kFullBars].  In the wide layout
  // warps take slabs in turn, so a stage's consecutive slabs go to different
  // warps; with a barrier per (stage, warp) every barrier is waited on by one
  // warp only, in order, and no wait can run a phase ahead of its barrier.
  constexpr int kFullBars = W ? kStages * NC : kStages;
  __shared__ uint64_t s_full[kFullBars], s_empty[kStages];
  __shared__ uint64_t s_inbar[2];                      // step inputs landed (one phase per use)
  __shared__ __align__(16) T s_in[2][3][D];            // q, k_t, v_t of two steps
  __shared__ float s_wm[kConsumers], s_wl[kConsumers];
  __shared__ float s_wacc[kConsumers][D];
  // Exchange buffers, filled by the peers' asynchronous DSMEM stores
  // (pushes), each tracked by an mbarrier of this CTA that completes one
  // phase per step when its bytes have arrived; read locally after the wait.
  __shared__ __align__(8) uint64_t s_bml, s_bacc, s_bcand;
  // every rank's (m, l) (and rank 0's new-token logit), in every CTA
  __shared__ __align__(16) uint4 s_mlx[kMaxCluster];
  __shared__ __align__(16) uint4 s_candx[kMaxCluster];     // every rank's candidate, in every CTA
  __shared__ float s_ML[2], s_lgnew, s_f[kMaxCluster];
  __shared__ ArgMin s_am[kConsumers];
  __shared__ int s_abort;
  __shared__ int s_spec;  // slabs of the next step the producer issued ahead

  const CacheView &c = a.c;
  const int P = (int)cluster.num_blocks();
  const int rank = (int)cluster.block_rank();
  const int h = blockIdx.x / P;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int sub = lane % LPR, grp = lane / LPR;
  const int chunk = a.chunk;
  const int s0 = rank * chunk;
  const int own = max(0, min(c.k, s0 + chunk) - s0);  // slots owned
  const size_t hk = (size_t)h * c.k;
  const size_t step_elems = (size_t)c.nh * D;

  // dynamic shared memory: [ring or resident K|V][score][pos][logit][score
  // compensation] (+ [K scale][V scale] for an fp8 cache)[every rank's acc
  // row, P x D, read on rank 0]
  uint8_t *kv = smem;
  const int kv_bytes = kResident ? 2 * chunk * ROWB : ring_bytes(kStages, W);
  float *sc = (float *)(smem + kv_bytes);
  int *ps = (int *)(sc + chunk);
  float *lg = (float *)(ps + chunk);
  float *cm = lg + chunk;  // Kahan compensation of each owned score, for this launch
  float *ksc = cm + chunk;
  float *vsc = ksc + chunk;
  float *accx = (float *)(smem + ((kv_bytes + (kFp8 ? 6 : 4) * chunk * 4 + 15) & ~15));

  if (tid == 0) {
    for (int i = 0; i < kFullBars; ++i) mbar_init(&s_full[i], 1);
    for (int i = 0; i < kStages; ++i) {
      mbar_init(&s_empty[i], W ? 1 : kConsumers);  // wide: one warp takes a slab
    }
    mbar_init(&s_inbar[0], 1);
    mbar_init(&s_inbar[1], 1);
    mbar_init(&s_bml, 1);
    mbar_init(&s_bacc, 1);
    mbar_init(&s_bcand, 1);
    s_abort = 0;
    s_spec = 0;
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
    if (own > 0 && !__all_sync(0xffffffffu, mbar_wait(&s_full[0], 0)) && lane == 0) s_abort = 1;
    __syncthreads();
  }

  // Step inputs do not depend on the cache: the producer lane copies each
  // step's q, k_t and v_t rows into shared memory one step ahead.
  auto fetch_inputs = [&](int st_i) {
    const size_t off = (size_t)st_i * step_elems + (size_t)h * D;
    uint64_t *bar = &s_inbar[st_i & 1];
    mbar_expect_tx(bar, 3 * D * (int)sizeof(T));
    bulk_load(s_in[st_i & 1][0], (const T *)a.s.q + off, D * sizeof(T), bar);
    bulk_load(s_in[st_i & 1][1], (const T *)a.s.kn + off, D * sizeof(T), bar);
    bulk_load(s_in[st_i & 1][2], (const T *)a.s.vn + off, D * sizeof(T), bar);
  };
  if (tid == kConsumerThreads) fetch_inputs(0);

  // The exchange barriers must be initialised in every CTA before any peer
  // pushes into them.
  cluster.sync();

  int g = 0;   // slabs consumed (ring position), consumers
  int gp = 0;  // slabs issued (ring position), producer lane
  for (int step = 0; step < a.nsteps; ++step) {
    if (*(volatile int *)&s_abort) break;  // uniform: read after the previous step's CTA barrier
    if (tid == 0) {  // bytes this CTA receives during the step
      mbar_expect_tx(&s_bml, P * 16);
      mbar_expect_tx(&s_bcand, P * 16);
      if (rank == 0) mbar_expect_tx(&s_bacc, P * D * 4);
    }
    // inputs of this step (buffer step&1) and, ahead, of the next one
    if (tid == kConsumerThreads && step + 1 < a.nsteps) fetch_inputs(step + 1);
    if (!__all_sync(0xffffffffu, mbar_wait(&s_inbar[step & 1], (step >> 1) & 1)) && lane == 0) s_abort = 1;
    const T *in_q = s_in[step & 1][0], *in_k = s_in[step & 1][1], *in_v = s_in[step & 1][2];
    const int n = min(a.s.n_valid + step, c.k);
    const int p = a.s.p + step;
    const int nrows = max(0, min(own, n - s0));  // owned slots already filled
    const int nst = kResident ? 0 : (nrows + TR - 1) / TR;
    const bool aborted = *(volatile int *)&s_abort;
    if (warp == kConsumers) {
      // ---- producer (streaming form only).  Slabs [spec, nst) of this step,
      // then the first slabs of the next step ahead of its decision: they land
      // while the cluster exchanges partials; the owner of the slot that
      // changes patches that row in the landed slab (below).
      if (!kResident && lane == 0 && !aborted) {
        bool ok = true;
        auto issue = [&](int i, int step_rows) -> bool {  // slab i of a step with `step_rows` owned rows
          const int st = gp % kStages;
          if (gp >= kStages && !mbar_wait_backoff(&s_empty[st], ((gp / kStages) - 1) & 1)) return false;
          const uint32_t bytes = (uint32_t)(min(TR, step_rows - i * TR) * ROWB);
          const size_t off = (hk + s0 + (size_t)i * TR) * ROWB;
          uint64_t *fb = &s_full[gp % kFullBars];
          mbar_expect_tx(fb, 2 * bytes);
          bulk_load(kv + st * 2 * SB, (const uint8_t *)c.K + off, bytes, fb);
          bulk_load(kv + st * 2 * SB + SB, (const uint8_t *)c.V + off, bytes, fb);
          ++gp;
          return true;
        };
        for (int i = s_spec; ok && i < nst; ++i) ok = issue(i, nrows);
        int spec = 0;
        if (ok && step + 1 < a.nsteps) {
          const int n1 = min(a.s.n_valid + step + 1, c.k);
          const int nrows1 = max(0, min(own, n1 - s0));
          const int nst1 = (nrows1 + TR - 1) / TR;
          for (; ok && spec < kStages && spec < nst1; ++spec) ok = issue(spec, nrows1);
          if (!ok) --spec;
        }
        s_spec = spec;
        if (!ok) {
          s_abort = 1;
          atomicOr(c.err, 1);
          for (int j = max(0, gp - kStages); j < gp; ++j) mbar_wait(&s_full[j % kFullBars], (j / kFullBars) & 1);
        }
      }
      g += nst;
    } else if (!aborted) {
      if constexpr (W) {
      // ---- consumers, wide-row layout (bf16 rows of 128): one warp takes a
      // whole 32-row slab (warp w the slabs w, w + NC, ...).  K: each lane
      // computes its own row's dot product with no cross-lane reduction; lane
      // i walks the row's sixteen 16-byte chunks in an order rotated by i
      // (chunk (c + i) mod 16 at step c), so the eight lanes of every
      // shared-memory phase touch eight different bank groups, and holds q
      // rotated the same way, so register indexing stays static.  V: lane i
      // owns output dimensions 4i .. 4i+3 and takes every row's weight by one
      // shuffle.
      uint32_t qr[16][4];  // q chunk (c + lane) mod 16, raw bf16 pairs
#pragma unroll
      for (int cch = 0; cch < 16; ++cch) {
        const uint4 u = *(const uint4 *)(in_q + (((cch + lane) & 15) << 3));
        qr[cch][0] = u.x; qr[cch][1] = u.y; qr[cch][2] = u.z; qr[cch][3] = u.w;
      }
      float m = -INFINITY, l = 0.f, acc[4] = {0.f, 0.f, 0.f, 0.f};
      const int nslab = kResident ? (nrows + TR - 1) / TR : nst;
      bool ok = true;
      for (int i = warp; i < nslab; i += kConsumers) {
        const int gi = g + i;
        const int st = gi % kStages;
        const uint8_t *ks, *vs;
        if (kResident) {
          ks = kv + (size_t)i * TR * ROWB;
          vs = kv + (size_t)chunk * ROWB + (size_t)i * TR * ROWB;
        } else {
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[gi % kFullBars], (gi / kFullBars) & 1)))) break;
          ks = kv + st * 2 * SB;
          vs = ks + SB;
        }
        const int rows = min(TR, nrows - i * TR);
        const bool valid = lane < rows;
        const uint8_t *krow = ks + (valid ? lane : 0) * ROWB;
        float d4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
        for (int cch = 0; cch < 16; ++cch) {
          const uint4 kc = *(const uint4 *)(krow + (((cch + lane) & 15) << 4));
          float dd = d4[cch & 3];
          dd = fma2_bf16(qr[cch][0], kc.x, dd);
          dd = fma2_bf16(qr[cch][1], kc.y, dd);
          dd = fma2_bf16(qr[cch][2], kc.z, dd);
          dd = fma2_bf16(qr[cch][3], kc.w, dd);
          d4[cch & 3] = dd;
        }
        float lgt = ((d4[0] + d4[1]) + (d4[2] + d4[3])) * a.qscale;
        lgt = valid ? lgt : -INFINITY;
        if (valid) lg[i * TR + lane] = lgt;
        const float wmax = warp_max(lgt);
        if (wmax > m) {  // warp-uniform: rescale only when the running max grows
          const float sc_ = ex2(m - wmax);
          l *= sc_;
#pragma unroll
          for (int u = 0; u < 4; ++u) acc[u] *= sc_;
          m = wmax;
        }
        const float pr = valid ? ex2(lgt - m) : 0.f;
        l += pr;  // this lane's row; summed over the warp at the end
        const uint8_t *vcol = vs + lane * 8;
        auto vrow = [&](int r) {
          const float w = __shfl_sync(0xffffffffu, pr, r);
          const uint2 v = *(const uint2 *)(vcol + r * ROWB);
          fma_pair(acc[0], acc[1], w, bf16lo(v.x), bf16hi(v.x));
          fma_pair(acc[2], acc[3], w, bf16lo(v.y), bf16hi(v.y));
        };
        if (rows == TR) {
#pragma unroll
          for (int r = 0; r < TR; ++r) vrow(r);
        } else {
          for (int r = 0; r < rows; ++r) vrow(r);  // warp-uniform bound: no stale row is read
        }
        if (!kResident) {
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[st]);
        }
      }
      g += nst;
      if (!ok && lane == 0) {
        s_abort = 1;
        atomicOr(c.err, 1);
      }
      if (rank == 0 && warp == 0) {  // the new token, from the step inputs (four dimensions per lane)
        float qv[4], kx[4], vx[4];
        auto ld4 = [&](const T *p4, float *x) {  // four bf16 values (8 bytes)
          const uint2 u = *(const uint2 *)p4;
          x[0] = bf16lo(u.x); x[1] = bf16hi(u.x); x[2] = bf16lo(u.y); x[3] = bf16hi(u.y);
        };
        ld4(in_q + 4 * lane, qv);
        ld4(in_k + 4 * lane, kx);
        float dot = 0.f;
#pragma unroll
        for (int u = 0; u < 4; ++u) dot = fmaf(qv[u], kx[u], dot);
        dot = warp_sum(dot) * a.qscale;
        if (lane == 0) s_lgnew = dot;
        const float mn = fmaxf(m, dot);
        const float sc_ = ex2(m - mn);
        l *= sc_;
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] *= sc_;
        m = mn;
        const float pr = ex2(dot - m);
        if (lane == 0) l += pr;
        ld4(in_v + 4 * lane, vx);
#pragma unroll
        for (int u = 0; u < 4; ++u) acc[u] = fmaf(pr, vx[u], acc[u]);
      }
      l = warp_sum(l);
#pragma unroll
      for (int u = 0; u < 4; ++u) s_wacc[warp][4 * lane + u] = acc[u];
      if (lane == 0) {
        s_wm[warp] = m;
        s_wl[warp] = l;
      }
      } else {
      // ---- consumers: logits and per-warp online softmax over the owned rows.
      // A lane group (LPR lanes) takes ITER rows per slab: K dot products
      // from packed q, one transposed reduction, one exp2 per lane for the
      // row it ends up holding, broadcast back for the V rows.
      QLane<S, EPL> qk;
      qk.load(in_q + sub * EPL, a.qscale);
      constexpr int LPI = LPR / ITER;  // lanes holding one reduced row
      float m = -INFINITY, l = 0.f, acc[EPL];
#pragma unroll
      for (int e = 0; e < EPL; ++e) acc[e] = 0.f;
      const int nslab = kResident ? (nrows + TR - 1) / TR : nst;
      const int myit = sub / LPI;  // the row this lane holds after the reduction
      bool ok = true;
      int st = g % kStages, ph = (g / kStages) & 1;  // ring stage and phase of slab g
      for (int i = 0; i < nslab; ++i) {
        const uint8_t *ks, *vs;
        if (kResident) {
          ks = kv + (size_t)i * TR * ROWB;
          vs = kv + (size_t)chunk * ROWB + (size_t)i * TR * ROWB;
        } else {
          if (!(ok = __all_sync(0xffffffffu, mbar_wait(&s_full[st], ph)))) break;
          ks = kv + st * 2 * SB;
          vs = ks + SB;
        }
        const int rows = min(TR, nrows - i * TR);
        // One slab: full slabs (every row of the slab filled, all but a CTA's
        // last) take a path without per-row bounds checks.
        auto slab = [&](auto full_tag) {
          constexpr bool kFull = decltype(full_tag)::value;
          float x[ITER];
#pragma unroll
          for (int it = 0; it < ITER; ++it) {
            const int r = warp * RPW + grp + it * kConsumers * RPW;
            x[it] = qk.dot(ks + (kFull || r < rows ? r : 0) * ROWB + sub * Lane<S>::VB);
          }
          const int rm = warp * RPW + grp + myit * kConsumers * RPW;
          const bool valid = kFull || rm < rows;
          float lgt = xreduce<ITER, LPR>(x, sub) * qk.scale;
          if (kFp8) lgt *= valid ? ksc[i * TR + rm] : 0.f;
          lgt = valid ? lgt : -INFINITY;
          if (valid && sub % LPI == 0) lg[i * TR + rm] = lgt;
          float wmax = lgt;  // over the warp's rows of this slab
#pragma unroll
          for (int o = LPI; o < 32; o <<= 1) wmax = fmaxf(wmax, __shfl_xor_sync(0xffffffffu, wmax, o));
          if (wmax > m) {  // warp-uniform: rescale only when the running max grows
            const float sc_ = ex2(m - wmax);
            l *= sc_;
#pragma unroll
            for (int e = 0; e < EPL; ++e) acc[e] *= sc_;
            m = wmax;
          }
          const float prm = valid ? ex2(lgt - m) : 0.f;
          if (sub % LPI == 0) l += prm;  // each row's weight once, in the lane that holds it
#pragma unroll
          for (int it = 0; it < ITER; ++it) {
            const int r = warp * RPW + grp + it * kConsumers * RPW;
            const float pr = __shfl_sync(0xffffffffu, prm, grp * LPR + it * LPI);
            if (kFull || r < rows) {
              const float pv = kFp8 ? pr * vsc[i * TR + r] : pr;
              float vx[EPL];
              unpack_lane<S>(vs + r * ROWB + sub * Lane<S>::VB, vx);
#pragma unroll
              for (int e = 0; e < EPL; e += 2) fma_pair(acc[e], acc[e + 1], pv, vx[e], vx[e + 1]);
            }
          }
        };
        if (rows == TR)
          slab(std::true_type{});
        else
          slab(std::false_type{});
        if (!kResident) {
          ++g;
          __syncwarp();
          if (lane == 0) mbar_arrive(&s_empty[st]);
          if (++st == kStages) {
            st = 0;
            ph ^= 1;
          }
        }
      }
      if (!ok && lane == 0) {
        s_abort = 1;
        atomicOr(c.err, 1);
      }
      if (rank == 0 && warp == 0) {  // the new token, from the step inputs
        float qv[EPL], kx[EPL];
        load_f32<T, EPL>(in_q + sub * EPL, qv);
        load_f32<T, EPL>(in_k + sub * EPL, kx);
        float dot = 0.f;
#pragma unroll
        for (int e = 0; e < EPL; ++e) dot = fmaf(qv[e], kx[e], dot);
#pragma unroll
        for (int o = LPR / 2; o; o >>= 1) dot += __shfl_xor_sync(0xffffffffu, dot, o);
        dot *= a.qscale;
        if (lane == 0) s_lgnew = dot;
        const float mn = fmaxf(m, dot);
        const float sc_ = ex2(m - mn);
        l *= sc_;
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] *= sc_;
        m = mn;
        if (grp == 0) {
          const float pr = ex2(dot - m);
          if (lane == 0) l += pr;
          float vx[EPL];
          load_f32<T, EPL>(in_v + sub * EPL, vx);
#pragma unroll
          for (int e = 0; e < EPL; ++e) acc[e] = fmaf(pr, vx[e], acc[e]);
        }
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) l += __shfl_xor_sync(0xffffffffu, l, o);  // row weights sit in single lanes
#pragma unroll
      for (int o = LPR; o < 32; o <<= 1) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) acc[e] += __shfl_xor_sync(0xffffffffu, acc[e], o);
      }
      if (grp == 0) {
#pragma unroll
        for (int e = 0; e < EPL; ++e) s_wacc[warp][sub * EPL + e] = acc[e];
      }
      if (lane == 0) {
        s_wm[warp] = m;
        s_wl[warp] = l;
      }
      }
      consumers_sync<NC>();
      // merge the warps into this CTA's partial (published for rank 0)
      float M = s_wm[0];
#pragma unroll
      for (int w = 1; w < kConsumers; ++w) M = fmaxf(M, s_wm[w]);
      float f[kConsumers];
#pragma unroll
      for (int w = 0; w < kConsumers; ++w) f[w] = (s_wm[w] == -INFINITY) ? 0.f : exp2f(s_wm[w] - M);
      for (int col = tid; col < D; col += kConsumerThreads) {
        float t = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) t = fmaf(f[w], s_wacc[w][col], t);
        st_async_b32(mapa(&accx[rank * D + col], 0), __float_as_uint(t), mapa(&s_bacc, 0));  // to rank 0
      }
      if (tid < P) {  // (m, l) to every rank
        float ls = 0.f;
#pragma unroll
        for (int w = 0; w < kConsumers; ++w) ls = fmaf(f[w], s_wl[w], ls);
        const uint4 v = make_uint4(__float_as_uint(M), __float_as_uint(ls), __float_as_uint(s_lgnew), 0u);
        st_async_v4(mapa(&s_mlx[rank], tid), v, mapa(&s_bml, tid));
      }
    }

    // ---- global softmax statistics (identical in every CTA), once every
    // rank's (m, l) has landed here (and, on rank 0, every acc row)
    if (warp == 0) {
      bool got = mbar_wait(&s_bml, step & 1);
      if (rank == 0) got = got && mbar_wait(&s_bacc, step & 1);
      if (!__all_sync(0xffffffffu, got) && lane == 0) s_abort = 1;
      float mr = -INFINITY, lr = 0.f;
      if (lane < P) {
        mr = __uint_as_float(s_mlx[lane].x);
        lr = __uint_as_float(s_mlx[lane].y);
      }
      // lanes 0..P-1 (P <= 8) hold values: three butterfly levels reduce them
      float Mg = mr;
#pragma unroll
      for (int o = kMaxCluster / 2; o; o >>= 1) Mg = fmaxf(Mg, __shfl_xor_sync(0xffffffffu, Mg, o));
      const float fr = (mr == -INFINITY) ? 0.f : exp2f(mr - Mg);
      float Lg = fr * lr;
#pragma unroll
      for (int o = kMaxCluster / 2; o; o >>= 1) Lg += __shfl_xor_sync(0xffffffffu, Lg, o);
      if (lane < P) s_f[lane] = fr;
      if (lane == 0) {
        s_ML[0] = Mg;
        s_ML[1] = Lg;
      }
    }
    __syncthreads();
    const float Mg = s_ML[0], invL = 1.f / s_ML[1];
    if (rank == 0 && warp == kConsumers) {
      // the step's output row, by the producer warp while the consumers add
      // the weights (off the path to the decision); its reads of the acc rows
      // precede the CTA barrier below, so no peer can push next step's rows
      // before they are done
      T *out = (T *)a.s.out + step * step_elems + (size_t)h * D;
      constexpr int CPL = D / 32;
      float o[CPL];
#pragma unroll
      for (int q = 0; q < CPL; ++q) o[q] = 0.f;
      for (int r = 0; r < P; ++r) {
        const float fr = s_f[r];
        if (fr != 0.f) {
#pragma unroll
          for (int q = 0; q < CPL; ++q) o[q] = fmaf(fr, accx[r * D + lane * CPL + q], o[q]);
        }
      }
#pragma unroll
      for (int q = 0; q < CPL; ++q) out[lane * CPL + q] = from_f32<T>(o[q] * invL);
    }

    // ---- exact weights into the owned scores; local argmin
    const long long lim = (long long)p - c.kl;  // eligible iff n_sink <= pos <= p - k_local
    ArgMin best{INFINITY, INT_MAX, -2};
    if (warp < kConsumers) {
      for (int j = tid; j < nrows; j += kConsumerThreads) {
        const float w = exp2f(lg[j] - Mg) * invL;
        float s_new = sc[j], cj = cm[j];
        kahan_add(s_new, cj, w);
        sc[j] = s_new;
        cm[j] = cj;
        const int pj = ps[j];
        if ((long long)pj <= lim && pj >= c.n_sink) {
          const ArgMin cand{rank_key(s_new, p, pj, c.score_mode), pj, s0 + j};
          if (am_less(cand, best)) best = cand;
        }
      }
    }
    // the new token's weight, from rank 0's logit (every CTA: the owner of
    // the slot it takes writes it as that slot's score)
    const float w_new = exp2f(__uint_as_float(s_mlx[0].z) - Mg) * invL;
    if (rank == 0 && tid == 0 && c.kl == 0 && p >= c.n_sink) {
      const ArgMin cand{w_new, p, -1};  // attended by one query: its mean is its weight
      if (am_less(cand, best)) best = cand;
    }
    if (warp < kConsumers) {
      best = warp_argmin(best);
      if (lane == 0) s_am[warp] = best;
    }
    __syncthreads();
    if (tid == 0) {
      ArgMin b = s_am[0];
      for (int w = 1; w < kConsumers; ++w)
        if (am_less(s_am[w], b)) b = s_am[w];
      const uint4 v = make_uint4(__float_as_uint(b.s), (uint32_t)b.p, (uint32_t)b.slot, 0u);
      for (int r = 0; r < P; ++r) st_async_v4(mapa(&s_candx[rank], r), v, mapa(&s_bcand, r));  // to every rank
    }

    // ---- the decision, taken identically by warp 0 of every CTA (lane r
    // holds rank r's candidate), then the owner's update
    if (warp == 0) {
      if (!__all_sync(0xffffffffu, mbar_wait(&s_bcand, step & 1)) && lane == 0) s_abort = 1;
      ArgMin b{INFINITY, INT_MAX, -2};
      if (lane < P) {
        const uint4 cv = s_candx[lane];
        b = ArgMin{__uint_as_float(cv.x), (int)cv.y, (int)cv.z};
      }
      b = warp_argmin(b);
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
      if (lane == 0 && rank == 0 && a.s.evicted) a.s.evicted[(size_t)step * c.nh + h] = ev;
      e = __shfl_sync(0xffffffffu, e, 0);
      const float dec_w = w_new;
      if (e >= s0 && e < s0 + own) {  // this CTA owns the slot that takes the new token
        const int j = e - s0;
        if (tid == 0) {
          ps[j] = p;
          sc[j] = dec_w;
          cm[j] = 0.f;
        }
        constexpr int PER = D / 32;  // fp8: lane L quantises elements L*PER ..
        uint32_t ck = 0u, cv = 0u;
        if (kFp8) {  // warp-uniform branch (e is the same in every lane)
          float xk[PER], xv[PER], sk, sv;
#pragma unroll
          for (int q = 0; q < PER; ++q) {
            xk[q] = to_f32<T>(in_k[lane * PER + q]);
            xv[q] = to_f32<T>(in_v[lane * PER + q]);
          }
          ck = quant_row_e4m3<PER>(xk, sk);
          cv = quant_row_e4m3<PER>(xv, sv);
          store_codes<PER>((uint8_t *)c.K + (hk + e) * ROWB, lane, ck);
          store_codes<PER>((uint8_t *)c.V + (hk + e) * ROWB, lane, cv);
          if (kResident) {
            store_codes<PER>(kv + (size_t)j * ROWB, lane, ck);
            store_codes<PER>(kv + (size_t)chunk * ROWB + (size_t)j * ROWB, lane, cv);
          }
          if (tid == 0) {
            ksc[j] = sk;
            vsc[j] = sv;
          }
        } else if (grp == 0) {  // lanes 0..LPR-1 copy the k_t / v_t row
          const int i = sub;
          const uint4 kq = *(const uint4 *)(in_k + i * EPL), vq = *(const uint4 *)(in_v + i * EPL);
          ((uint4 *)((T *)c.K + (hk + e) * D))[i] = kq;
          ((uint4 *)((T *)c.V + (hk + e) * D))[i] = vq;
          if (kResident) {
            ((uint4 *)(kv + (size_t)j * ROWB))[i] = kq;
            ((uint4 *)(kv + (size_t)chunk * ROWB + (size_t)j * ROWB))[i] = vq;
          }
        }
        fence_proxy_async_smem();
        asm volatile("fence.proxy.async.global;" ::: "memory");  // before our next bulk reads of row e
        if (!kResident && step + 1 < a.nsteps && j / TR < s_spec) {
          // The producer already loaded the slab holding row j for the next
          // step: let that copy land, then overwrite the stale row in it.
          const int gpos = g + j / TR;  // ring position of that slab (g = next step's first)
          const int st = gpos % kStages;
          if (!__all_sync(0xffffffffu, mbar_wait(&s_full[gpos % kFullBars], (gpos / kFullBars) & 1)) && lane == 0)
            s_abort = 1;
          uint8_t *slab = kv + st * 2 * SB;
          if (kFp8) {
            store_codes<PER>(slab + (j % TR) * ROWB, lane, ck);
            store_codes<PER>(slab + SB + (j % TR) * ROWB, lane, cv);
          } else if (grp == 0) {
            ((uint4 *)(slab + (j % TR) * ROWB))[sub] = *(const uint4 *)(in_k + sub * EPL);
            ((uint4 *)(slab + SB + (j % TR) * ROWB))[sub] = *(const uint4 *)(in_v + sub * EPL);
          }
        }
      }
    }
    __syncthreads();
  }
  if (*(volatile int *)&s_abort && tid == 0) atomicOr(c.err, 1);
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

// Per-slot shared-memory words beside K/V: score, tag, logit, score
// compensation (+ two scales for an fp8 cache).
template <typename S> constexpr int slot_words() { return is_fp8<S>() ? 6 : 4; }

template <typename S, int D> constexpr int row_bytes() { return D * (int)sizeof(S); }

template <typename S, int D>
int resident_rows_ok(int chunk) {
  return 2 * chunk * row_bytes<S, D>() <= kResidentMaxBytes;
}

template <typename S, int D, bool R, int St, bool W = false>
int smem_bytes(int chunk, int P) {
  const int base = (R ? 2 * chunk * row_bytes<S, D>() : ring_bytes(St, W)) + slot_words<S>() * chunk * 4;
  return ((base + 15) & ~15) + P * D * 4;  // + every rank's acc row
}

int chunk_of(const CacheView &c) { return (c.k + c.nsplit - 1) / c.nsplit; }

template <typename T, typename S, int D, bool R, int St, int NC, bool W = false>
cudaError_t launch_cluster_t(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st) {
  const int P = c.nsplit;
  CArgs a{c, s, nsteps, chunk_of(c), kLog2e / sqrtf((float)D)};
  const int smem = smem_bytes<S, D, R, St, W>(a.chunk, P);
  if (smem > 200 * 1024) return cudaErrorInvalidValue;
  static bool attr_done[64] = {};
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64 || !attr_done[dev]) {
    cudaError_t e = cudaFuncSetAttribute(decode_cluster_kernel<T, S, D, R, St, NC, W>,
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
  return cudaLaunchKernelEx(&cfg, decode_cluster_kernel<T, S, D, R, St, NC, W>, a);
}

// CTAs of this instance that fit on the device at once (0 on an error).
template <typename T, typename S, int D, bool R, int St, int NC, bool W = false>
long long resident_ctas(const CacheView &c, int chunk) {
  int dev = 0, sms = 0, per_sm = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 0;
  if (cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
  const int smem = smem_bytes<S, D, R, St, W>(chunk, c.nsplit);
  if (smem > 200 * 1024) return 0;
  if (cudaFuncSetAttribute(decode_cluster_kernel<T, S, D, R, St, NC, W>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           200 * 1024) != cudaSuccess)
    return 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, decode_cluster_kernel<T, S, D, R, St, NC, W>,
                                                    threads_for(NC), smem) != cudaSuccess)
    return 0;
  return (long long)per_sm * sms;
}

template <typename T, typename S, int D, bool R, int St, int NC, bool W = false>
bool all_resident(const CacheView &c, int chunk) {
  const long long fit = resident_ctas<T, S, D, R, St, NC, W>(c, chunk);
  return fit > 0 && (long long)c.nh * c.nsplit <= fit;
}

// K/V resident in shared memory when a CTA's rows fit AND every CTA of the
// grid is resident at once (each CTA runs all steps of its head, so a second
// wave would start only when the first finished).
template <typename T, typename S, int D, int NC>
bool resident_nc(const CacheView &c) {
  const int chunk = chunk_of(c);
  return resident_rows_ok<S, D>(chunk) && all_resident<T, S, D, true, 1, NC>(c, chunk);
}

// Streaming: a 3-stage ring, unless two stages are what lets every CTA be
// resident at once (a partial last wave of whole-run CTAs streams at a
// fraction of the bandwidth).
// The wide-row layout for bf16 rows of 128 (the consumer loop's W branch).
template <typename T, typename S, int D> constexpr bool wide_rows() {
  return std::is_same<T, __nv_bfloat16>::value && std::is_same<S, __nv_bfloat16>::value && D == 128;
}

template <typename T, typename S, int D, int NC>
cudaError_t dispatch_nc(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st) {
  const int chunk = chunk_of(c);
  if (resident_nc<T, S, D, NC>(c)) return launch_cluster_t<T, S, D, true, 1, NC>(c, s, nsteps, st);
  if constexpr (wide_rows<T, S, D>()) {
    // Wide rows where the grid spans at least two waves (per-CTA throughput
    // counts more than the step's latency), with two ring stages (five CTAs
    // per SM) for clusters of four or more, whose exchanges take longer and
    // want more CTAs to overlap them, else three.  Measured on GB300, us per
    // step (lane groups / wide, 3 stages / wide, 2 stages): 8K prompt
    // (clusters of 8) 101.6 / 119.6 / 91.3; OPT-30B (clusters of 2) 74.6 /
    // 70.8 / 73.2; OPT-6.7B (one wave) 7.53 / 8.75 / 10.3.
    const long long grid = (long long)c.nh * c.nsplit;
    if (chunk >= 64 && grid >= 2LL * 7 * num_sms_current_device()) {
      if (c.nsplit >= 4) return launch_cluster_t<T, S, D, false, 2, NC, true>(c, s, nsteps, st);
      return launch_cluster_t<T, S, D, false, 3, NC, true>(c, s, nsteps, st);
    }
  }
  if (!all_resident<T, S, D, false, 3, NC>(c, chunk) && all_resident<T, S, D, false, 2, NC>(c, chunk))
    return launch_cluster_t<T, S, D, false, 2, NC>(c, s, nsteps, st);
  return launch_cluster_t<T, S, D, false, 3, NC>(c, s, nsteps, st);
}

// The consumer-warp count for a CTA that owns chunk_of(c) slots.
template <typename T, typename S, int D>
cudaError_t dispatch_t(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st) {
  return chunk_of(c) > kShortChunk ? dispatch_nc<T, S, D, 4>(c, s, nsteps, st)
                                   : dispatch_nc<T, S, D, 2>(c, s, nsteps, st);
}

#define H2O_CLUSTER_DISPATCH(FN, ...)                                              \
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

}  // namespace

// Cluster size: the smallest power of two that leaves each CTA at most
// kShortChunk slots (the two-consumer-warp kernel), doubled (up to 8) while
// the grid fills less than 90 % of one wave of 7 CTAs per SM.  Measured on
// GB300 (us per decode step, cluster sizes 1 / 2 / 4 / 8): OPT-6.7B shape
// (256 heads, k = 512) - / 11.6 / 8.2 / 13.8; OPT-30B shape (3584 heads,
// k = 408) 103.4 / 81.9 / 99.7 / -; 8K-prompt shape (1024 heads, k = 1690)
// 133.8 / 123.9 / 121.7 / 114.6; long stream (32 heads, k = 256) 10.4 / 4.89
// / 3.24 / 2.62 — the rule picks the fastest in each case.  Where a wave of
// CTAs holds less than L2 (the OPT-30B shape at size 2: 532 heads, 111 MB),
// its steps read the cache from L2.
int decode_cluster_size(int nh, int k, int sms) {
  int P = 1;
  while (P < kMaxCluster && (k + P - 1) / P > kShortChunk) P *= 2;
  const long long wave = 7LL * (sms > 0 ? sms : 1);
  while (P < kMaxCluster && (long long)nh * P * 10 < wave * 9) P *= 2;
  return P;
}

bool decode_cluster_supported(const CacheView &c) {
  if (c.nsplit < 1 || c.nsplit > kMaxCluster) return false;
  const int chunk = (c.k + c.nsplit - 1) / c.nsplit;
  const int row = c.d * (c.kv_fp8 ? 1 : c.dtype == 1 ? 2 : 4);
  const int kv = (2 * chunk * row <= kResidentMaxBytes) ? 2 * chunk * row : ring_bytes(3);
  return kv + (c.kv_fp8 ? 6 : 4) * chunk * 4 + 16 + c.nsplit * c.d * 4 <= 200 * 1024;
}

cudaError_t launch_decode_cluster(const CacheView &c, const DecodeStep &s, int nsteps, cudaStream_t st) {
  if (!decode_cluster_supported(c) || nsteps < 1) return cudaErrorInvalidValue;
  H2O_CLUSTER_DISPATCH(dispatch_t, c, s, nsteps, st);
  return cudaErrorInvalidValue;
}

}  // namespace h2o
