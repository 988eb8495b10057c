// prefill_tc.cu — tensor-core prefill passes for bf16 caches (sm_103a:
// tcgen05.mma with TMEM accumulators, TMA tile loads, mbarrier pipeline).
//
// H2O summary page, "Algorithm / figure walkthrough" step 1: the prompt's
// accumulated attention score of key j is its causal column sum
//   colsum_j = sum_{i >= j} exp(q_i.k_j / sqrt(d) - LSE_i).
//
// Column-sum pass (the score pass, colsum_pair_tc).  A CTA owns two adjacent
// 128-key tiles, resident in shared memory as the MMA's A operands (M = 128
// TMEM lanes, one key per thread); query tiles of 128 stream through a TMA
// ring as the shared B operand (N = 128) and each S^T = K Q^T lands in a
// double-buffered TMEM accumulator of its key tile, so one key tile's MMA
// overlaps the other's epilogue.  Each epilogue thread turns its key row into
// exp2(s * log2(e)/sqrt(d) - LSE_i * log2(e)) and adds it into its own sum:
// deterministic and atomic-free.  Only the first query tile of a key tile
// touches the diagonal and needs the causal mask; query rows past L are
// zero-filled by TMA and masked by LSE = +inf.
//
// LSE pass (when the caller does not want O).  The same pipeline with the
// roles swapped: a CTA owns 128 queries (A operand, TMEM lanes) and streams
// the key tiles 0..diagonal; each thread keeps an online (max, sum) of its
// row in base 2.
//
// Warp roles of these two: warp 8 issues TMA and MMA; warps 0-7 run the
// epilogue (warp w reads TMEM lanes 32(w%4)..+31, columns 64(w/4)..+63).
//
// Attention pass (O and LSE, pass 1 of the prefill): two query tiles per CTA
// ping-ponging on the tensor core, P kept in tensor memory (attn_pair_tc,
// described at the kernel).
//
// Every mbarrier wait is bounded; on a timeout the CTA flags the cache's error
// word, drains what it issued and frees its TMEM before returning.
#include <cudaTypedefs.h>

#include "common.cuh"
#include "sm100.cuh"

namespace h2o {
namespace {

using namespace sm100;

constexpr int kRows = 128;            // tile rows (TMEM lanes / MMA M and N)
constexpr int kBox = kRows * 128;     // bytes of one 64-column bf16 box
constexpr int kStages = 2;            // streamed-tile ring depth
constexpr int kEpiWarps = 8;   // epilogue warps: 2 per TMEM lane quarter, 64 columns each
constexpr int kThreads = 32 * (kEpiWarps + 1);  // + one producer warp (TMA, MMA, column vector)

template <int D> struct TileGeo {
  static constexpr int kBoxes = D / 64;
  static constexpr int kTileBytes = kBox * kBoxes;
  static constexpr int kKSteps = D / 16;  // UMMA K = 16 for bf16
  // resident tile + ring, each 1024-aligned, then the small state
  static constexpr int kSmem = kTileBytes * (1 + kStages) + 2 * kRows * 4 + 3 * kRows * 4 + 256 + 1024;
};

struct __align__(8) SmallState {
  uint64_t res_bar;           // resident tile landed (one phase per segment)
  uint64_t a_free;            // the MMAs of the first segment are done with the resident tile
  uint64_t ld_bar[kStages];   // streamed tile landed
  uint64_t ld_free[kStages];  // the MMA that read the stage is done
  uint64_t mma_full[2];       // accumulator ready
  uint64_t acc_empty[2];      // epilogue warps done with the accumulator
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

// This warp's 32 TMEM lanes x 64 columns: two loads in flight, one wait.
__device__ __forceinline__ void tmem_ld64(uint32_t taddr, uint32_t (&r)[64]) {
  tmem_ld32(taddr, *reinterpret_cast<uint32_t(*)[32]>(&r[0]));
  tmem_ld32(taddr + 32, *reinterpret_cast<uint32_t(*)[32]>(&r[32]));
  tmem_ld_wait();
  tmem_regs_ready(*reinterpret_cast<uint32_t(*)[32]>(&r[0]));
  tmem_regs_ready(*reinterpret_cast<uint32_t(*)[32]>(&r[32]));
}

// Bounded wait whose outcome is the same for the whole warp (so the warp's
// collective TMEM loads after it stay uniform even on a timeout).
__device__ __forceinline__ bool wait_warp(uint64_t *bar, uint32_t parity) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity));
}

__device__ __forceinline__ uint8_t *align1024(uint8_t *p) {
  return (uint8_t *)(((uintptr_t)p + 1023) & ~(uintptr_t)1023);
}

// Issue the K-loop of one 128x128 tile product: acc = A * B^T over d.
template <int D>
__device__ __forceinline__ void mma_tile(uint32_t acc, uint32_t a_base, uint32_t b_base) {
  constexpr uint32_t idesc = idesc_bf16_f32(128, 128, false);
#pragma unroll
  for (int kk = 0; kk < TileGeo<D>::kKSteps; ++kk) {
    const uint32_t off = (uint32_t)((kk >> 2) * kBox + (kk & 3) * 32);
    umma_bf16(acc, sdesc_sw128(a_base + off, 16, 1024), sdesc_sw128(b_base + off, 16, 1024), idesc, kk > 0);
  }
}

template <int D>
__device__ __forceinline__ void load_tile(uint8_t *dst, const CUtensorMap *map, uint64_t *bar, int row, int h) {
  mbar_expect_tx(bar, TileGeo<D>::kTileBytes);
#pragma unroll
  for (int b = 0; b < TileGeo<D>::kBoxes; ++b) tma_load_3d(dst + b * kBox, map, bar, b * 64, row, h);
}

// One run of the pipeline: resident tile from row r0 of the A map, streamed
// tiles j = 0..n-1 from rows s0 + 128 j of the B map.
struct Seg {
  int r0, s0, n;
};

// Shared skeleton, warp-specialised, over one or two segments that share the
// ring and the accumulators (the streamed-tile count j runs on across the
// segment boundary).  Warp 8 (the producer) issues the TMA loads and the MMAs
// into two TMEM accumulators; warps 0-7 wait for an accumulator, call
// `epi(segment, j_in_segment, taddr)` with the TMEM address of their 32 lanes
// and 64-column half, and release it.  At the segment boundary the producer
// waits for the first segment's last MMA (a_free) and reloads the resident
// tile.  No CTA-wide barrier inside the loop.
template <int D, class Epi>
__device__ __forceinline__ bool tile_pipeline(uint8_t *smem, SmallState &st, const CUtensorMap *mapA,
                                              const CUtensorMap *mapB, Seg s0_, Seg s1_, int h, Epi &&epi) {
  using G = TileGeo<D>;
  const int n0 = s0_.n, n = s0_.n + s1_.n;
  auto brow = [&](int j) { return j < n0 ? s0_.s0 + kRows * j : s1_.s0 + kRows * (j - n0); };
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  uint8_t *sA = smem;
  uint8_t *sB = smem + G::kTileBytes;
  if (tid == 0) {
    mbar_init(&st.res_bar, 1);
    mbar_init(&st.a_free, 1);
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&st.ld_bar[s], 1);
      mbar_init(&st.ld_free[s], 1);
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&st.mma_full[b], 1);
      mbar_init(&st.acc_empty[b], kEpiWarps);
    }
    mbar_init(&st.drain, 1);
    st.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&st.tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = st.tmem_base;

  if (warp == kEpiWarps) {
    // ------------------------------------------------------------ producer
    int loads = 0, mmas = 0;
    bool ok = true, a_reloading = false;
    if (lane == 0) {
      load_tile<D>(sA, mapA, &st.res_bar, s0_.r0, h);
      for (; loads < n && loads < kStages; ++loads)
        load_tile<D>(sB + loads * G::kTileBytes, mapB, &st.ld_bar[loads], brow(loads), h);
      ok = mbar_wait(&st.res_bar, 0);
    }
    ok = __shfl_sync(0xffffffffu, ok, 0);
    for (int j = 0; ok && j < n; ++j) {
      // the whole warp observes the accumulator free
      if (j >= 2 && !(ok = wait_warp(&st.acc_empty[j & 1], ((j - 2) >> 1) & 1))) break;
      if (lane == 0) {
        if (j == n0 && j > 0) {  // segment boundary: the resident tile of the second segment
          ok = mbar_wait(&st.a_free, 0);
          if (ok) {
            load_tile<D>(sA, mapA, &st.res_bar, s1_.r0, h);
            a_reloading = true;
            ok = mbar_wait(&st.res_bar, 1);
            a_reloading = !ok;
          }
        }
        if (ok) ok = mbar_wait(&st.ld_bar[j % kStages], (j / kStages) & 1);
        if (ok) {
          tc_fence_after();
          mma_tile<D>(tbase + (uint32_t)(j & 1) * 128, smem_u32(sA), smem_u32(sB + (j % kStages) * G::kTileBytes));
          umma_commit(&st.mma_full[j & 1]);
          umma_commit(&st.ld_free[j % kStages]);
          if (j == n0 - 1 && n > n0) umma_commit(&st.a_free);
          mmas = j + 1;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
      if (!ok) break;
      // refill the stage of tile j-1 (its MMA is done or nearly) with tile j-1+kStages
      if (lane == 0 && j >= 1 && loads < n && loads == j - 1 + kStages) {
        const int sj = (j - 1) % kStages;
        ok = mbar_wait(&st.ld_free[sj], ((j - 1) / kStages) & 1);
        if (ok) {
          load_tile<D>(sB + sj * G::kTileBytes, mapB, &st.ld_bar[sj], brow(loads), h);
          ++loads;
        }
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
    if (!ok && lane == 0) {
      st.abort = 1;
      // Drain: tensor-core work and TMA copies this CTA started must land
      // before its shared memory and TMEM are released.
      umma_commit(&st.drain);
      mbar_wait(&st.drain, 0);
      for (int j = mmas; j < loads; ++j) mbar_wait(&st.ld_bar[j % kStages], (j / kStages) & 1);
      if (a_reloading) mbar_wait(&st.res_bar, 1);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const uint32_t lane_off = ((uint32_t)((warp & 3) * 32) << 16) + (uint32_t)(warp >> 2) * 64;
    for (int j = 0; j < n; ++j) {
      if (!wait_warp(&st.mma_full[j & 1], (j >> 1) & 1)) {
        if (lane == 0) st.abort = 1;
        break;
      }
      tc_fence_after();
      epi(j >= n0 ? 1 : 0, j >= n0 ? j - n0 : j, tbase + lane_off + (uint32_t)(j & 1) * 128);
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&st.acc_empty[j & 1]);
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const bool ok = !*(volatile int *)&st.abort;
  if (warp == 0) tmem_dealloc(tbase, 256);
  return ok;
}

// ---------------------------------------------------------- row log-sum-exp
template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    lse_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
           float *__restrict__ lse, int L, int nqt, float qscale, int *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  using G = TileGeo<D>;
  float *xch = (float *)(smem + G::kTileBytes * (1 + kStages));  // [2][128] hand-over of the second halves
  SmallState &st = *(SmallState *)(xch + 2 * kRows);
  if (*(volatile int *)err) return;
  // Head-major (a head's CTAs share its K tiles in L2), heaviest query tile first.
  const int h = blockIdx.x / nqt, qt = nqt - 1 - blockIdx.x % nqt;
  const int q0 = qt * kRows;
  const int nk = qt + 1;  // key tiles 0 .. diagonal
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = (warp & 3) * 32 + lane;  // query within the tile (TMEM lane)
  const int c_off = (warp >> 2) * 64;      // this warp's key columns
  float m = -INFINITY, l = 0.f;  // base-2 running max and sum over this thread's columns
  auto epi = [&](int, int j, uint32_t taddr) {
    const bool diag = (j == nk - 1);
    uint32_t r[64];
    tmem_ld64(taddr, r);
    float cm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // partial maxima
#pragma unroll
    for (int i = 0; i < 64; ++i) {
      float x = __uint_as_float(r[i]) * qscale;
      if (diag && c_off + i > row) x = -INFINITY;  // key after the query
      r[i] = __float_as_uint(x);
      cm4[i & 3] = fmaxf(cm4[i & 3], x);
    }
    const float cm = fmaxf(fmaxf(cm4[0], cm4[1]), fmaxf(cm4[2], cm4[3]));
    if (cm == -INFINITY) return;  // every column masked (second half of the diagonal)
    const float mn = fmaxf(m, cm);
    float s4[4] = {0.f, 0.f, 0.f, 0.f};
#pragma unroll
    for (int i = 0; i < 64; ++i) s4[i & 3] += ex2(__uint_as_float(r[i]) - mn);
    const float sum = (s4[0] + s4[1]) + (s4[2] + s4[3]);
    l = l * ex2(m - mn) + sum;
    m = mn;
  };
  const bool ok = tile_pipeline<D>(smem, st, &tmQ, &tmK, Seg{q0, 0, nk}, Seg{0, 0, 0}, h, epi);
  if (ok && warp >= 4 && warp < kEpiWarps) {
    xch[row] = m;
    xch[kRows + row] = l;
  }
  __syncthreads();
  if (ok) {
    if (warp < 4 && q0 + row < L) {
      const float m2 = xch[row], l2 = xch[kRows + row];
      const float mm = fmaxf(m, m2);
      const float ll = (m == -INFINITY ? 0.f : l * ex2(m - mm)) + (m2 == -INFINITY ? 0.f : l2 * ex2(m2 - mm));
      lse[(size_t)h * L + q0 + row] = (mm + __log2f(ll)) * kLn2;
    }
  } else if (tid == 0) {
    atomicOr(err, 8);
  }
}

// ------------------------------------------ attention pass, two query tiles
// Causal attention over the prompt, O and the row log-sum-exp, with two
// adjacent 128-query tiles per CTA (A = tile 2p, B = tile 2p+1) sharing every
// K/V tile, so the tensor core works on one tile while the other tile's
// softmax runs.  Warp 9 loads (TMA: both Q tiles, then a two-stage K ring and
// a two-stage V ring); warp 8 issues the MMAs; warps 0-3 are tile A's softmax
// and warps 4-7 tile B's, one thread per query row (TMEM lane), all 128 key
// columns of the row in registers, so a row's maximum needs no exchange.
// TMEM (512 columns): S_A at 0, O_A at 128, S_B at 256, O_B at 384.  The
// softmax turns S into bf16 P = exp2(s*c - m) and stores it back into the
// first 64 columns of the same S region; the PV MMA reads P as its A operand
// straight from tensor memory (V is the MN-major B operand in shared memory).
// MMA order per key tile j: PV_A(j), S_A(j+1), PV_B(j), S_B(j+1) — the
// tensor core executes one CTA's MMAs in issue order, so S_A(j+1) overwrites
// P_A(j) only after PV_A(j) has read it.  O is rescaled in TMEM (lazily, when
// a row's max grows by more than 8 in base 2) by the row's own thread after
// the previous PV has landed.  Barriers: q_full, k_full/v_full (TMA landed),
// k_empty/v_empty (the MMAs that read a stage are done), s_full[t] (S ready),
// p_full[t] (P written: one arrive per softmax warp), pv_done[t].
template <int D> struct PairGeo {
  static constexpr int kTile = TileGeo<D>::kTileBytes;  // 128 rows x D bf16
  static constexpr int kSmem = kTile * 6 + 256 + 1024;   // V[2], K[2], Q_A, Q_B, barriers, alignment
};

struct __align__(8) PairState {
  uint64_t q_full, k_full[2], v_full[2], k_empty[2], v_empty[2];
  uint64_t s_full[2], p_full[2], pv_done[2];  // per query tile
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

constexpr int kPairMmaWarp = 8, kPairLoadWarp = 9;
constexpr int kPairThreads = 32 * 10;

// This warp's 32 TMEM lanes x 128 columns: four loads in flight, one wait.
__device__ __forceinline__ void tmem_ld128(uint32_t taddr, uint32_t (&r)[128]) {
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_ld32(taddr + 32 * c, *reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
  tmem_ld_wait();
#pragma unroll
  for (int c = 0; c < 4; ++c) tmem_regs_ready(*reinterpret_cast<uint32_t(*)[32]>(&r[32 * c]));
}

// D[tmem] (+)= A[tmem] * B[smem], issued by one thread (A: M lanes x K, two
// bf16 per 32-bit column).
__device__ __forceinline__ void umma_bf16_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n\t}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}

template <int D>
__global__ void __launch_bounds__(kPairThreads, 1)
    attn_pair_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                 const __grid_constant__ CUtensorMap tmV, float *__restrict__ lse, __nv_bfloat16 *__restrict__ O,
                 int L, int nqt, int npair, float qscale, int *err) {
  using G = PairGeo<D>;
  constexpr int kT = G::kTile;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *sV = smem;           // 2 stages
  uint8_t *sK = smem + 2 * kT;  // 2 stages
  uint8_t *sQ = smem + 4 * kT;  // tile A, then tile B
  PairState &st = *(PairState *)(smem + 6 * kT);
  if (*(volatile int *)err) return;
  // Head-major (a head's CTAs share its K/V tiles in L2), heaviest pair first.
  const int h = blockIdx.x / npair, pr = npair - 1 - blockIdx.x % npair;
  const int qtA = 2 * pr, qtB = 2 * pr + 1;
  const int nA = qtA + 1;                    // key tiles 0 .. diagonal
  const int nB = qtB < nqt ? qtB + 1 : 0;    // 0: no tile B (odd tile count)
  const int nK = nB ? nB : nA;               // key tiles loaded
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  if (tid == 0) {
    mbar_init(&st.q_full, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&st.k_full[b], 1);
      mbar_init(&st.v_full[b], 1);
      mbar_init(&st.k_empty[b], 1);
      mbar_init(&st.v_empty[b], 1);
      mbar_init(&st.s_full[b], 1);
      mbar_init(&st.p_full[b], 4);
      mbar_init(&st.pv_done[b], 1);
    }
    mbar_init(&st.drain, 1);
    st.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&st.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = st.tmem_base;
  auto tS = [&](int t) { return tbase + (uint32_t)(t * 256); };
  auto tO = [&](int t) { return tbase + (uint32_t)(t * 256 + 128); };

  if (warp == kPairLoadWarp) {
    // ------------------------------------------------------------- loads
    if (lane == 0) {
      bool ok = true;
      int kl = 0, vl = 0;
      mbar_expect_tx(&st.q_full, (nB ? 2 : 1) * G::kTile);
#pragma unroll
      for (int b = 0; b < TileGeo<D>::kBoxes; ++b) {
        tma_load_3d(sQ + b * kBox, &tmQ, &st.q_full, b * 64, qtA * kRows, h);
        if (nB) tma_load_3d(sQ + kT + b * kBox, &tmQ, &st.q_full, b * 64, qtB * kRows, h);
      }
      for (int j = 0; j < nK; ++j) {
        const int s = j & 1;
        if (j >= 2 && !(ok = mbar_wait_backoff(&st.k_empty[s], ((j - 2) >> 1) & 1))) break;
        load_tile<D>(sK + s * kT, &tmK, &st.k_full[s], kRows * j, h);
        kl = j + 1;
        if (j >= 2 && !(ok = mbar_wait_backoff(&st.v_empty[s], ((j - 2) >> 1) & 1))) break;
        load_tile<D>(sV + s * kT, &tmV, &st.v_full[s], kRows * j, h);
        vl = j + 1;
      }
      if (!ok) {
        st.abort = 1;
        // the copies still in flight land before shared memory is released
        mbar_wait(&st.q_full, 0);
        for (int j = kl > 2 ? kl - 2 : 0; j < kl; ++j) mbar_wait(&st.k_full[j & 1], (j >> 1) & 1);
        for (int j = vl > 2 ? vl - 2 : 0; j < vl; ++j) mbar_wait(&st.v_full[j & 1], (j >> 1) & 1);
      }
    }
  } else if (warp == kPairMmaWarp) {
    // -------------------------------------------------------------- MMAs
    if (lane == 0) {
      constexpr uint32_t idO = idesc_bf16_f32(128, D, true);
      auto issue_S = [&](int t, int j) {
        mma_tile<D>(tS(t), smem_u32(sQ + t * kT), smem_u32(sK + (j & 1) * kT));
        umma_commit(&st.s_full[t]);
      };
      auto issue_PV = [&](int t, int j) {
        const uint32_t va = smem_u32(sV + (j & 1) * kT);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk)  // 128 keys, 16 per MMA; P holds two keys per column
          umma_bf16_ts(tO(t), tS(t) + (uint32_t)(kk * 8), sdesc_sw128(va + (uint32_t)(kk * 2048), kBox, 1024), idO,
                       (j > 0 || kk > 0) ? 1u : 0u);
        umma_commit(&st.pv_done[t]);
      };
      bool ok = mbar_wait(&st.q_full, 0) && mbar_wait(&st.k_full[0], 0);
      if (ok) {
        tc_fence_after();
        issue_S(0, 0);
        if (nB) issue_S(1, 0);
        umma_commit(&st.k_empty[0]);
      }
      for (int j = 0; ok && j < nK; ++j) {
        const int s = j & 1;
        bool v_ready = false;
        if (j < nA) {
          if (!(ok = mbar_wait(&st.p_full[0], j & 1) && mbar_wait(&st.v_full[s], (j >> 1) & 1))) break;
          v_ready = true;
          tc_fence_after();
          issue_PV(0, j);
        }
        const bool next = j + 1 < nK;
        if (next) {
          if (!(ok = mbar_wait(&st.k_full[(j + 1) & 1], ((j + 1) >> 1) & 1))) break;
          tc_fence_after();
          if (j + 1 < nA) issue_S(0, j + 1);
        }
        if (j < nB) {
          if (!(ok = mbar_wait(&st.p_full[1], j & 1) && (v_ready || mbar_wait(&st.v_full[s], (j >> 1) & 1)))) break;
          tc_fence_after();
          issue_PV(1, j);
        }
        umma_commit(&st.v_empty[s]);
        if (next) {
          if (j + 1 < nB) issue_S(1, j + 1);
          umma_commit(&st.k_empty[(j + 1) & 1]);
        }
      }
      if (!ok) {
        st.abort = 1;
        // every MMA this CTA issued completes before TMEM and shared memory go
        umma_commit(&st.drain);
        mbar_wait(&st.drain, 0);
      }
    }
  } else {
    // ----------------------------------------------------------- softmax
    const int t = warp >> 2;          // query tile
    const int quarter = warp & 3;     // TMEM lanes 32*quarter ..
    const int row = quarter * 32 + lane;
    const int n = t ? nB : nA;
    const int q = (t ? qtB : qtA) * kRows + row;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float m_run = -INFINITY, l_run = 0.f;  // base-2 running max (scaled) and sum of this row
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (!(ok = wait_warp(&st.s_full[t], j & 1))) break;
      tc_fence_after();
      uint32_t r[128];
      tmem_ld128(tS(t) + lane_off, r);
      if (j == n - 1) {  // diagonal tile: key column c is visible iff c <= row
#pragma unroll
        for (int i = 0; i < 128; ++i)
          if (i > row) r[i] = __float_as_uint(-INFINITY);
      }
      float mx4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
      for (int i = 0; i < 128; ++i) mx4[i & 3] = fmaxf(mx4[i & 3], __uint_as_float(r[i]));
      const float m_tile = fmaxf(fmaxf(mx4[0], mx4[1]), fmaxf(mx4[2], mx4[3])) * qscale;
      float m_new = m_run;
      bool resc = false;
      if (m_run == -INFINITY) {
        m_new = m_tile;  // the row's first logits: nothing accumulated yet
      } else if (m_tile > m_run + 8.f) {
        m_new = m_tile;
        resc = true;
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O must hold every earlier P V before it is rescaled (j >= 1 here)
        if (!(ok = wait_warp(&st.pv_done[t], (j - 1) & 1))) break;
        tc_fence_after();
        const float f = resc ? ex2(m_run - m_new) : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < D; cc += 32) {
          uint32_t o[32];
          tmem_ld32(tO(t) + lane_off + (uint32_t)cc, o);
          tmem_ld_wait();
          tmem_regs_ready(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(tO(t) + lane_off + (uint32_t)cc, o);
        }
        tmem_st_wait();
        l_run *= f;
      }
      m_run = m_new;
      const float nm = -m_run;
      uint32_t pk[64];
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};  // partial row sums
#pragma unroll
      for (int i = 0; i < 64; ++i) {  // masked logits are -inf: exp2 gives 0
        const float a = ex2(fmaf(__uint_as_float(r[2 * i]), qscale, nm));
        const float b = ex2(fmaf(__uint_as_float(r[2 * i + 1]), qscale, nm));
        ls4[i & 3] += a + b;
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        pk[i] = *reinterpret_cast<uint32_t *>(&v);
      }
      l_run += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
      // P over the first 64 columns of the S region (two keys per column)
      tmem_st32(tS(t) + lane_off, *reinterpret_cast<uint32_t(*)[32]>(&pk[0]));
      tmem_st32(tS(t) + lane_off + 32, *reinterpret_cast<uint32_t(*)[32]>(&pk[32]));
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(&st.p_full[t]);
    }
    if (ok && n > 0) ok = wait_warp(&st.pv_done[t], (n - 1) & 1);
    if (ok && n > 0) {
      tc_fence_after();
      const float inv = 1.f / l_run;
      __nv_bfloat16 *orow = O + ((size_t)h * L + (q < L ? q : 0)) * D;
#pragma unroll 1
      for (int c0 = 0; c0 < D; c0 += 32) {  // collective loads: every lane, every chunk
        uint32_t o[32];
        tmem_ld32(tO(t) + lane_off + (uint32_t)c0, o);
        tmem_ld_wait();
        tmem_regs_ready(o);
        if (q < L) {
          uint32_t pk[16];
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            __nv_bfloat162 v =
                __floats2bfloat162_rn(__uint_as_float(o[2 * i]) * inv, __uint_as_float(o[2 * i + 1]) * inv);
            pk[i] = *reinterpret_cast<uint32_t *>(&v);
          }
          uint4 *dst = reinterpret_cast<uint4 *>(orow + c0);
#pragma unroll
          for (int i = 0; i < 4; ++i) dst[i] = make_uint4(pk[4 * i], pk[4 * i + 1], pk[4 * i + 2], pk[4 * i + 3]);
        }
      }
      if (q < L) lse[(size_t)h * L + q] = (m_run + __log2f(l_run)) * kLn2;
    } else if (!ok) {
      st.abort = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (st.abort && tid == 0) atomicOr(err, 16);
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// --------------------------------------------- column sums, two key tiles
// The score pass with two adjacent 128-key tiles per CTA (a = tile 2p,
// b = tile 2p+1), both resident in shared memory as MMA A operands, sharing
// every streamed query tile (B operand, a four-stage TMA ring).  For query
// tile j the MMA warp issues S^T_a(j) and S^T_b(j) into per-key-tile double
// TMEM accumulators (512 columns: a0, a1, b0, b1), so the tensor core works
// on one key tile while the other key tile's epilogue runs.  Warps 0-7 are
// key tile a's epilogue and warps 8-15 key tile b's: two threads per key row
// (TMEM lane), 64 query columns each, each adding
// exp2(s * log2(e)/sqrt(d) - LSE_q * log2(e)) over its columns into its own
// running sum; the two halves of a row are added once at the end (fixed
// order: deterministic, no atomics).  Warp 16 issues the MMAs, warp 17
// loads.  The load warp stages
// -LSE * log2(e) of each query tile beside its Q tile (-inf past L, so the
// zero-filled rows add nothing).  Key tile a reads query tiles a .. nqt-1,
// key tile b query tiles b .. nqt-1; the first tile of each is its diagonal
// (query column c visible iff c >= key row).
constexpr int kCsStages = 4;
constexpr int kCsEpiWarps = 16;  // 8 per key tile: 2 per TMEM lane quarter, 64 columns each
constexpr int kCsMmaWarp = 16, kCsLoadWarp = 17;
constexpr int kCsThreads = 32 * 18;

template <int D> struct CsGeo {
  static constexpr int kTile = TileGeo<D>::kTileBytes;
  static constexpr int kSmem = kTile * (2 + kCsStages) + kCsStages * kRows * 4 + 2 * kRows * 4 + 256 + 1024;
};

struct __align__(8) CsState {
  uint64_t k_full, q_full[kCsStages], q_empty[kCsStages];
  uint64_t acc_full[2][2], acc_empty[2][2];  // [key tile][buffer]
  uint64_t drain;
  uint32_t tmem_base;
  int abort;
};

template <int D>
__global__ void __launch_bounds__(kCsThreads, 1)
    colsum_pair_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                   const float *__restrict__ lse, float *__restrict__ colsum, int L, int nqt, int npair,
                   float qscale, int *err) {
  using G = CsGeo<D>;
  constexpr int kT = G::kTile;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *sK = smem;                                     // key tiles a, b
  uint8_t *sQ = smem + 2 * kT;                            // query ring
  float *sNl = (float *)(smem + (2 + kCsStages) * kT);    // [stage][128] -LSE*log2(e)
  float *sXch = sNl + kCsStages * kRows;                   // [2][128] upper-half sums of the key rows
  CsState &st = *(CsState *)(sXch + 2 * kRows);
  if (*(volatile int *)err) return;
  // Head-major (a head's CTAs share its Q tiles in L2), heaviest pair first.
  const int h = blockIdx.x / npair, pr = npair - 1 - blockIdx.x % npair;
  const int kta = 2 * pr, ktb = 2 * pr + 1;
  const bool has_b = ktb < nqt;
  const int n = nqt - kta;  // query tiles streamed: kta .. nqt-1 (key tile b skips the first)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  float cs_acc = 0.f;  // this thread's key-row sum (epilogue warps)

  if (tid == 0) {
    mbar_init(&st.k_full, 1);
    for (int s = 0; s < kCsStages; ++s) {
      mbar_init(&st.q_full[s], 2);       // TMA bytes + the load warp's -LSE vector
      mbar_init(&st.q_empty[s], 1 + kCsEpiWarps);  // the MMAs' commit + every epilogue warp
    }
    for (int t = 0; t < 2; ++t)
      for (int b = 0; b < 2; ++b) {
        mbar_init(&st.acc_full[t][b], 1);
        mbar_init(&st.acc_empty[t][b], kCsEpiWarps / 2);
      }
    mbar_init(&st.drain, 1);
    st.abort = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&st.tmem_base, 512);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tbase = st.tmem_base;
  auto tAcc = [&](int t, int b) { return tbase + (uint32_t)((t * 2 + b) * 128); };

  if (warp == kCsLoadWarp) {
    // ------------------------------------------------------------- loads
    bool ok = true;
    int issued = 0;
    if (lane == 0) {
      mbar_expect_tx(&st.k_full, (has_b ? 2 : 1) * kT);
#pragma unroll
      for (int b = 0; b < TileGeo<D>::kBoxes; ++b) {
        tma_load_3d(sK + b * kBox, &tmK, &st.k_full, b * 64, kta * kRows, h);
        if (has_b) tma_load_3d(sK + kT + b * kBox, &tmK, &st.k_full, b * 64, ktb * kRows, h);
      }
    }
    const float *lse_h = lse + (size_t)h * L;
    for (int i = 0; i < n; ++i) {
      const int s = i % kCsStages, qt = kta + i;
      if (i >= kCsStages && !(ok = __all_sync(0xffffffffu, mbar_wait_backoff(&st.q_empty[s],
                                                                             ((i / kCsStages) - 1) & 1))))
        break;
      if (lane == 0) {
        mbar_expect_tx(&st.q_full[s], kT);
#pragma unroll
        for (int b = 0; b < TileGeo<D>::kBoxes; ++b)
          tma_load_3d(sQ + s * kT + b * kBox, &tmQ, &st.q_full[s], b * 64, qt * kRows, h);
      }
      issued = i + 1;
#pragma unroll
      for (int u = 0; u < kRows / 32; ++u) {
        const int q = qt * kRows + u * 32 + lane;
        sNl[s * kRows + u * 32 + lane] = q < L ? -__ldg(lse_h + q) * kLog2e : -INFINITY;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&st.q_full[s]);
    }
    if (!ok && lane == 0) {
      st.abort = 1;
      mbar_wait(&st.k_full, 0);
      for (int i = issued > kCsStages ? issued - kCsStages : 0; i < issued; ++i)
        mbar_wait(&st.q_full[i % kCsStages], (i / kCsStages) & 1);
    }
  } else if (warp == kCsMmaWarp) {
    // -------------------------------------------------------------- MMAs
    if (lane == 0) {
      bool ok = mbar_wait(&st.k_full, 0);
      for (int i = 0; ok && i < n; ++i) {
        const int s = i % kCsStages;
        if (!(ok = mbar_wait(&st.q_full[s], (i / kCsStages) & 1))) break;
        // key tile a: its i-th query tile
        if (i >= 2 && !(ok = mbar_wait(&st.acc_empty[0][i & 1], ((i - 2) >> 1) & 1))) break;
        tc_fence_after();
        mma_tile<D>(tAcc(0, i & 1), smem_u32(sK), smem_u32(sQ + s * kT));
        umma_commit(&st.acc_full[0][i & 1]);
        // key tile b: its (i-1)-th query tile
        if (has_b && i >= 1) {
          const int ib = i - 1;
          if (ib >= 2 && !(ok = mbar_wait(&st.acc_empty[1][ib & 1], ((ib - 2) >> 1) & 1))) break;
          tc_fence_after();
          mma_tile<D>(tAcc(1, ib & 1), smem_u32(sK + kT), smem_u32(sQ + s * kT));
          umma_commit(&st.acc_full[1][ib & 1]);
        }
        umma_commit(&st.q_empty[s]);
      }
      if (!ok) {
        st.abort = 1;
        umma_commit(&st.drain);
        mbar_wait(&st.drain, 0);
      }
    }
  } else {
    // ---------------------------------------------------------- epilogue
    const int t = warp >> 3;           // key tile
    const int half = (warp >> 2) & 1;  // query columns 64*half ..
    const int quarter = warp & 3;      // TMEM lanes 32*quarter ..
    const int row = quarter * 32 + lane;
    const int kt = t ? ktb : kta;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    float &acc = cs_acc;
    bool ok = true;
    {
      for (int i = 0; i < n; ++i) {
        const int s = i % kCsStages;
        if (t == 1 && (i == 0 || !has_b)) {
          // the first query tile belongs to key tile a only (and without a key
          // tile b none does): release the stage, every use counts 16 warps
          __syncwarp();
          if (lane == 0) mbar_arrive(&st.q_empty[s]);
          continue;
        }
        const int it = t ? i - 1 : i;  // this key tile's own tile count
        if (!(ok = wait_warp(&st.acc_full[t][it & 1], (it >> 1) & 1) &&
                   wait_warp(&st.q_full[s], (i / kCsStages) & 1)))
          break;
        tc_fence_after();
        uint32_t r[64];
        tmem_ld64(tAcc(t, it & 1) + lane_off + (uint32_t)(half * 64), r);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(&st.acc_empty[t][it & 1]);  // the accumulator is in registers
        const float4 *nl4 = reinterpret_cast<const float4 *>(sNl + s * kRows);
        float a4[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: short dependency chains
        // columns c0 .. c0+63 from v; on the diagonal column c counts iff c >= key row
        auto sum64 = [&](const uint32_t (&v)[64], int c0) {
          if (it == 0) {
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
              const float4 nv = nl4[c0 / 4 + c4];
              const float nn[4] = {nv.x, nv.y, nv.z, nv.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const float e = ex2(fmaf(__uint_as_float(v[4 * c4 + u]), qscale, nn[u]));
                a4[u] += (c0 + 4 * c4 + u >= row) ? e : 0.f;
              }
            }
          } else {
#pragma unroll
            for (int c4 = 0; c4 < 16; ++c4) {
              const float4 nv = nl4[c0 / 4 + c4];
              a4[0] += ex2(fmaf(__uint_as_float(v[4 * c4]), qscale, nv.x));
              a4[1] += ex2(fmaf(__uint_as_float(v[4 * c4 + 1]), qscale, nv.y));
              a4[2] += ex2(fmaf(__uint_as_float(v[4 * c4 + 2]), qscale, nv.z));
              a4[3] += ex2(fmaf(__uint_as_float(v[4 * c4 + 3]), qscale, nv.w));
            }
          }
        };
        sum64(r, half * 64);
        acc += (a4[0] + a4[1]) + (a4[2] + a4[3]);
        __syncwarp();
        if (lane == 0) mbar_arrive(&st.q_empty[s]);  // done with this stage's -LSE vector
      }
      if (!ok) st.abort = 1;
      else if (half == 1) sXch[t * kRows + row] = acc;  // the upper half hands its sum over
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp < kCsEpiWarps) {
    const int t = warp >> 3, half = (warp >> 2) & 1, row = (warp & 3) * 32 + lane;
    const int key = (t ? ktb : kta) * kRows + row;
    if (!st.abort && half == 0 && (t == 0 || has_b) && key < L)
      colsum[(size_t)h * L + key] = cs_acc + sXch[t * kRows + row];
  }
  if (st.abort && tid == 0) atomicOr(err, 4);
  if (warp == 0) tmem_dealloc(tbase, 512);
}

// ----------------------------------------------------------------- host side
PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static bool tried = false;
  if (!tried) {
    tried = true;
    void *p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = (PFN_cuTensorMapEncodeTiled_v12000)p;
  }
  return fn;
}

// [nh][L][d] bf16 viewed as a 3-D tensor; boxes of 64 columns x 128 rows of
// one head, 128-byte swizzle; rows past L read as zero.
bool make_map(CUtensorMap *m, const void *base, int d, int L, int nh) {
  auto fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {(cuuint64_t)d, (cuuint64_t)L, (cuuint64_t)nh};
  cuuint64_t strides[2] = {(cuuint64_t)d * 2, (cuuint64_t)L * d * 2};
  cuuint32_t box[3] = {64, (cuuint32_t)kRows, 1};
  cuuint32_t es[3] = {1, 1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box, es,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// Each CTA of the LSE pass holds 256 TMEM columns, so at most two may share
// an SM's 512: the d = 64 kernel requests the d = 128 shared memory footprint
// to keep a third CTA off the SM instead of blocking in tcgen05.alloc.
constexpr int kTwoPerSmSmem = TileGeo<128>::kSmem;

template <int D>
cudaError_t colsum_pair_t(const CacheView &c, const void *Q, const void *K, const float *lse, float *colsum, int L,
                          cudaStream_t st) {
  CUtensorMap mq, mk;
  if (!make_map(&mq, Q, D, L, c.nh) || !make_map(&mk, K, D, L, c.nh)) return cudaErrorInvalidValue;
  const int smem = CsGeo<128>::kSmem;  // one CTA per SM (512 TMEM columns) for both widths
  cudaError_t e = cudaFuncSetAttribute(colsum_pair_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nqt = (L + kRows - 1) / kRows;
  const int npair = (nqt + 1) / 2;
  const long long grid = (long long)npair * c.nh;
  colsum_pair_tc<D><<<(unsigned)grid, kCsThreads, smem, st>>>(mq, mk, lse, colsum, L, nqt, npair,
                                                               kLog2e / sqrtf((float)D), c.err);
  return cudaGetLastError();
}


// One CTA per SM: 512 TMEM columns each (the d = 64 instance requests the
// d = 128 shared-memory footprint so that no second CTA waits in
// tcgen05.alloc).
constexpr int kPairSmem = PairGeo<128>::kSmem;

template <int D>
cudaError_t attn_pair_t(const CacheView &c, const void *Q, const void *K, const void *V, float *lse, void *O,
                        int L, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, Q, D, L, c.nh) || !make_map(&mk, K, D, L, c.nh) || !make_map(&mv, V, D, L, c.nh))
    return cudaErrorInvalidValue;
  const int smem = kPairSmem;
  cudaError_t e = cudaFuncSetAttribute(attn_pair_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nqt = (L + kRows - 1) / kRows;
  const int npair = (nqt + 1) / 2;
  const long long grid = (long long)npair * c.nh;
  attn_pair_tc<D><<<(unsigned)grid, kPairThreads, smem, st>>>(mq, mk, mv, lse, (__nv_bfloat16 *)O, L, nqt, npair,
                                                             kLog2e / sqrtf((float)D), c.err);
  return cudaGetLastError();
}

template <int D>
cudaError_t lse_t(const CacheView &c, const void *Q, const void *K, float *lse, int L, cudaStream_t st) {
  CUtensorMap mq, mk;
  if (!make_map(&mq, Q, D, L, c.nh) || !make_map(&mk, K, D, L, c.nh)) return cudaErrorInvalidValue;
  const int smem = kTwoPerSmSmem;
  cudaError_t e = cudaFuncSetAttribute(lse_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nqt = (L + kRows - 1) / kRows;
  const long long grid = (long long)nqt * c.nh;
  lse_tc<D><<<(unsigned)grid, kThreads, smem, st>>>(mq, mk, lse, L, nqt, kLog2e / sqrtf((float)D), c.err);
  return cudaGetLastError();
}

}  // namespace

bool prefill_tc_supported(const CacheView &c, int L) {
  return c.dtype == 1 && (c.d == 64 || c.d == 128) && L >= 1 && (long long)c.nh * ((L + 127) / 128) < (1LL << 31) &&
         encode_fn() != nullptr;
}

// Pass 1 on the tensor cores: with an O output, one attention pass writes O
// and the row log-sum-exp; without it, the LSE-only pass (no PV work).
cudaError_t launch_prefill_attn_tc(const CacheView &c, const void *Q, const void *K, const void *V, void *O,
                                   float *lse, int L, cudaStream_t st) {
  if (!O) return c.d == 128 ? lse_t<128>(c, Q, K, lse, L, st) : lse_t<64>(c, Q, K, lse, L, st);
  return c.d == 128 ? attn_pair_t<128>(c, Q, K, V, lse, O, L, st) : attn_pair_t<64>(c, Q, K, V, lse, O, L, st);
}

cudaError_t launch_prefill_colsum_tc(const CacheView &c, const void *Q, const void *K, const float *lse,
                                     float *colsum, int L, cudaStream_t st) {
  return c.d == 128 ? colsum_pair_t<128>(c, Q, K, lse, colsum, L, st) : colsum_pair_t<64>(c, Q, K, lse, colsum, L, st);
}

}  // namespace h2o
