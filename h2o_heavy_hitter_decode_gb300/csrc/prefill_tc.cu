// prefill_tc.cu — tensor-core prefill passes for bf16 caches (sm_103a:
// tcgen05.mma with TMEM accumulators, TMA tile loads, mbarrier pipeline).
//
// H2O summary page, "Algorithm / figure walkthrough" step 1: the prompt's
// accumulated attention score of key j is its causal column sum
//   colsum_j = sum_{i >= j} exp(q_i.k_j / sqrt(d) - LSE_i).
//
// Column-sum pass (the score pass).  A CTA owns a tile of 128 keys, which is
// the MMA's A operand (M = 128 TMEM lanes, one key per thread) and stays in
// shared memory; query tiles of 128 stream in through a two-stage TMA ring as
// the B operand (N = 128).  S^T = K Q^T lands in one of two TMEM accumulator
// buffers, so the MMA of query tile j+1 runs while the epilogue warps turn
// tile j into exp2(s * log2(e)/sqrt(d) - LSE_i * log2(e)) and add it along
// their TMEM row: every key's sum stays in one thread, deterministic and
// atomic-free.  Only the first query tile of a key tile touches the diagonal
// and needs the causal mask; query rows past L are zero-filled by TMA and
// masked by LSE = +inf.  Each CTA runs two key tiles back to back (tile p,
// then tile nkt-1-p, reloading the resident tile in between), so every CTA
// streams nkt + 1 query tiles whatever its place in the causal triangle.
//
// LSE pass.  The same pipeline with the roles swapped: a CTA owns 128 queries
// (A operand, TMEM lanes) and streams the key tiles 0..diagonal; each thread
// keeps an online (max, sum) of its row in base 2.
//
// Warp roles: thread 0 issues TMA and MMA; all four warps run the epilogue
// (warp w reads TMEM lanes 32w..32w+31).  Every mbarrier wait is bounded; on
// a timeout the CTA flags the cache's error word, drains what it issued and
// frees its TMEM before returning.
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
  uint64_t mma_full[2];       // accumulator (and its column vector) ready
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
// into two TMEM accumulators and, per tile, fills that tile's column vector
// with `prep(j, lane)` before marking the accumulator full; warps 0-7 wait
// for it, call `epi(segment, j_in_segment, taddr)` with the TMEM address of
// their 32 lanes and 64-column half, and release the accumulator.  At the
// segment boundary the producer waits for the first segment's last MMA
// (a_free) and reloads the resident tile.  No CTA-wide barrier inside the
// loop.
template <int D, bool kPrep, class Prep, class Epi>
__device__ __forceinline__ bool tile_pipeline(uint8_t *smem, SmallState &st, const CUtensorMap *mapA,
                                              const CUtensorMap *mapB, Seg s0_, Seg s1_, int h, Prep &&prep,
                                              Epi &&epi) {
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
      mbar_init(&st.mma_full[b], kPrep ? 2 : 1);
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
    if (kPrep) prep.load(0, lane);
    for (int j = 0; ok && j < n; ++j) {
      // the whole warp observes the accumulator (and its column vector) free
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
      if (kPrep) {  // the accumulator buffer's column vector (free: its epilogue is done)
        prep.store(j, lane);
        if (j + 1 < n) prep.load(j + 1, lane);
        __syncwarp();
        if (lane == 0) mbar_arrive(&st.mma_full[j & 1]);
      }
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

// ------------------------------------------------------------- column sums
// A CTA takes key tile p and key tile nkt-1-p of one head (two segments of
// the pipeline): nkt - p and p + 1 query tiles, nkt + 1 in all, so the causal
// triangle splits into equal CTAs.
template <int D>
__global__ void __launch_bounds__(kThreads, 2)
    colsum_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
              const float *__restrict__ lse, float *__restrict__ colsum, int L, int nkt, float qscale, int *err) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  using G = TileGeo<D>;
  float *nl2 = (float *)(smem + G::kTileBytes * (1 + kStages));  // [2][128]: -LSE*log2(e) per query
  float *raw = nl2 + 2 * kRows;                                   // [3][128]: LSE slices in flight
  SmallState &st = *(SmallState *)(raw + 3 * kRows);
  if (*(volatile int *)err) return;
  // Head-major (a head's CTAs share its Q tiles in L2).
  const int npair = (nkt + 1) / 2;
  const int h = blockIdx.x / npair, pr = blockIdx.x % npair;
  const int kta = pr, ktb = nkt - 1 - pr;
  const int k0a = kta * kRows, k0b = ktb * kRows;
  const int na = nkt - kta, nb = (ktb != kta) ? nkt - ktb : 0;  // query tiles of each segment
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int row = (warp & 3) * 32 + lane;  // key within the tile (TMEM lane)
  const int c_off = (warp >> 2) * 64;      // this warp's query columns
  const float *lse_h = lse + (size_t)h * L;
  // Column vector of streamed tile j (query tile k0 + 128 j' of its
  // segment): -LSE * log2(e) (-inf past L, so those zero-filled query rows
  // add nothing).  The producer lanes fetch each tile's LSE slice with
  // asynchronous 4-byte copies two tiles ahead (a three-slot staging ring),
  // so no global load latency sits on the path that issues the MMAs.
  struct Prep {
    const float *lse_h;
    float *nl2, *raw;
    int k0a, k0b, na, L, n;
    __device__ int q0(int j) const { return j < na ? k0a + kRows * j : k0b + kRows * (j - na); }
    __device__ void fetch(int j, int ln) {  // copies of tile j, one commit group
      if (j < n) {
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const int q = q0(j) + ln + 32 * i;
          if (q < L) {
            asm volatile("cp.async.ca.shared.global [%0], [%1], 4;" ::"r"(
                             sm100::smem_u32(raw + (j % 3) * kRows + ln + 32 * i)),
                         "l"(lse_h + q)
                         : "memory");
          }
        }
      }
      asm volatile("cp.async.commit_group;" ::: "memory");
    }
    __device__ void load(int j, int ln) {
      if (j == 0) {
        fetch(0, ln);
        fetch(1, ln);
      }
    }
    __device__ void store(int j, int ln) {  // tile j landed (at most one newer group pending)
      asm volatile("cp.async.wait_group 1;" ::: "memory");
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        const int q = q0(j) + ln + 32 * i;
        nl2[(j & 1) * kRows + ln + 32 * i] = q < L ? -raw[(j % 3) * kRows + ln + 32 * i] * kLog2e : -INFINITY;
      }
      fetch(j + 2, ln);
    }
  } prep{lse_h, nl2, raw, k0a, k0b, na, L, na + nb};
  float acc[2] = {0.f, 0.f};  // this thread's key row, per segment
  auto epi = [&](int seg, int j, uint32_t taddr) {
    const float *nl = nl2 + ((seg ? na + j : j) & 1) * kRows + c_off;
    uint32_t r[64];
    tmem_ld64(taddr, r);
    float a4[4] = {0.f, 0.f, 0.f, 0.f};  // four partial sums: short dependency chains
    if (j == 0) {  // diagonal tile: query column c contributes iff c >= key row
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        const float e = ex2(fmaf(__uint_as_float(r[i]), qscale, nl[i]));
        a4[i & 3] += (c_off + i >= row) ? e : 0.f;
      }
    } else {
#pragma unroll
      for (int i = 0; i < 64; ++i) a4[i & 3] += ex2(fmaf(__uint_as_float(r[i]), qscale, nl[i]));
    }
    const float a = (a4[0] + a4[1]) + (a4[2] + a4[3]);
    if (seg) acc[1] += a;
    else acc[0] += a;
  };
  const bool ok = tile_pipeline<D, true>(smem, st, &tmK, &tmQ, Seg{k0a, k0a, na}, Seg{k0b, k0b, nb}, h, prep, epi);
  // the two column halves of each key row: the second half hands its sums over
  float *half = nl2;  // [2][128], free after the pipeline
  if (ok && warp >= 4 && warp < kEpiWarps) {
    half[row] = acc[0];
    half[kRows + row] = acc[1];
  }
  __syncthreads();
  if (ok) {
    if (warp < 4) {
      if (k0a + row < L) colsum[(size_t)h * L + k0a + row] = acc[0] + half[row];
      if (nb > 0 && k0b + row < L) colsum[(size_t)h * L + k0b + row] = acc[1] + half[kRows + row];
    }
  } else if (tid == 0) {
    atomicOr(err, 4);
  }
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
  struct NoPrep {
    __device__ void load(int, int) {}
    __device__ void store(int, int) {}
  } prep;
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
  const bool ok = tile_pipeline<D, false>(smem, st, &tmQ, &tmK, Seg{q0, 0, nk}, Seg{0, 0, 0}, h, prep, epi);
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

// ------------------------------------------------------- attention pass
// Causal attention over the prompt in one pass: O and the row log-sum-exp.
// One CTA per 128 queries.  Warp 8 is the producer: TMA for Q (resident) and
// the K and V rings, the S = Q K^T MMAs into two TMEM buffers and the
// O += P V MMAs (V is the MN-major B operand) into a TMEM accumulator.  Warps
// 0-7 (two per TMEM lane quarter, 64 key columns each) turn S into bf16
// P = exp2(s*c - m) in shared memory (128-byte swizzled K-major layout, the A
// operand of the PV MMA) with an online row max m and an fp32 row sum l.  The
// two warps of a row exchange their half-row maxima through each other's P
// rows.  O is rescaled (tcgen05.ld/st) only when a row's max grows by more
// than 2^8 over the max its P values were taken against, so P stays <= 256
// and rescales are rare; O / l and LSE = (m + log2 l) ln 2 are written at the
// end.  Barriers: kfull/vfull (TMA landed), sfull (S_j computed), sfree (S_j
// read), pfull (P_j written), pvdone (O += P_j V_j done: P buffer and V stage
// free), pair (half-row exchange between the two warps of a row).
template <int D> struct OutGeo {
  static constexpr int kTile = TileGeo<D>::kTileBytes;  // 128 rows x D bf16
  static constexpr int kP = 128 * 128 * 2;               // P tile: 128 queries x 128 keys
  static constexpr int kSmem = kTile * 5 + kP * 2 + 256 + 1024;
};

struct __align__(8) OutState {
  uint64_t res, kfull[2], vfull[2], sfull[2], sfree[2], pfull[2], pvdone[2], drain;
  uint64_t pair[2][4];  // [tile parity][lane quarter]: both warps of a row wrote their half-row max
  uint64_t pair_l[4];   // [lane quarter]: both warps wrote their half-row sum
  uint32_t tmem_base;
  int abort;
};

constexpr int kOutSoftmaxWarps = 8;  // 2 per TMEM lane quarter, 64 key columns each
constexpr int kOutThreads = 32 * (kOutSoftmaxWarps + 1);

template <int D>
__global__ void __launch_bounds__(kOutThreads, 1)
    attn_out_tc(const __grid_constant__ CUtensorMap tmQ, const __grid_constant__ CUtensorMap tmK,
                const __grid_constant__ CUtensorMap tmV, float *__restrict__ lse, __nv_bfloat16 *__restrict__ O,
                int L, int nh, int nqt, float qscale, int *err) {
  using G = OutGeo<D>;
  constexpr int kT = G::kTile;
  extern __shared__ uint8_t smem_raw[];
  uint8_t *smem = align1024(smem_raw);
  uint8_t *sV = smem;              // 2 stages (first: keeps MMA reads of V inside the tile area)
  uint8_t *sK = smem + 2 * kT;     // 2 stages
  uint8_t *sQ = smem + 4 * kT;     // resident
  uint8_t *sP = smem + 5 * kT;     // 2 buffers of kP
  OutState &st = *(OutState *)(sP + 2 * G::kP);
  if (*(volatile int *)err) return;
  // Head-major (a head's CTAs share its K/V tiles in L2), heaviest query tile first.
  const int h = blockIdx.x / nqt, qt = nqt - 1 - blockIdx.x % nqt;
  const int q0 = qt * kRows;
  const int n = qt + 1;  // key tiles 0 .. diagonal
  const int tid = threadIdx.x, warp = tid >> 5;

  if (tid == 0) {
    mbar_init(&st.res, 1);
    for (int b = 0; b < 2; ++b) {
      mbar_init(&st.kfull[b], 1);
      mbar_init(&st.vfull[b], 1);
      mbar_init(&st.sfull[b], 1);
      mbar_init(&st.sfree[b], 32 * kOutSoftmaxWarps);
      mbar_init(&st.pfull[b], 32 * kOutSoftmaxWarps);
      mbar_init(&st.pvdone[b], 1);
    }
    mbar_init(&st.drain, 1);
    for (int qq = 0; qq < 4; ++qq) {
      mbar_init(&st.pair[0][qq], 64);
      mbar_init(&st.pair[1][qq], 64);
      mbar_init(&st.pair_l[qq], 64);
    }
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
  const uint32_t tbase = st.tmem_base;  // S buffers at columns 0 and 128, O at 256
  const uint32_t tO = tbase + 256;

  if (warp == kOutSoftmaxWarps) {
    if ((tid & 31) == 0) {
      constexpr uint32_t idO = idesc_bf16_f32(128, D, true);
      int kl = 0, vl = 0, mS = 0, mPV = 0;  // TMA loads and MMAs issued
      bool ok = true;
      load_tile<D>(sQ, &tmQ, &st.res, q0, h);
      for (; kl < n && kl < 2; ++kl) load_tile<D>(sK + kl * kT, &tmK, &st.kfull[kl], kRows * kl, h);
      for (; vl < n && vl < 2; ++vl) load_tile<D>(sV + vl * kT, &tmV, &st.vfull[vl], kRows * vl, h);
      ok = mbar_wait(&st.res, 0);
      auto issue_S = [&](int j) -> bool {
        if (!mbar_wait(&st.kfull[j & 1], (j >> 1) & 1)) return false;
        if (j >= 2 && !mbar_wait(&st.sfree[j & 1], ((j - 2) >> 1) & 1)) return false;
        tc_fence_after();
        mma_tile<D>(tbase + (uint32_t)(j & 1) * 128, smem_u32(sQ), smem_u32(sK + (j & 1) * kT));
        umma_commit(&st.sfull[j & 1]);
        return true;
      };
      if (ok) ok = issue_S(0);
      if (ok) mS = 1;
      for (int j = 0; ok && j < n; ++j) {
        if (j + 1 < n) {
          if (!(ok = issue_S(j + 1))) break;
          mS = j + 2;
        }
        if (j >= 1 && vl < n) {  // V stage of tile j-1 frees when its PV is done
          if (!(ok = mbar_wait(&st.pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1))) break;
          load_tile<D>(sV + (vl & 1) * kT, &tmV, &st.vfull[vl & 1], kRows * vl, h);
          ++vl;
        }
        if (kl < n) {  // K stage of tile j frees when S_j is done
          if (!(ok = mbar_wait(&st.sfull[j & 1], (j >> 1) & 1))) break;
          load_tile<D>(sK + (kl & 1) * kT, &tmK, &st.kfull[kl & 1], kRows * kl, h);
          ++kl;
        }
        if (!(ok = mbar_wait(&st.pfull[j & 1], (j >> 1) & 1))) break;
        if (!(ok = mbar_wait(&st.vfull[j & 1], (j >> 1) & 1))) break;
        tc_fence_after();
        const uint32_t pa = smem_u32(sP + (j & 1) * G::kP), va = smem_u32(sV + (j & 1) * kT);
#pragma unroll
        for (int kk = 0; kk < 8; ++kk) {  // 128 keys, 16 per MMA
          const uint64_t ad = sdesc_sw128(pa + (uint32_t)((kk >> 2) * kBox + (kk & 3) * 32), 16, 1024);
          const uint64_t bd = sdesc_sw128(va + (uint32_t)(kk * 2048), kBox, 1024);
          umma_bf16(tO, ad, bd, idO, (j > 0 || kk > 0) ? 1u : 0u);
        }
        umma_commit(&st.pvdone[j & 1]);
        mPV = j + 1;
      }
      if (!ok) {
        st.abort = 1;
        // Drain every MMA and TMA copy this CTA issued before releasing
        // shared memory and TMEM.
        umma_commit(&st.drain);
        mbar_wait(&st.drain, 0);
        for (int j = mS; j < kl; ++j) mbar_wait(&st.kfull[j & 1], (j >> 1) & 1);
        for (int j = mPV; j < vl; ++j) mbar_wait(&st.vfull[j & 1], (j >> 1) & 1);
      }
      (void)mPV;
    }
  } else {
    // Softmax warps: query row `row` (TMEM lane), key columns c_off .. c_off+63.
    const int lane = tid & 31;
    const int quarter = warp & 3;
    const int row = quarter * 32 + lane;
    const int half = warp >> 2;
    const int c_off = half * 64;
    const int q = q0 + row;
    const uint32_t lane_off = (uint32_t)(quarter * 32) << 16;
    const int sw = row & 7;
    constexpr int kHalfD = D / 2;  // output columns of this warp
    float m_run = -INFINITY, l_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n; ++j) {
      if (j >= 2 && !(ok = wait_warp(&st.pvdone[j & 1], ((j - 2) >> 1) & 1))) break;
      if (!(ok = wait_warp(&st.sfull[j & 1], (j >> 1) & 1))) break;
      tc_fence_after();
      const bool diag = (j == n - 1);
      uint32_t r[64];
      tmem_ld64(tbase + lane_off + (uint32_t)(j & 1) * 128 + (uint32_t)c_off, r);
      float hm4[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};  // partial maxima
#pragma unroll
      for (int i = 0; i < 64; ++i) {
        float x = __uint_as_float(r[i]) * qscale;
        if (diag && c_off + i > row) x = -INFINITY;  // key after the query
        r[i] = __float_as_uint(x);
        hm4[i & 3] = fmaxf(hm4[i & 3], x);
      }
      const float hm = fmaxf(fmaxf(hm4[0], hm4[1]), fmaxf(hm4[2], hm4[3]));
      tc_fence_before();
      mbar_arrive(&st.sfree[j & 1]);  // the logits are in registers: S buffer free
      // Half-row maxima: each warp writes into the partner's rows of this P
      // buffer (free: its last PV is done), which the partner reads before it
      // overwrites them with its own P.
      uint8_t *pbuf = sP + (j & 1) * G::kP;
      *reinterpret_cast<float *>(pbuf + (1 - half) * kBox + row * 128) = hm;
      mbar_arrive(&st.pair[j & 1][quarter]);
      if (!(ok = wait_warp(&st.pair[j & 1][quarter], (j >> 1) & 1))) break;
      const float m_tile = fmaxf(hm, *reinterpret_cast<const float *>(pbuf + half * kBox + row * 128));
      float m_new = m_run;
      bool resc = false;
      if (m_run == -INFINITY) {
        m_new = m_tile;  // the row's first logits: nothing accumulated yet
      } else if (m_tile > m_run + 8.f) {
        m_new = m_tile;
        resc = true;
      }
      if (__any_sync(0xffffffffu, resc)) {
        // O must hold every earlier P V before it is rescaled
        if (!(ok = wait_warp(&st.pvdone[(j - 1) & 1], ((j - 1) >> 1) & 1))) break;
        tc_fence_after();
        const float f = resc ? ex2(m_run - m_new) : 1.f;
#pragma unroll 1
        for (int cc = 0; cc < kHalfD; cc += 32) {
          uint32_t o[32];
          const uint32_t ta = tO + lane_off + (uint32_t)(half * kHalfD + cc);
          tmem_ld32(ta, o);
          tmem_ld_wait();
          tmem_regs_ready(o);
#pragma unroll
          for (int i = 0; i < 32; ++i) o[i] = __float_as_uint(__uint_as_float(o[i]) * f);
          tmem_st32(ta, o);
        }
        tmem_st_wait();
        l_run *= f;
      }
      m_run = m_new;
      uint32_t pk[32];
      float ls4[4] = {0.f, 0.f, 0.f, 0.f};  // partial row sums
#pragma unroll
      for (int i = 0; i < 32; ++i) {
        const float a = ex2(__uint_as_float(r[2 * i]) - m_run);  // masked: exp2(-inf) = 0
        const float b = ex2(__uint_as_float(r[2 * i + 1]) - m_run);
        ls4[i & 3] += a + b;
        __nv_bfloat162 v = __floats2bfloat162_rn(a, b);
        pk[i] = *reinterpret_cast<uint32_t *>(&v);
      }
      l_run += (ls4[0] + ls4[1]) + (ls4[2] + ls4[3]);
      // 64 keys = one 128-byte row of box `half`: eight 16-byte chunks, swizzled by row.
      uint8_t *prow = pbuf + half * kBox + row * 128;
#pragma unroll
      for (int cch = 0; cch < 8; ++cch)
        *reinterpret_cast<uint4 *>(prow + ((cch ^ sw) << 4)) =
            make_uint4(pk[4 * cch], pk[4 * cch + 1], pk[4 * cch + 2], pk[4 * cch + 3]);
      fence_proxy_async_smem();
      tc_fence_before();
      mbar_arrive(&st.pfull[j & 1]);
    }
    if (ok) ok = wait_warp(&st.pvdone[(n - 1) & 1], ((n - 1) >> 1) & 1);
    if (ok) {
      tc_fence_after();
      // Row sum: the halves hand each other l through P buffer 0 (free now).
      *reinterpret_cast<float *>(sP + (1 - half) * kBox + row * 128 + 4) = l_run;
      mbar_arrive(&st.pair_l[quarter]);
      ok = wait_warp(&st.pair_l[quarter], 0);
    }
    if (ok) {
      const float l_row = l_run + *reinterpret_cast<const float *>(sP + half * kBox + row * 128 + 4);
      const float inv = 1.f / l_row;
      __nv_bfloat16 *orow = O + ((size_t)h * L + (q < L ? q : 0)) * D + half * kHalfD;
#pragma unroll 1
      for (int c0 = 0; c0 < kHalfD; c0 += 32) {  // collective loads: every lane, every chunk
        uint32_t o[32];
        tmem_ld32(tO + lane_off + (uint32_t)(half * kHalfD + c0), o);
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
      if (half == 0 && q < L) lse[(size_t)h * L + q] = (m_run + __log2f(l_row)) * kLn2;
    } else {
      st.abort = 1;
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (st.abort && tid == 0) atomicOr(err, 16);
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

// Each CTA of the LSE and column-sum passes holds 256 TMEM columns, so at most
// two may share an SM's 512: the d = 64 kernels request the d = 128 shared
// memory footprint to keep a third CTA off the SM instead of blocking in
// tcgen05.alloc.
constexpr int kTwoPerSmSmem = TileGeo<128>::kSmem;

template <int D>
cudaError_t colsum_t(const CacheView &c, const void *Q, const void *K, const float *lse, float *colsum, int L,
                     cudaStream_t st) {
  CUtensorMap mq, mk;
  if (!make_map(&mq, Q, D, L, c.nh) || !make_map(&mk, K, D, L, c.nh)) return cudaErrorInvalidValue;
  const int smem = kTwoPerSmSmem;
  cudaError_t e = cudaFuncSetAttribute(colsum_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nkt = (L + kRows - 1) / kRows;
  const long long grid = (long long)((nkt + 1) / 2) * c.nh;  // key-tile pairs
  colsum_tc<D><<<(unsigned)grid, kThreads, smem, st>>>(mq, mk, lse, colsum, L, nkt, kLog2e / sqrtf((float)D),
                                                      c.err);
  return cudaGetLastError();
}

template <int D>
cudaError_t attn_out_t(const CacheView &c, const void *Q, const void *K, const void *V, float *lse, void *O,
                       int L, cudaStream_t st) {
  CUtensorMap mq, mk, mv;
  if (!make_map(&mq, Q, D, L, c.nh) || !make_map(&mk, K, D, L, c.nh) || !make_map(&mv, V, D, L, c.nh))
    return cudaErrorInvalidValue;
  const int smem = OutGeo<D>::kSmem;
  cudaError_t e = cudaFuncSetAttribute(attn_out_tc<D>, cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (e != cudaSuccess) return e;
  const int nqt = (L + kRows - 1) / kRows;
  const long long grid = (long long)nqt * c.nh;
  attn_out_tc<D><<<(unsigned)grid, kOutThreads, smem, st>>>(mq, mk, mv, lse, (__nv_bfloat16 *)O, L, c.nh, nqt,
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
  return c.d == 128 ? attn_out_t<128>(c, Q, K, V, lse, O, L, st) : attn_out_t<64>(c, Q, K, V, lse, O, L, st);
}

cudaError_t launch_prefill_colsum_tc(const CacheView &c, const void *Q, const void *K, const float *lse,
                                     float *colsum, int L, cudaStream_t st) {
  return c.d == 128 ? colsum_t<128>(c, Q, K, lse, colsum, L, st) : colsum_t<64>(c, Q, K, lse, colsum, L, st);
}

}  // namespace h2o
