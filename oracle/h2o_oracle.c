/* h2o_oracle.c — plain fp64 CPU oracle of H2O (Heavy-Hitter Oracle) KV-cache
 * eviction.  TEST INFRASTRUCTURE ONLY (parity tests, smoke check, CPU baseline);
 * the CUDA library never links or calls it and shares no code with it.
 *
 * The steps follow the H2O summary page ("H2O: Heavy-Hitter Oracle for
 * Efficient Generative Inference", "The mechanism" and "Algorithm / figure
 * walkthrough") in its notation: a cache set S of at most k = k_heavy + k_local
 * entries, each carrying its accumulated attention score F_score.  Nothing is
 * blocked, fused or reordered: every softmax is formed in full from its
 * definition, in double precision, one query at a time.
 *
 * Parity pins (what ties this file to something other than itself) live in
 * tests/test_oracle_pins.py: hand-derived rational worked examples (plain
 * H2O, a pinned sink, the mean-weight ranking), a library attention routine
 * for the Full (k >= length), Local (k_heavy = 0) and sinks-plus-window
 * (n_sink = k_heavy) special cases, Definition 4.3's invariants, conservation
 * of score mass, and brute-force enumeration on tiny inputs.
 */
#include "h2o_oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

static double dot(const double *a, const double *b, int d) {
  double s = 0.0;
  for (int c = 0; c < d; ++c) s += a[c] * b[c];
  return s;
}

/* ------------------------------------------------------ fp8 cache rows */

/* Nearest e4m3 value (OCP FP8 "E4M3FN": 1 sign, 4 exponent bits with bias 7,
 * 3 mantissa bits, no infinities; largest finite 448, smallest subnormal
 * 2^-9), ties to even, saturating at 448.  Written from the format's
 * definition: the quantum of a normal value in [2^E, 2^(E+1)) is 2^(E-3),
 * below 2^-6 it is the subnormal step 2^-9. */
static double e4m3_round(double x) {
  const double a = fabs(x);
  if (a >= 448.0) return copysign(448.0, x);
  double quantum = ldexp(1.0, -9);
  if (a >= ldexp(1.0, -6)) {
    int e;
    frexp(a, &e); /* a = f * 2^e, f in [0.5, 1): a in [2^(e-1), 2^e) */
    quantum = ldexp(1.0, e - 1 - 3);
  }
  return copysign(nearbyint(a / quantum) * quantum, x); /* default mode: ties to even */
}

/* Store one row the way an fp8 cache holds it ("H2O-c"-style composition
 * with quantisation, explainer page "Limitations" and the quantisation
 * compatibility claim): one fp32 scale per row, scale = amax / 448 in fp32
 * (0 for an all-zero row), code_c = e4m3(x_c / scale) with the division in
 * fp32; the row reads back as code_c * scale (exact in double). */
static void fp8_store_row(const double *x, int d, double *row, double *scale) {
  float amax = 0.f;
  for (int c = 0; c < d; ++c) {
    const float a = fabsf((float)x[c]);
    if (a > amax) amax = a;
  }
  const float sc = amax / 448.0f;
  for (int c = 0; c < d; ++c)
    row[c] = (sc > 0.f) ? e4m3_round((double)((float)x[c] / sc)) * (double)sc : 0.0;
  *scale = (double)sc;
}

/* Copy a K/V row into a cache slot: verbatim, or as an fp8 row. */
static void store_row(const double *x, int d, int fp8, double *row, double *scale) {
  if (fp8) {
    fp8_store_row(x, d, row, scale);
  } else {
    memcpy(row, x, sizeof(double) * (size_t)d);
    if (scale) *scale = 1.0;
  }
}

/* ---------------------------------------------------------------- prefill */

typedef struct {
  double colsum;
  int j;
} cand_t;

/* Order for the heavy-hitter choice: larger colsum first; equal colsums put the
 * higher position first (the reading adopted for ties: the newer one stays). */
static int cand_cmp(const void *pa, const void *pb) {
  const cand_t *a = (const cand_t *)pa, *b = (const cand_t *)pb;
  if (a->colsum > b->colsum) return -1;
  if (a->colsum < b->colsum) return 1;
  return (a->j > b->j) ? -1 : (a->j < b->j) ? 1 : 0;
}

static int int_cmp(const void *pa, const void *pb) {
  int a = *(const int *)pa, b = *(const int *)pb;
  return (a > b) - (a < b);
}

/* Step 1 of the walkthrough (fill the cache from the prompt, scoring it at
 * once when the prompt is longer than k), read as: every prompt query attends causally to
 * the prompt (no eviction inside the prompt), each key's F_score is the sum
 * of the softmax weights it received (its causal column sum), and if L > k the
 * cache keeps the k_local most recent positions (the protected local block)
 * plus the k_heavy largest F_scores among the older ones.
 *
 * Policy variants (the page's "Limitations" contrasts H2O with attention-sink
 * streaming and notes the bias of the running sum towards old tokens):
 *   - n_sink > 0 pins positions 0 .. n_sink-1 (they take n_sink of the
 *     k_heavy slots; the other k_heavy - n_sink go to the largest keys among
 *     positions n_sink .. L-k_local-1);
 *   - score_mode 1 ranks by the mean weight instead of the sum: F_score
 *     divided by the number of queries that attended to the position, which
 *     for prompt position j is L - j. */
static double rank_key(double F, int64_t attended, int score_mode) {
  return score_mode ? F / (double)attended : F;
}

static void prefill_head(int d, int L, int kh, int kl, int ns, int mode, int fp8, const double *Q,
                         const double *K, const double *V, double *O, double *lse, double *colsum,
                         int32_t *pos, double *score, double *Ks, double *Vs, double *Ksc, double *Vsc,
                         int32_t *n_valid, double *margin, double *dropped_mass) {
  const int k = kh + kl;
  const double scale = 1.0 / sqrt((double)d);
  double *e = (double *)malloc(sizeof(double) * (size_t)L);
  double *F = (double *)calloc((size_t)L, sizeof(double)); /* F_score per position */

  for (int i = 0; i < L; ++i) {
    const double *qi = Q + (size_t)i * d;
    double m = -INFINITY;
    for (int j = 0; j <= i; ++j) {
      e[j] = scale * dot(qi, K + (size_t)j * d, d);
      if (e[j] > m) m = e[j];
    }
    double l = 0.0;
    for (int j = 0; j <= i; ++j) {
      e[j] = exp(e[j] - m);
      l += e[j];
    }
    if (O) {
      double *oi = O + (size_t)i * d;
      for (int c = 0; c < d; ++c) oi[c] = 0.0;
      for (int j = 0; j <= i; ++j) {
        const double w = e[j] / l;
        const double *vj = V + (size_t)j * d;
        for (int c = 0; c < d; ++c) oi[c] += w * vj[c];
      }
    }
    if (lse) lse[i] = m + log(l);
    for (int j = 0; j <= i; ++j) F[j] += e[j] / l;
  }
  if (colsum) memcpy(colsum, F, sizeof(double) * (size_t)L);

  /* Choose S_0. */
  int *keep = (int *)malloc(sizeof(int) * (size_t)(k > 0 ? k : 1));
  int n = 0;
  double mg = INFINITY, dropped = 0.0;
  if (L <= k) {
    for (int j = 0; j < L; ++j) keep[n++] = j;
  } else {
    const int nc = L - kl; /* candidates for the heavy-hitter slots: 0 .. L-kl-1 */
    const int nfree = kh - ns; /* heavy slots left after the pinned sinks */
    cand_t *c = (cand_t *)malloc(sizeof(cand_t) * (size_t)nc);
    for (int j = 0; j < ns; ++j) keep[n++] = j;
    int m = 0;
    for (int j = ns; j < nc; ++j) {
      c[m].colsum = rank_key(F[j], L - j, mode);
      c[m].j = j;
      ++m;
    }
    qsort(c, (size_t)m, sizeof(cand_t), cand_cmp);
    for (int r = 0; r < nfree; ++r) keep[n++] = c[r].j;
    for (int r = nfree; r < m; ++r) dropped += F[c[r].j];
    if (nfree > 0 && m > nfree) mg = c[nfree - 1].colsum - c[nfree].colsum;
    for (int j = L - kl; j < L; ++j) keep[n++] = j;
    free(c);
    qsort(keep, (size_t)n, sizeof(int), int_cmp);
  }
  for (int s = 0; s < k; ++s) {
    double *ks = Ks + (size_t)s * d, *vs = Vs + (size_t)s * d;
    if (s < n) {
      const int j = keep[s];
      pos[s] = j;
      score[s] = F[j];
      store_row(K + (size_t)j * d, d, fp8, ks, Ksc ? Ksc + s : NULL);
      store_row(V + (size_t)j * d, d, fp8, vs, Vsc ? Vsc + s : NULL);
    } else {
      pos[s] = -1;
      score[s] = 0.0;
      memset(ks, 0, sizeof(double) * (size_t)d);
      memset(vs, 0, sizeof(double) * (size_t)d);
      if (Ksc) Ksc[s] = fp8 ? 0.0 : 1.0;
      if (Vsc) Vsc[s] = fp8 ? 0.0 : 1.0;
    }
  }
  *n_valid = n;
  if (margin) *margin = mg;
  if (dropped_mass) *dropped_mass = dropped;
  free(keep);
  free(e);
  free(F);
}

int h2o_oracle_prefill(int nh, int d, int L, int k_heavy, int k_local, int n_sink, int score_mode,
                       int kv_fp8, const double *Q, const double *K, const double *V,
                       double *O, double *lse, double *colsum,
                       int32_t *pos, double *score, double *Ks, double *Vs, double *Ksc, double *Vsc,
                       int32_t *n_valid, double *margin, double *dropped_mass) {
  if (nh < 0 || d < 1 || L < 1 || k_heavy < 0 || k_local < 0 || k_heavy + k_local < 1)
    return -1;
  if (n_sink < 0 || n_sink > k_heavy || (score_mode != 0 && score_mode != 1)) return -1;
  if (kv_fp8 != 0 && kv_fp8 != 1) return -1;
  if (!Q || !K || !V || !pos || !score || !Ks || !Vs || !n_valid) return -1;
  const int k = k_heavy + k_local;
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < nh; ++h) {
    const size_t hl = (size_t)h * L;
    prefill_head(d, L, k_heavy, k_local, n_sink, score_mode, kv_fp8, Q + hl * d, K + hl * d,
                 V + hl * d, O ? O + hl * d : NULL, lse ? lse + hl : NULL, colsum ? colsum + hl : NULL,
                 pos + (size_t)h * k, score + (size_t)h * k, Ks + (size_t)h * k * d,
                 Vs + (size_t)h * k * d, Ksc ? Ksc + (size_t)h * k : NULL,
                 Vsc ? Vsc + (size_t)h * k : NULL, n_valid + h, margin ? margin + h : NULL,
                 dropped_mass ? dropped_mass + h : NULL);
  }
  return 0;
}

/* ----------------------------------------------------------------- decode */

/* Steps 2-4 of the walkthrough for one head.  At position p the query attends
 * over C = S ∪ {p}; each member of C adds its softmax weight to its F_score
 * (the new entry starts at its own weight).  If |C| <= k the new entry is
 * admitted; otherwise the entry with the lowest (F_score, position) among
 * those not in the local block (positions <= p - k_local) leaves the cache.
 * Variants: positions below n_sink are never candidates; score_mode 1 ranks
 * by F_score over the number of queries that attended to the entry, which at
 * step p is p - position + 1 (an entry, once cached, saw every later query). */
static void decode_head(int d, int kh, int kl, int ns, int mode, int fp8, int64_t p0, int T, int nh,
                        int h, int32_t *pos, double *score, double *Ks, double *Vs, double *Ksc,
                        double *Vsc, int32_t *n_valid,
                        const double *q, const double *kn, const double *vn, double *out,
                        int32_t *evicted, double *margin, double *evicted_mass) {
  const int k = kh + kl;
  const double scale = 1.0 / sqrt((double)d);
  double *w = (double *)malloc(sizeof(double) * (size_t)(k + 1));
  for (int t = 0; t < T; ++t) {
    const int64_t p = p0 + t;
    const size_t row = ((size_t)t * nh + h) * d;
    const double *qt = q + row, *kt = kn + row, *vt = vn + row;
    const int n = *n_valid;

    /* Softmax over C: slots 0..n-1 then the new entry at index n. */
    double m = -INFINITY;
    for (int j = 0; j < n; ++j) {
      w[j] = scale * dot(qt, Ks + (size_t)j * d, d);
      if (w[j] > m) m = w[j];
    }
    w[n] = scale * dot(qt, kt, d);
    if (w[n] > m) m = w[n];
    double l = 0.0;
    for (int j = 0; j <= n; ++j) {
      w[j] = exp(w[j] - m);
      l += w[j];
    }
    for (int j = 0; j <= n; ++j) w[j] /= l;

    if (out) {
      double *o = out + row;
      for (int c = 0; c < d; ++c) o[c] = 0.0;
      for (int j = 0; j < n; ++j) {
        const double *vj = Vs + (size_t)j * d;
        for (int c = 0; c < d; ++c) o[c] += w[j] * vj[c];
      }
      for (int c = 0; c < d; ++c) o[c] += w[n] * vt[c];
    }

    /* Accumulate F_score. */
    for (int j = 0; j < n; ++j) score[j] += w[j];
    const double w_new = w[n];

    int32_t ev = -1;
    double mg = INFINITY;
    if (n + 1 <= k) {
      /* |S| < k: admit. */
      pos[n] = (int32_t)p;
      score[n] = w_new;
      store_row(kt, d, fp8, Ks + (size_t)n * d, Ksc ? Ksc + n : NULL);
      store_row(vt, d, fp8, Vs + (size_t)n * d, Vsc ? Vsc + n : NULL);
      *n_valid = n + 1;
    } else {
      /* Full: lowest (F_score, position) outside the local block leaves. */
      int best = -2; /* slot index, -1 = the new entry, -2 = none yet */
      double best_s = INFINITY, second_s = INFINITY;
      int64_t best_p = 0;
      for (int j = -1; j < n; ++j) {
        const int64_t pj = (j < 0) ? p : (int64_t)pos[j];
        if (pj > p - kl) continue; /* protected: one of the k_local newest */
        if (pj < ns) continue;     /* protected: an attention sink */
        const double sj = rank_key((j < 0) ? w_new : score[j], p - pj + 1, mode);
        if (best == -2 || sj < best_s || (sj == best_s && pj < best_p)) {
          if (best != -2) second_s = best_s;
          best = j;
          best_s = sj;
          best_p = pj;
        } else if (sj < second_s) {
          second_s = sj;
        }
      }
      /* best == -2 cannot happen: of the k+1 entries, k_local are in the
       * local block and at most n_sink <= k_heavy are sinks, so at least
       * k_heavy + 1 - n_sink >= 1 are candidates. */
      if (best >= 0) {
        ev = pos[best];
        if (evicted_mass) *evicted_mass += score[best];
        pos[best] = (int32_t)p;
        score[best] = w_new;
        store_row(kt, d, fp8, Ks + (size_t)best * d, Ksc ? Ksc + best : NULL);
        store_row(vt, d, fp8, Vs + (size_t)best * d, Vsc ? Vsc + best : NULL);
      } else {
        ev = (int32_t)p; /* the new entry itself (only when k_local = 0) */
        if (evicted_mass) *evicted_mass += w_new;
      }
      mg = second_s - best_s;
    }
    if (evicted) evicted[(size_t)t * nh + h] = ev;
    if (margin) margin[(size_t)t * nh + h] = mg;
  }
  free(w);
}

int h2o_oracle_decode(int nh, int d, int k_heavy, int k_local, int n_sink, int score_mode,
                      int kv_fp8, int64_t p0, int T,
                      int32_t *pos, double *score, double *Ks, double *Vs, double *Ksc, double *Vsc,
                      int32_t *n_valid,
                      const double *q, const double *kn, const double *vn,
                      double *out, int32_t *evicted, double *margin, double *evicted_mass) {
  if (nh < 0 || d < 1 || T < 0 || k_heavy < 0 || k_local < 0 || k_heavy + k_local < 1 || p0 < 0)
    return -1;
  if (n_sink < 0 || n_sink > k_heavy || (score_mode != 0 && score_mode != 1)) return -1;
  if (p0 + (int64_t)T > (int64_t)0x7fffffff) return -1;
  if (kv_fp8 != 0 && kv_fp8 != 1) return -1;
  if (!pos || !score || !Ks || !Vs || !n_valid || (T > 0 && (!q || !kn || !vn))) return -1;
  const int k = k_heavy + k_local;
#pragma omp parallel for schedule(dynamic, 1)
  for (int h = 0; h < nh; ++h) {
    decode_head(d, k_heavy, k_local, n_sink, score_mode, kv_fp8, p0, T, nh, h, pos + (size_t)h * k,
                score + (size_t)h * k, Ks + (size_t)h * k * d, Vs + (size_t)h * k * d,
                Ksc ? Ksc + (size_t)h * k : NULL, Vsc ? Vsc + (size_t)h * k : NULL, n_valid + h, q, kn, vn, out,
                evicted, margin, evicted_mass ? evicted_mass + h : NULL);
  }
  return 0;
}

void h2o_oracle_set_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}

int h2o_oracle_max_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}
