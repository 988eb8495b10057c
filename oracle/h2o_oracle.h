/* h2o_oracle.h — plain fp64 CPU oracle of H2O (Heavy-Hitter Oracle) KV-cache
 * eviction.
 *
 * TEST INFRASTRUCTURE ONLY: the parity tests, the smoke check and the bench's
 * CPU-baseline leg call this; the product (the CUDA library) never does, and
 * this code shares nothing with it.
 *
 * What it computes follows the H2O summary page ("H2O: Heavy-Hitter Oracle
 * for Efficient Generative Inference", sections "The mechanism" and
 * "Algorithm / figure walkthrough"):
 *   - F_score of a cached key = the softmax attention weights it received,
 *     summed over every query that attended to it;
 *   - the cache set S_i keeps at most k = k_heavy + k_local entries; while
 *     |S| < k a new entry is admitted, once full the newest is admitted and
 *     the lowest-F_score entry outside the k_local most recent positions is
 *     evicted (Definition 4.3: |S_i| = k, |S_i \ S_{i-1}| <= 1).
 * Readings where the page is silent (each also in the function comments):
 *   - the decode query attends over S_{t-1} plus itself (k+1 entries), scale
 *     1/sqrt(d); the new entry's F_score starts at its own weight;
 *   - the prompt is scored by causal-softmax column sums (no eviction inside
 *     the prompt); if L > k the last k_local positions are kept plus the
 *     k_heavy largest column sums of the rest;
 *   - ties: eviction takes the lowest (score, position) pair; prefill keeps the
 *     largest (colsum, position) pairs, i.e. the higher position survives.
 * Policy variants (both parameters 0 give plain H2O):
 *   - n_sink (0 <= n_sink <= k_heavy): positions 0 .. n_sink-1 are pinned
 *     attention sinks, never evicted, taking n_sink of the heavy slots; with
 *     n_sink = k_heavy the cache is exactly sinks + a recent window;
 *   - score_mode 1: eviction and selection rank entries by their mean weight,
 *     F_score / (number of queries that attended to the entry) — L - j for
 *     prompt position j after the prefill, p - j + 1 after the step at p.
 *     The stored F_score stays the plain sum.
 * fp8 cache (kv_fp8 = 1): every K/V row written into a slot is stored as
 *   e4m3 codes with one fp32 scale per row (scale = amax/448 in fp32, 0 for
 *   an all-zero row; code = nearest-even e4m3 of x/scale, the division in
 *   fp32, saturating at 448) and read back as code * scale.  The prefill's
 *   own attention and each decode step's new token use the input values.
 *
 * All arrays are row-major doubles (int32 for positions).  A "head" is one
 * (batch, head) pair; heads are independent.
 */
#ifndef H2O_ORACLE_H
#define H2O_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* Prefill of nh heads.  Q, K, V: [nh][L][d].  Outputs (any may be NULL):
 *   O [nh][L][d] causal attention output, lse [nh][L] natural-log
 *   log-sum-exp of each query row, colsum [nh][L] column sums of the causal
 *   softmax, and the initial cache of each head in k slots:
 *   pos [nh][k] (ascending positions, -1 past n_valid), score [nh][k],
 *   Ks, Vs [nh][k][d] (the values the cache reads back); Ksc, Vsc [nh][k]
 *   (may be NULL) the per-row scales (1 without kv_fp8; 0 for empty slots
 *   with it); n_valid [nh]; margin [nh] = smallest kept minus largest
 *   dropped heavy-candidate ranking key (the colsum, or the mean weight in
 *   score_mode 1; +inf when nothing is dropped by score);
 *   dropped_mass [nh] = sum of dropped colsums.
 * Returns 0, or -1 on bad arguments. */
int h2o_oracle_prefill(int nh, int d, int L, int k_heavy, int k_local, int n_sink, int score_mode,
                       int kv_fp8, const double *Q, const double *K, const double *V,
                       double *O, double *lse, double *colsum,
                       int32_t *pos, double *score, double *Ks, double *Vs, double *Ksc, double *Vsc,
                       int32_t *n_valid, double *margin, double *dropped_mass);

/* T decode steps of nh heads starting at absolute position p0 (the first new
 * token's position).  State (k slots per head) is read and updated in place:
 *   pos [nh][k], score [nh][k], Ks, Vs [nh][k][d], Ksc, Vsc [nh][k] (may be
 *   NULL), n_valid [nh].
 * Step inputs q, kn, vn: [T][nh][d] (step-major).  Outputs (any may be NULL):
 *   out [T][nh][d] attention output of each step;
 *   evicted [T][nh] position evicted at that step (-1 = admitted without
 *   eviction; the new position itself if it was the one evicted);
 *   margin [T][nh] gap between the two smallest ranking keys among the
 *   eviction candidates (+inf when there was no choice);
 *   evicted_mass [nh] (accumulated: sum of F_scores of evicted entries).
 * Returns 0, or -1 on bad arguments. */
int h2o_oracle_decode(int nh, int d, int k_heavy, int k_local, int n_sink, int score_mode,
                      int kv_fp8, int64_t p0, int T,
                      int32_t *pos, double *score, double *Ks, double *Vs, double *Ksc, double *Vsc,
                      int32_t *n_valid,
                      const double *q, const double *kn, const double *vn,
                      double *out, int32_t *evicted, double *margin, double *evicted_mass);

/* OpenMP thread count used across heads (<= 0 leaves the default). */
void h2o_oracle_set_threads(int n);
int h2o_oracle_max_threads(void);

#ifdef __cplusplus
}
#endif
#endif
