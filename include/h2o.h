/* h2o.h — C ABI of libh2o.so: H2O (Heavy-Hitter Oracle) KV-cache eviction on
 * one NVIDIA GB300 (sm_103a).
 *
 * The method is the one of "H2O: Heavy-Hitter Oracle for Efficient Generative
 * Inference of Large Language Models" as summarised on its explainer page
 * ("The mechanism"; "Algorithm / figure walkthrough" steps 1-5;
 * Definition 4.3).  Each (batch b, head h) pair owns an independent cache set
 * S of k = k_heavy + k_local slots.  Every cached key carries F_score, the sum
 * of the softmax attention weights it has received.  At a decode step the new
 * query attends over S plus the new token (k+1 entries, scale 1/sqrt(d)); the
 * exact weights are added to the scores (the new token starts at its own
 * weight); the entry with the lowest (score, position) outside the k_local
 * newest positions is evicted and the new token takes its slot in place.
 * Prefill scores the prompt by causal-softmax column sums and keeps the last
 * k_local positions plus the k_heavy largest column sums of the rest.
 *
 * Conventions for every call below:
 *   - Pointers named as device pointers must be device memory of the device
 *     the cache was created on (or memory that device can address); host
 *     pointers are ordinary host memory.  The caller owns all memory: the
 *     library allocates nothing on the device.
 *   - Tensors are dense row-major in the cache's input type (fp32, or bf16
 *     stored as uint16 bit patterns), with the head index flattened as b*H + h:
 *     prompt tensors [B][H][L][d]; one decode step [B][H][d]; n decode steps
 *     [n][B][H][d].  Device pointers must be 16-byte aligned.
 *   - Work is enqueued asynchronously on the cache's stream (set at create or
 *     with h2o_set_stream); no call synchronises unless it says so.
 *   - Errors are returned as h2o_status and never abort; arguments are checked
 *     on the host before anything is launched, and on error nothing is
 *     launched and the cache is unchanged.
 */
#ifndef H2O_H
#define H2O_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct h2o_cache *h2o_cache_t; /* opaque host-side handle */

typedef enum {
  H2O_OK = 0,
  H2O_EINVAL = 1,   /* bad argument (shape, null or misaligned pointer, range) */
  H2O_ESTATE = 2,   /* call not valid in the cache's state (e.g. decode before prefill) */
  H2O_ECUDA = 3,    /* a CUDA runtime call failed; h2o_last_cuda_error() has the code */
  H2O_ENOMEM = 4,   /* host allocation failed */
  H2O_EDEVICE = 5,  /* the device flagged an internal inconsistency (h2o_get_error) */
  H2O_EUNSUPPORTED = 6 /* valid request this library does not handle (e.g. d not 64/128) */
} h2o_status;

/* Element types of a cache.  H2O_F32 / H2O_BF16: inputs, outputs and the
 * stored K/V slots all in that type.  H2O_BF16_FP8KV: bf16 inputs and
 * outputs; the K/V slots are stored as e4m3 codes (1 byte per element) with
 * one fp32 scale per slot row, the way the explainer page's "Limitations"
 * section says H2O composes with quantisation.  A row x written into a slot
 * gets scale = max|x| / 448 (fp32; 0 for an all-zero row) and codes
 * e4m3(x / scale) (fp32 division, nearest-even, saturating at 448); it reads
 * back as code * scale.  The prefill passes and each decode step's own new
 * token use the bf16 inputs themselves. */
typedef enum { H2O_F32 = 0, H2O_BF16 = 1, H2O_BF16_FP8KV = 2 } h2o_dtype;

/* Bytes of device workspace a cache of this shape needs (0 if the shape is
 * invalid).  The workspace holds, per head: the K and V slots [k][d], the
 * position tags [k] (int32, -1 = empty), the scores [k] (fp32), and the
 * decode step's split partials and counters.  Shape rules: B, H >= 1;
 * d in {64, 128}; k_heavy, k_local >= 0; k = k_heavy + k_local >= 1. */
size_t h2o_cache_workspace_bytes(int B, int H, int d, int k_heavy, int k_local, h2o_dtype dtype);

/* Create a cache over caller-owned device memory `workspace` (at least
 * h2o_cache_workspace_bytes(...) bytes, 256-byte aligned, owned by the caller
 * until h2o_cache_destroy).  `cuda_stream` is a cudaStream_t (NULL = legacy
 * default stream).  Enqueues the initialisation of the workspace (all slots
 * empty).  On success *out receives the handle. */
h2o_status h2o_cache_create(int B, int H, int d, int k_heavy, int k_local, h2o_dtype dtype,
                            void *workspace, void *cuda_stream, h2o_cache_t *out);

/* Free the host-side handle (the workspace stays the caller's).  NULL is OK. */
h2o_status h2o_cache_destroy(h2o_cache_t cache);

/* Change the stream later calls enqueue on. */
h2o_status h2o_set_stream(h2o_cache_t cache, void *cuda_stream);

/* Prefill ("Algorithm / figure walkthrough" step 1): causal attention over the
 * L prompt positions, then the initial cache set.
 *   Q, K, V  device [B][H][L][d], cache dtype.
 *   O        device [B][H][L][d] attention output, or NULL to skip it.
 *   lse      device [B][H][L] fp32, required: natural-log log-sum-exp of each
 *            query row's scaled logits.
 *   colsum   device [B][H][L] fp32, required: colsum_j = sum_{i>=j}
 *            softmax_i(j), the prompt's accumulated attention score.
 * If L <= k every position is kept (slots 0..L-1); otherwise the last k_local
 * positions plus the k_heavy largest column sums among positions
 * 0..L-k_local-1 (equal sums: the higher position is kept).  Kept positions
 * fill slots 0..n-1 in ascending order with score = colsum.  Valid once per
 * cache (H2O_ESTATE otherwise).  L >= 1 and L < 2^31 - 1. */
h2o_status h2o_prefill(h2o_cache_t cache, const void *Q, const void *K, const void *V, int L,
                       void *O, float *lse, float *colsum);

/* The same prefill for batch rows b0 .. b0+nb-1 only (every head of those
 * rows), so a caller can prefill sequences as their prompts arrive, or
 * overlap the copy of one group of rows with the prefill of another.
 * Q, K, V, O, lse, colsum point at those rows: [nb][H][L][d] and
 * [nb][H][L].  Every row of a cache is prefilled exactly once and with the
 * same L (H2O_EINVAL for a different L, H2O_ESTATE for a row already done);
 * decode may start once all B rows are done (H2O_ESTATE before).
 * h2o_prefill is this call with b0 = 0, nb = B. */
h2o_status h2o_prefill_rows(h2o_cache_t cache, int b0, int nb, const void *Q, const void *K, const void *V,
                            int L, void *O, float *lse, float *colsum);

/* One decode step ("Algorithm / figure walkthrough" steps 2-4) for every head,
 * one kernel launch: attend over the cached entries plus the new token,
 * add the exact weights into the scores, evict, write the new token in place.
 *   q_t, k_t, v_t  device [B][H][d]; out device [B][H][d].
 * H2O_ESTATE before prefill/import. */
h2o_status h2o_decode_step(h2o_cache_t cache, const void *q_t, const void *k_t, const void *v_t,
                           void *out);

/* n decode steps in sequence (one launch per step, or one launch for all of
 * them: see h2o_set_decode_form), inputs [n][B][H][d], out [n][B][H][d].
 * evicted: device [n][B][H] int32 or NULL; receives the position evicted at
 * each step (-1 when the new token was admitted without eviction; the new
 * position itself when it was the lowest-scoring candidate, which can only
 * happen with k_local = 0). */
h2o_status h2o_decode_steps(h2o_cache_t cache, int n, const void *q, const void *k, const void *v,
                            void *out, int32_t *evicted);

/* How h2o_decode_steps runs n >= 2 steps (all forms compute the same thing;
 * single steps always use form 1):
 *   0  automatic (default): 4 for a bf16 or fp32 cache and 3 for an fp8
 *      cache if the shape allows it, else 2 when all its CTAs fit on the
 *      device at once, else 1;
 *   1  one launch per step, chained with programmatic dependent launch;
 *   2  one cooperative launch: each (head, split) CTA loops over the steps,
 *      waiting (bounded, acquire) only on its own head's previous step;
 *   3  one launch with a thread-block cluster of up to 8 CTAs per head:
 *      scores and tags stay in shared memory, partials and eviction
 *      candidates move over distributed shared memory (asynchronous stores
 *      completing on the receivers' mbarriers), every CTA takes the same
 *      decision; no global scratch.
 *   4  form 3 with each step's eviction decision taken while the next
 *      step's attention pass runs: the next pass covers the cache before the
 *      decision, and the decision's one changed slot is then corrected in
 *      its partial (the evicted row's term removed, the admitted row's
 *      added).  Same results as the other forms up to fp32 rounding.
 * A form the shape or device cannot run makes h2o_decode_steps return
 * H2O_EUNSUPPORTED (nothing launched). */
h2o_status h2o_set_decode_form(h2o_cache_t cache, int form);

/* The form (1 to 4 as above) the last decode call of this cache ran with;
 * 0 before any decode call. */
h2o_status h2o_decode_form_used(h2o_cache_t cache, int *form);

/* Eviction policy variants of one cache (explainer page "Limitations":
 * attention-sink streaming as the contrasting policy, and the bias of summed
 * scores towards older tokens).  Both 0 (the default) is plain H2O.
 *   n_sink      0 <= n_sink <= k_heavy: positions 0 .. n_sink-1 are pinned
 *               attention sinks, never evicted; they take n_sink of the
 *               k_heavy slots, so the prefill keeps them, the k_heavy - n_sink
 *               best-ranked positions of n_sink .. L-k_local-1 and the
 *               k_local newest.  n_sink = k_heavy is a sinks-plus-window
 *               cache.
 *   score_mode  0: rank entries by accumulated score; 1: by accumulated score
 *               divided by the number of queries that attended to the entry
 *               (L - j after the prefill for prompt position j, p - j + 1
 *               after the decode step at p).  The stored scores stay plain
 *               sums either way.
 * Applies to every later prefill and decode call; host-only, no device
 * work.  H2O_EINVAL for out-of-range values (nothing changes). */
h2o_status h2o_cache_set_policy(h2o_cache_t cache, int n_sink, int score_mode);
/* Current policy (either pointer may be NULL). */
h2o_status h2o_cache_get_policy(h2o_cache_t cache, int *n_sink, int *score_mode);

/* Copy the cache state out to device buffers: pos [B][H][k] int32,
 * score [B][H][k] fp32, K, V [B][H][k][d] in the stored type (e4m3 codes for
 * H2O_BF16_FP8KV; see h2o_cache_export_scales) (any may be NULL); next_pos and
 * n_valid (host, may be NULL) receive the position the next decode token
 * takes and the number of filled slots.  Asynchronous like every call. */
h2o_status h2o_cache_export(h2o_cache_t cache, int32_t *pos, float *score, void *K, void *V,
                            int64_t *next_pos, int *n_valid);

/* Replace the cache state with caller data (device pos, score, K, V in the
 * layouts of h2o_cache_export, all required; slots >= n_valid must hold
 * pos = -1).  Marks the cache as prefilled.  next_pos >= 0,
 * 0 <= n_valid <= k. */
h2o_status h2o_cache_import(h2o_cache_t cache, const int32_t *pos, const float *score,
                            const void *K, const void *V, int64_t next_pos, int n_valid);

/* Per-row scales of an H2O_BF16_FP8KV cache: device (or host) fp32
 * [B][H][k] arrays for K and V, in the slot order of h2o_cache_export (whose
 * K/V then hold the e4m3 codes, 1 byte per element).  Export: either pointer
 * may be NULL.  Import (both required) after h2o_cache_import, before the
 * next decode call.  H2O_EUNSUPPORTED for other cache types.  Asynchronous. */
h2o_status h2o_cache_export_scales(h2o_cache_t cache, float *K_scale, float *V_scale);
h2o_status h2o_cache_import_scales(h2o_cache_t cache, const float *K_scale, const float *V_scale);

/* Shape and counters of a cache (host pointers, any may be NULL). */
h2o_status h2o_cache_info(h2o_cache_t cache, int *B, int *H, int *d, int *k_heavy, int *k_local,
                          int *dtype, int64_t *next_pos, int *n_valid, int *n_split);

/* Phase timing.  While enabled, each prefill pass and each h2o_decode_steps
 * call is bracketed by CUDA events recorded on the cache's stream:
 * phase 0 = prefill attention (pass 1), 1 = prefill column sums (pass 2),
 * 2 = prefill select + gather, 3 = decode steps.  h2o_profile_read
 * synchronises on the recorded events and returns, per phase, the summed
 * elapsed milliseconds (ms[4]) and the number of kernel launches covered
 * (launches[4]: a multi-step decode form counts one launch per grid, not one
 * per step); it then clears the record.  Either output may be NULL. */
h2o_status h2o_profile_enable(h2o_cache_t cache, int on);
h2o_status h2o_profile_read(h2o_cache_t cache, double *ms, int64_t *launches);

/* Allocation-free decode step (no counterpart in the H2O paper: it is a
 * deployment convenience of this library).
 *
 * Some callers cannot allocate device memory: inference servers that reserve
 * all of HBM up front and hand a plugin only its input and output tensors, C
 * hosts that receive device pointers from another runtime and hold no
 * allocator, and latency-critical loops where a cudaMalloc (which may
 * synchronise the device) is not acceptable.  This entry point runs one decode
 * step for every head — the same kernel and arithmetic as h2o_decode_step —
 * with its scratch (split partials, logits, arrival counters) in a fixed
 * array compiled into the library, so it allocates nothing and needs no
 * h2o_cache_t.
 *
 *   K, V       device [B][H][k][d] cache slots (cache dtype), read and updated.
 *   pos        device [B][H][k] int32 position tags (-1 = empty), updated.
 *   score      device [B][H][k] fp32 accumulated scores, updated.
 *   n_valid    filled slots before this step (0..k), the same for every head.
 *   position   position of the new token (0 <= position < 2^31 - 1).
 *   q_t, k_t, v_t  device [B][H][d]; out device [B][H][d];
 *   evicted    device [B][H] int32 or NULL (as in h2o_decode_steps).
 *   cuda_stream    cudaStream_t to enqueue on (NULL = legacy default stream).
 * The caller advances n_valid (while < k) and position after each call.
 * Layouts are those of h2o_cache_export, so a cache's exported state can be
 * continued here.
 *
 * Limits and sharing: the scratch array holds H2O_STATIC_SCRATCH_BYTES; a
 * shape whose scratch would not fit is rejected with H2O_EINVAL before
 * anything is launched.  Every GPU that loads the library holds the array
 * until the process exits.  All calls share it and it keeps the last call's
 * contents (each call clears what must start at zero), so calls that overlap
 * on the GPU — on different streams, or from different host threads — race
 * and must be serialised by the caller.  The first call on a device looks up
 * the array's device address (cudaGetSymbolAddress, with that device
 * current); make that first call before any stream capture on that device.
 * The address is kept per device together with the context it was looked up
 * in, and looked up again when the calling thread runs that device under
 * another context.  A cudaDeviceReset of the device can reload the library's
 * module at another address under the same primary-context handle, so this
 * entry point is not supported on a device after it has been reset.
 * A CUDA failure returns H2O_ECUDA; the kernel's own consistency flag lives
 * in the shared scratch and is not reported here. */
#define H2O_STATIC_SCRATCH_BYTES (16u << 20)
h2o_status h2o_decode_step_static(int B, int H, int d, int k_heavy, int k_local, h2o_dtype dtype,
                                  void *K, void *V, int32_t *pos, float *score, int n_valid,
                                  int64_t position, const void *q_t, const void *k_t,
                                  const void *v_t, void *out, int32_t *evicted, void *cuda_stream);

/* Synchronises the stream and reads the device-side error flag: H2O_OK, or
 * H2O_EDEVICE if a kernel found an inconsistency (for example no eviction
 * candidate).  The flag is sticky. */
h2o_status h2o_get_error(h2o_cache_t cache);

/* Human-readable name of a status; the last CUDA error code seen by the
 * library (0 = none). */
const char *h2o_status_str(h2o_status s);
int h2o_last_cuda_error(void);

/* Measurement helper (not part of the method): `reps` sweeps of 16-byte
 * reads over the device buffer `buf` of `bytes` (a multiple of 16, 16-byte
 * aligned) through L2, by 4 CTAs of 512 threads per SM, enqueued on
 * cuda_stream.  `sink` is a device uint32 the kernel may write (so the reads
 * are not optimised away).  Timed by the caller (events around the call), it
 * gives the read bandwidth of a buffer of that size: above the L2 capacity the
 * HBM read rate, below it the L2 read rate that a decode over an L2-resident
 * K/V cache runs against.  H2O_EINVAL on bad arguments, nothing launched. */
h2o_status h2o_probe_read(const void *buf, size_t bytes, int reps, uint32_t *sink, void *cuda_stream);

/* Compiled-in target, for checks: returns 1030 for sm_103a. */
int h2o_build_arch(void);

/* What the CUDA runtime loaded on the current device for this library's
 * kernels (cudaFuncGetAttributes of one of them): the PTX ISA target and the
 * binary architecture, major*10 + minor (103 and 103 for an sm_103a build
 * running as its own cubin).  Host pointers, either may be NULL.
 * H2O_ECUDA without a usable device. */
h2o_status h2o_kernel_arch(int *ptx_version, int *binary_version);

#ifdef __cplusplus
}
#endif
#endif
