/*
 * spec_verify.h -- C ABI of the GB300 (sm_103a) batched speculative-decoding
 * verifier: modified rejection sampling in plain and mu/NULL-gated modes.
 *
 * What one call computes, for every sequence b of a batch of B sequences with
 * k draft positions over a vocabulary of V tokens:
 *
 *   p_j = softmax(Lt[b,j,:] / T), j = 0..k      (target rows, temperature T)
 *   q_j = softmax(Ld[b,j,:] / T), j = 0..k-1    (draft rows)
 *     -- the effective distributions are full-vocabulary temperature softmaxes
 *        evaluated in fp32 (mlxcel PR #992, "What changed").
 *   mu_j = q_j in plain mode; in gated mode mu_j(x) = q_j(x) on admitted tokens
 *     (q_j(x) >= threshold, equality passes) and 0 elsewhere, NOT renormalised
 *     (Strata PR #3416 "Preserve target probabilities in gated MTP", section
 *     "Approach"; equality rule: regolith audit, "schedule behavior").
 *   For j = 0, 1, ...: gated and q_j(D_j) < threshold -> explicit NULL row,
 *     stop; otherwise accept D_j iff p_j(D_j) > 0 and u0 * mu_j(D_j) <= p_j(D_j)
 *     (mlxcel PR #992, "What changed": the accept test and its load-bearing
 *     p > 0 conjunct); stop at the first position not accepted (mlxcel PR
 *     #992, "Two metric corrections").
 *   At the stop position j* < k (rejection or NULL) emit a sample of the
 *     normalised positive part of p_j* - mu_j*; when all k drafts pass emit an
 *     ordinary bonus sample of p_k (Strata PR #3416, "Approach").  Samples are
 *     inverse-CDF picks in token order: the smallest v whose inclusive prefix
 *     sum exceeds u1 * Z.  A residual with no mass falls back to sampling p.
 *   Uniforms: u = Philox4x32-10 (Salmon et al., SC'11) with key = (seed lo32,
 *     seed hi32) and counter = (s lo32, j, draw, s hi32), s = seq_offset + b;
 *     u = (out.x >> 8) * 2^-24.  u0 uses draw 0 at position j, u1 draw 1 at j*.
 *
 * Outputs per sequence: accepted_len = j*, tokens = D_0..D_{j*-1}, the
 * residual/bonus token, then -1 padding; accept_prob[j] = min(1, p/mu) for
 * every position (0 for a NULL row, also filled past j*); optional flags and
 * batch counters.
 *
 * Memory: every logits, token and output pointer is DEVICE memory owned by the
 * caller (except the *_host entry point); rows are contiguous, row-major, V
 * innermost.  The handle owns only its workspace.  Calls are asynchronous on
 * the given stream; one handle must not run two calls at once.
 *
 * Errors: arguments the host can check are validated before any launch and
 * yield a non-zero sv_status with nothing launched.  Problems only the device
 * sees -- a draft token outside [0, V), a row with a NaN or +inf logit or with
 * every logit -inf, a per-sequence threshold outside (0, 1] -- never trap: that
 * sequence gets accepted_len = -1, tokens = -1, flags = SV_FLAG_INVALID,
 * accept_prob = 0, and counters[SV_CNT_INVALID] is incremented.
 */
#ifndef SPEC_VERIFY_H
#define SPEC_VERIFY_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct spec_verify_s* spec_verify_t; /* opaque handle */

typedef enum {
  SV_OK = 0,
  SV_EINVAL = 1,        /* bad argument (shape, pointer, temperature, threshold, dtype) */
  SV_ENOMEM = 2,        /* device or host allocation failed */
  SV_ECUDA = 3,         /* a CUDA runtime call or a launch failed */
  SV_EUNSUPPORTED = 4   /* a size outside the library's limits (see SV_MAX_K, SV_MAX_V) */
} sv_status;

typedef enum { SV_F32 = 0, SV_BF16 = 1 } sv_dtype;

typedef enum { SV_PLAIN = 0, SV_GATED_MU = 1 } sv_gate;

/* per-position flags written to `flags` */
enum {
  SV_FLAG_UNREACHED = 0, /* past the stop position */
  SV_FLAG_ACCEPT = 1,
  SV_FLAG_REJECT = 2,
  SV_FLAG_NULL = 3,      /* gated mode: the offered token failed the gate */
  SV_FLAG_INVALID = 4    /* the sequence was rejected as invalid input */
};

/* slots of the optional `counters` output (uint64, accumulated: the caller zeroes them) */
enum {
  SV_CNT_TESTED = 0,     /* positions tested: accepted ones plus each stop position < k */
  SV_CNT_ACCEPTED = 1,   /* accepted draft tokens */
  SV_CNT_NULL = 2,       /* NULL rows */
  SV_CNT_REJECTED = 3,   /* rejections */
  SV_CNT_BONUS = 4,      /* sequences that accepted all k drafts */
  SV_CNT_BOUNDARY = 5,   /* draws whose uniform (or gated q(D), or the prefix product of the
                            cumulative floor) lay within 1e-6 of its boundary */
  SV_CNT_INVALID = 6,    /* sequences rejected as invalid input */
  SV_CNT_DEGENERATE = 7, /* residuals with no mass that fell back to sampling p */
  SV_NUM_COUNTERS = 8
};

#define SV_MAX_K 32            /* draft positions per sequence */
#define SV_MAX_V (1 << 22)     /* vocabulary size */

/* Create a verifier for batches of up to max_B sequences, k draft positions and
 * vocabulary V on CUDA device `device`.  Allocates the device workspace:
 * max_B * (2k+1) * ceil(V / 2048) * 8 bytes of chunk statistics plus
 * max_B * k * ceil(V / 2048) * 32 bytes of gate-candidate slots.
 * Returns SV_EINVAL for max_B < 1, k < 1 or V < 1, SV_EUNSUPPORTED beyond
 * SV_MAX_K / SV_MAX_V, SV_ENOMEM or SV_ECUDA on CUDA failures; *out is set to
 * NULL on any error. */
sv_status spec_verify_init(spec_verify_t* out, int max_B, int k, int V, int device);

/* Verify a batch (the spec call).
 *   target_logits [B, k+1, V] of dtype tdt, draft_logits [B, k, V] of dtype ddt,
 *   draft_tokens [B, k] int32 -- device, read-only.
 *   temperature: finite, >= 0.  0 is greedy decoding: p_j and q_j are one-hot
 *     at the row's first largest logit (the T -> 0 limit), so a position is
 *     accepted iff D_j is the target argmax (gated: NULL iff D_j is not the
 *     draft argmax), alpha is 1 or 0, the stop row emits its target argmax,
 *     no uniform is drawn, and row_stats holds (max L, max L).  A positive
 *     temperature is applied as the fp32 factor log2(e) / T; a temperature so
 *     small that a row's largest logit, scaled, overflows fp32
 *     (|max L| log2(e) / T above 3.4e38: T below about 1e-37 when that logit
 *     has size 30) makes the row's normaliser non-finite, and the sequence
 *     fails closed as invalid input.
 *   gate_mode / threshold: the default mode and threshold of every sequence;
 *     threshold must lie in (0, 1] when gate_mode is SV_GATED_MU.
 *   gate_mode_per_seq [B] uint8 (0 plain, 1 gated) and threshold_per_seq [B]
 *     float: optional device arrays overriding the defaults (NULL = use them).
 *   seed / Philox key; uniforms are keyed on the sequence index b.
 *   accepted_len [B] int32, tokens [B, k+1] int32, accept_prob [B, k] float:
 *     required device outputs.  flags [B, k] int8 and counters [8] uint64
 *     (accumulated, see SV_CNT_*): optional device outputs (NULL = skip).
 *   cuda_stream: a cudaStream_t (NULL = legacy default stream).
 * B = 0 is a no-op.  Asynchronous: returns once the work is enqueued. */
sv_status spec_verify_run(spec_verify_t h,
                          const void* target_logits, sv_dtype tdt,
                          const void* draft_logits, sv_dtype ddt,
                          const int32_t* draft_tokens,
                          int B, float temperature,
                          sv_gate gate_mode, float threshold,
                          const uint8_t* gate_mode_per_seq,
                          const float* threshold_per_seq,
                          uint64_t seed,
                          int32_t* accepted_len, int32_t* tokens, float* accept_prob,
                          int8_t* flags, uint64_t* counters,
                          void* cuda_stream);

/* spec_verify_run with three extras:
 *   seq_offset: the Philox counter uses s = seq_offset + b, so a batch split
 *     across calls (or GPUs) draws the same uniforms as the whole batch.
 *   u_accept [B, k] / u_residual [B]: optional device arrays of explicit
 *     uniforms in [0, 1) that replace the Philox draws u0 and u1 (a test hook
 *     for probing decisions away from their boundaries); NULL = Philox.
 *   row_stats [B, 2k+1, 2] float: optional device output, (max, log-sum-exp)
 *     of L/T for target rows 0..k then draft rows 0..k-1 of each sequence. */
sv_status spec_verify_run_ex(spec_verify_t h,
                             const void* target_logits, sv_dtype tdt,
                             const void* draft_logits, sv_dtype ddt,
                             const int32_t* draft_tokens,
                             int B, float temperature,
                             sv_gate gate_mode, float threshold,
                             const uint8_t* gate_mode_per_seq,
                             const float* threshold_per_seq,
                             uint64_t seed, uint64_t seq_offset,
                             const float* u_accept, const float* u_residual,
                             int32_t* accepted_len, int32_t* tokens, float* accept_prob,
                             int8_t* flags, uint64_t* counters, float* row_stats,
                             void* cuda_stream);

/* Closed-form acceptance of every draft position (mlxcel PR #992, "The
 * acceptance ceiling"): for a draft drawn from q_j,
 *   min_sum [B, k]  = sum_x min(p_j(x), mu_j(x)): the acceptance probability of
 *                     modified rejection sampling, i.e. the mean of accept_prob
 *                     over D_j ~ q_j (plain mode: 1 - TV(p_j, q_j), the
 *                     ceiling of every distribution-preserving rule);
 *   pq_sum [B, k]   = sum_x p_j(x) q_j(x): the sampler-match rule's;
 *   argmax_q [B, k] = q_j(argmax p_j): the argmax rule's (first largest p_j).
 * Device float outputs, each optional (NULL skips it; all NULL: nothing runs).
 * Inputs as spec_verify_run; mu_j follows each sequence's gate and the
 * handle's gate policy, whose cumulative floor reads the drafted prefix
 * draft_tokens[b, 0..j-1] (otherwise draft_tokens is not used).  Temperature 0
 * gives the one-hot values (1 or 0).  A position whose rows p_j or q_j are
 * invalid (a NaN or +inf logit, or every logit -inf) -- or, with a cumulative
 * floor, one behind an invalid earlier draft row or an out-of-range drafted
 * token -- gets NaN, as does every position of a gated sequence whose own
 * threshold is outside (0, 1] with no schedule.  Cost: the stream pass over
 * every row, then a second read of each pair (p_j, q_j), j < k.  Host errors
 * and asynchrony as spec_verify_run; it shares the handle's workspace, so it
 * must not overlap a run on the same handle. */
sv_status spec_verify_diagnostics(spec_verify_t h,
                                  const void* target_logits, sv_dtype tdt,
                                  const void* draft_logits, sv_dtype ddt,
                                  const int32_t* draft_tokens,
                                  int B, float temperature,
                                  sv_gate gate_mode, float threshold,
                                  const uint8_t* gate_mode_per_seq,
                                  const float* threshold_per_seq,
                                  float* min_sum, float* pq_sum, float* argmax_q,
                                  void* cuda_stream);

/* spec_verify_run with HOST buffers for every input and output (same shapes;
 * gate_mode_per_seq / threshold_per_seq / flags / counters optional, host).
 * Copies the inputs to device staging buffers, verifies, copies the outputs
 * back and synchronises the stream before returning; counters are overwritten,
 * not accumulated.  The staging buffers (sized for max_B) are allocated on the
 * first call and kept by the handle.  Pinned host memory makes the copies
 * asynchronous DMA; pageable memory works but is slower.  Logits in
 * page-locked host memory that the device can address are not copied when
 * the call reads them about once -- no sampler filters, and no dense residual
 * pass (temperature 0, or every row gated with scalar settings or the
 * handle's schedule on the candidate fast path): the kernels then read them
 * in place over the host link, and the caller must keep them unchanged until
 * the call returns (it returns after the stream has synchronised). */
sv_status spec_verify_run_host(spec_verify_t h,
                               const void* target_logits, sv_dtype tdt,
                               const void* draft_logits, sv_dtype ddt,
                               const int32_t* draft_tokens,
                               int B, float temperature,
                               sv_gate gate_mode, float threshold,
                               const uint8_t* gate_mode_per_seq,
                               const float* threshold_per_seq,
                               uint64_t seed,
                               int32_t* accepted_len, int32_t* tokens, float* accept_prob,
                               int8_t* flags, uint64_t* counters,
                               void* cuda_stream);

/* Gate policy of the gated sequences of every later call on this handle
 * (regolith audit "rank-1 moce and step-aware speculative retention", section
 * "schedule behavior"):
 *   schedule [n_schedule] host floats, each finite and in [0, 1], with
 *     1 <= n_schedule <= SV_MAX_K; or NULL with n_schedule = 0 for none.
 *     Step j uses schedule[min(j, n_schedule - 1)] (the last entry repeats)
 *     IN PLACE OF the sequence's threshold, which is then neither used nor
 *     checked; 0 removes the per-step floor at that step.
 *   min_cum: finite, in [0, 1].  When positive, step j also requires the
 *     drafted prefix's product of draft probabilities to stay at or above it:
 *     prod_{i<j} q_i(D_i) * q_j(x) >= min_cum (reset to 1 for every sequence
 *     and call).  0 disables this floor.
 * Both floors must hold (logical and); equality passes.  A failed gate is the
 * explicit NULL row as before, and mu_j keeps q_j on every token x the same
 * predicate admits at step j, so the output law stays p.  Temperature 0 uses
 * the same predicate on one-hot q.  The host copies the schedule; later calls
 * carry the policy in their launch arguments, so calls already enqueued keep
 * the policy they were issued with.  Default: no schedule, min_cum = 0.
 * Returns SV_EINVAL for a NULL handle or a malformed policy, and then leaves
 * the previous policy in place.  spec_verify_run_noalloc has no handle and
 * always runs without a policy. */
sv_status spec_verify_set_gate_policy(spec_verify_t h, const float* schedule, int n_schedule,
                                      float min_cum);

/* Sampler filters of the target rows (p) and the draft rows (q) of every later
 * call on this handle: mlxcel PR #992, "What changed" -- the effective
 * distribution is the sampler's own chain: temperature, top-k, top-p, min-p,
 * then the softmax of the survivors; top_k == 1 is greedy.
 *   top_k >= 0: keep the tokens whose logit is at least the k-th largest (ties
 *     at the boundary kept); 0 = off; 1 = only the first largest logit.
 *   top_p in (0, 1]: on the top-k survivors renormalised, in decreasing
 *     probability, keep the shortest prefix whose mass reaches top_p, plus the
 *     tokens tied with its last one; 1 = off.
 *   min_p in [0, 1]: keep p >= min_p * max p; 0 = off.
 * With any filter on (and temperature > 0) a verifying call first finds each
 * row's kept set (a logit threshold, or the kept index of a top_k = 1 row)
 * into a buffer of the handle (max_B * (2k+1) * (16 + ceil(V / 2048) * 132)
 * bytes, allocated on the first filtered call -- make that call outside any
 * stream capture; SV_ENOMEM if it fails).  When every filtered side holds
 * bf16 logits and none has top_k = 1, one read of each row decides it (a
 * histogram over the bf16 values); otherwise a statistics pass over the
 * logits runs first, and for a top-k filter (2 <= top_k <= ceil(V / 2048)
 * <= 512) a gathering pass collects each row's candidates chunk by chunk.
 * Its verifying kernels then read every logit outside a row's kept set as
 * -inf (a NaN is kept, so the row stays invalid): 3 to 7 launches instead of
 * 2 and two to four reads of the logits.  row_stats then describe the filtered
 * rows.  spec_verify_diagnostics applies the same filters the same way (its
 * kernels read every logit outside a row's kept set as -inf; the launches of
 * the kept sets come in front of its own).  Decisions of top-p and min-p sit
 * on fp32 arithmetic (the top-p masses are summed as integers, so they do not
 * depend on the order of the additions).  Default: all off.  Returns SV_EINVAL (filters unchanged) for
 * a NULL handle or a value outside its range. */
sv_status spec_verify_set_filters(spec_verify_t h, int top_k_target, float top_p_target,
                                  float min_p_target, int top_k_draft, float top_p_draft,
                                  float min_p_draft);

/* Kernel launches of a verifying call with sampler filters on (temperature > 0),
 * at most: 7 with a gathered top-k filter, 4 otherwise; 3 when every filtered
 * side holds bf16 logits and none has top_k = 1. */
int spec_verify_launches_per_filtered_run(void);

/* Release the handle and its device memory (NULL is a no-op).  Synchronises
 * the handle's device first. */
sv_status spec_verify_free(spec_verify_t h);

/* Static, never-NULL description of a status code. */
const char* spec_verify_status_string(sv_status s);

/* Number of kernel launches one spec_verify_run call makes (for launch
 * accounting in benchmarks). */
int spec_verify_launches_per_run(void);

/* Timing aid: the next spec_verify_run* call on this handle records
 * ev_before / ev_after (cudaEvent_t values created by the caller on the
 * handle's device) on its stream immediately before and after its first
 * launch, the bandwidth-bound stream pass, so that pass can be timed alone.
 * One-shot: the marks are cleared by that call.  Passing NULL for both clears
 * pending marks.  Returns SV_EINVAL for a NULL handle or only one NULL event. */
sv_status spec_verify_mark_next(spec_verify_t h, void* ev_before, void* ev_after);

/* ---------------------------------------------------------------------------
 * Allocation-free entry point.  The pages have no counterpart of this call; it
 * exists for callers that may not allocate device memory where they verify --
 * a serving loop whose device memory is reserved up front by its own caching
 * allocator, or one that must not call cudaMalloc / cudaFree between decode
 * steps because they synchronise the device.  spec_verify_init allocates the
 * handle's workspace, so such callers cannot create a handle at that point.
 *
 * spec_verify_run_noalloc verifies exactly like spec_verify_run (same kernels,
 * same arguments plus k and V, same results bit for bit) on the CURRENT CUDA
 * device.  Its workspace is a static device buffer of SV_NOALLOC_SCRATCH_BYTES
 * compiled into the library; it calls no allocating CUDA or library function.
 * Sizes beyond the buffer return SV_EUNSUPPORTED with nothing launched:
 *   B * k * ceil(V / 2048) * 4 <= SV_NOALLOC_MAX_CAND_SLOTS
 *   B * k                      <= SV_NOALLOC_MAX_ROWS
 *   B * (2k+1) * ceil(V / 2048) * 8 + B * (2k+1) * 4 (each rounded up to 256)
 *                              <= SV_NOALLOC_STATS_BYTES
 * (B = 64, k = 5, V = 128256 uses 80,640 slots and 0.36 MiB of statistics;
 * B = 256, k = 8, V = 151936 does not fit.)
 *
 * Set-up: the first call on a device (per process) looks up the buffer's
 * device address, sets the kernels' attributes and fills the candidate slots
 * with their empty marker (a synchronous memset).  Make that first call
 * outside any stream capture.  What must hold before every call: every
 * candidate slot empty (all bits set) and every row-overflow flag zero; set-up
 * establishes it and every call that completes restores it.  A call that
 * returns SV_ECUDA may have launched its first kernel and not its second, so
 * it marks the device's set-up as undone: the next call on that device does
 * the set-up again (after a cudaDeviceSynchronize, so outside any capture).
 * A device reset (cudaDeviceReset) reloads the library's device code and so
 * refills the buffer with zeros, which the library cannot detect: after a
 * reset, reload the library (or restart the process) before calling this
 * entry point again.
 *
 * Concurrency: all calls on a device share the one buffer, so they must not
 * overlap -- issue them on one stream or otherwise order them.  Two calls in
 * flight at once race on the buffer and produce wrong results.
 *
 * Other errors as spec_verify_run; SV_EINVAL also for k < 1 or V < 1. */
#define SV_NOALLOC_SCRATCH_BYTES (8u << 20)
#define SV_NOALLOC_MAX_CAND_SLOTS (1u << 19)                 /* 4 MiB of 8-byte slots */
#define SV_NOALLOC_MAX_ROWS (1u << 14)                       /* 64 KiB of flags */
#define SV_NOALLOC_STATS_BYTES (SV_NOALLOC_SCRATCH_BYTES - (4u << 20) - (64u << 10))
sv_status spec_verify_run_noalloc(const void* target_logits, sv_dtype tdt,
                                  const void* draft_logits, sv_dtype ddt,
                                  const int32_t* draft_tokens,
                                  int B, int k, int V, float temperature,
                                  sv_gate gate_mode, float threshold,
                                  const uint8_t* gate_mode_per_seq,
                                  const float* threshold_per_seq,
                                  uint64_t seed,
                                  int32_t* accepted_len, int32_t* tokens, float* accept_prob,
                                  int8_t* flags, uint64_t* counters,
                                  void* cuda_stream);

#ifdef __cplusplus
}
#endif
#endif
