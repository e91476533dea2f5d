/*
 * spec_verify_oracle.h -- plain CPU oracle for batched speculative-decoding
 * verification (modified rejection sampling, plain and mu/NULL-gated modes).
 *
 * TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only the test suite,
 * the smoke check and the CPU-baseline leg of the benchmark load this code.
 * It shares no source with the CUDA library: its Philox generator, softmax,
 * decision rule and inverse-CDF sampler are written out here independently,
 * in double precision, one sequence at a time, with no blocking or fusion.
 *
 * Sources the arithmetic follows (web pages, cited by title and section):
 *   [S]  Strata PR #3416 "[Engine] Preserve target probabilities in gated
 *        MTP" -- sections "Problem and result" (the worked example and the
 *        biased original gate) and "Approach" (retained measure mu, explicit
 *        NULL row, min(1, p(D)/mu(D)) acceptance, residual (p - mu)+,
 *        ordinary bonus sample).
 *   [M]  mlxcel PR #992 "modified rejection sampling" -- sections "The
 *        acceptance ceiling" (sum min(p,q) = 1 - TV, sampler-match sum p*q,
 *        argmax rule), "What changed" (accept test p(t) > 0 && u*q(t) <= p(t),
 *        residual normalise(relu(p - q)), fp32 effective distribution) and
 *        "Two metric corrections" (a chain stops at its first rejection).
 *   [R]  regolith audit "rank-1 moce and step-aware speculative retention",
 *        section "schedule behavior" (equality passes the gate; a failed gate
 *        ends the contiguous prefix; per-step threshold schedules whose last
 *        entry repeats; the cumulative prefix-product floor; both floors
 *        composed by logical and).
 *   [P]  J. K. Salmon, M. A. Moraes, R. O. Dror, D. E. Shaw, "Parallel random
 *        numbers: as easy as 1, 2, 3", SC'11 -- the Philox4x32 bijection.
 *
 * Readings where the pages are silent are listed beside each function.
 */
#ifndef SPEC_VERIFY_ORACLE_H
#define SPEC_VERIFY_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* largest k the oracle accepts */
#define ORACLE_MAX_K 64

/* element types of the logits arrays */
enum { ORACLE_F32 = 0, ORACLE_BF16 = 1 };

/* decision rules.  ORACLE_RULE_MU is the method; the others are controls
 * (known-correct or known-wrong rules) that the statistical tests need. */
enum {
  ORACLE_RULE_MU = 0,            /* plain MRS (gate off) / mu-NULL rule (gate on) */
  ORACLE_RULE_ORIGINAL_GATE = 1, /* [S] biased: unfiltered q, failed gate samples p */
  ORACLE_RULE_SAMPLER_MATCH = 2, /* [M] lossless: accept iff a fresh p draw equals D */
  ORACLE_RULE_ARGMAX = 3,        /* [M] biased: accept iff D == argmax p, emit argmax */
  ORACLE_RULE_RESAMPLE_P = 4,    /* [M] biased: on rejection sample p, not the residual */
  ORACLE_RULE_RENORM_MU = 5,     /* plausible mistake: mu renormalised over admitted set */
  ORACLE_RULE_RESIDUAL_Q = 6,    /* plausible mistake: gated residual uses (p - q)+ */
  ORACLE_RULE_MU_STEP_ONLY = 7   /* plausible mistake: mu ignores the cumulative floor */
};

/* per-position flags (same values as the CUDA library's outputs) */
enum {
  ORACLE_FLAG_UNREACHED = 0,
  ORACLE_FLAG_ACCEPT = 1,
  ORACLE_FLAG_REJECT = 2,
  ORACLE_FLAG_NULL = 3,
  ORACLE_FLAG_INVALID = 4
};

/* Philox4x32 with 10 rounds [P]: out = bijection_key(ctr). */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]);

/* U(seed, seq, pos, draw): key = (seed lo32, seed hi32), counter =
 * (seq lo32, pos, draw, seq hi32); u = (out[0] >> 8) * 2^-24, in [0, 1). */
double oracle_uniform(uint64_t seed, uint64_t seq, uint32_t pos, uint32_t draw);

/* Temperature softmax of one row of V logits (element type dt):
 * p[v] = exp(L[v]/T - m) / sum_w exp(L[w]/T - m), m = max_v L[v]/T.
 * T = 0 is greedy decoding: p is one-hot at the first largest logit, and
 * *row_max = *row_lse = max_v L[v].
 * Writes p (may be NULL), *row_max = m and *row_lse = m + ln(sum).
 * Returns 0, or 1 when the row is invalid (a NaN or +inf logit, or every
 * logit -inf). */
int oracle_softmax_row(const void* logits, int dt, int64_t V, double T,
                       double* p, double* row_max, double* row_lse);

/* Inverse-CDF pick over the weights r[0..V): the smallest v whose inclusive
 * prefix sum exceeds u * Z (Z = sum r); if rounding leaves none, the last v
 * with r[v] > 0; -1 if every weight is zero.  *margin (may be NULL) receives
 * the distance of u to the two edges of the chosen interval, in units of Z. */
int64_t oracle_inverse_cdf(const double* r, int64_t V, double u, double* margin);

/*
 * Verify a batch.  Shapes (row-major, V innermost):
 *   Lt [B, k+1, V] (dt tdt), Ld [B, k, V] (dt ddt), D [B, k] int32.
 *   gate[B]   0 = plain, 1 = mu/NULL gated;  tau[B] thresholds (gated rows).
 *   u0 [B, k], u1 [B]: explicit uniforms, or NULL to draw them from Philox:
 *     u0[b,j] = U(seed, seq_offset + b, j, 0), u1[b] = U(seed, seq_offset+b, j*, 1).
 * Outputs (all host):
 *   accepted_len[B] (-1 for an invalid sequence), tokens[B, k+1] (-1 padded),
 *   alpha[B, k] (acceptance probability of every position, also past j*),
 *   flags[B, k], and optionally row_stats[B, 2k+1, 2] = (max, lse) of L/T for
 *   target rows 0..k then draft rows 0..k-1, margin[B] = the smallest distance
 *   of a used uniform (or of q(D), or of any q on the residual row) to its
 *   decision boundary, margin_pick[B] = the part of that minimum that comes
 *   from the residual / bonus pick (its interval edges and, in gated mode, the
 *   gate membership of the residual row's tokens), degenerate[B] = 1 when the
 *   residual had zero mass.
 * T = 0 runs the same rule on the one-hot (greedy) distributions of
 * oracle_softmax_row.
 * nthreads >= 1 threads split the sequences.  Returns 0, or 1 on bad args.
 */
int oracle_verify(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                  int B, int k, int64_t V, double T,
                  const uint8_t* gate, const double* tau,
                  uint64_t seed, uint64_t seq_offset,
                  const double* u0, const double* u1, int rule,
                  int32_t* accepted_len, int32_t* tokens, double* alpha, int8_t* flags,
                  double* row_stats, double* margin, double* margin_pick,
                  int32_t* degenerate, int nthreads);

/*
 * oracle_verify with the gate policy of [R] "schedule behavior" for the gated
 * sequences (gate[b] = 1):
 *   tau_sched [n_sched] (n_sched >= 1, or NULL): per-step thresholds that
 *     replace tau[b]; step j uses tau_sched[min(j, n_sched - 1)] (the last
 *     entry repeats).  Entries may be 0 (no per-step floor at that step).
 *   min_cum in [0, 1]: the cumulative floor; when positive, step j also needs
 *     prod_{i<j} q_i(D_i) * q_j(x) >= min_cum (products in double, reset to 1
 *     for every sequence).  0 disables it.
 * Both floors must hold (logical and); equality passes.  The retained measure
 * mu_j keeps q_j on every token x that the same predicate admits at step j
 * (with the drafted prefix's product), so a failed gate is still an explicit
 * NULL row and the residual is (p_j - mu_j)+.  margin also covers the
 * cumulative decision, |product - min_cum|.  Returns 1 on bad args.
 */
int oracle_verify_policy(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                         int B, int k, int64_t V, double T,
                         const uint8_t* gate, const double* tau,
                         const double* tau_sched, int n_sched, double min_cum,
                         uint64_t seed, uint64_t seq_offset,
                         const double* u0, const double* u1, int rule,
                         int32_t* accepted_len, int32_t* tokens, double* alpha, int8_t* flags,
                         double* row_stats, double* margin, double* margin_pick,
                         int32_t* degenerate, int nthreads);

/*
 * The sampler's filter chain on one row [M] "What changed" (temperature,
 * top-k, top-p, min-p, then the softmax; top_k == 1 is greedy):
 *   top_k >= 1: keep the tokens whose logit is at least the k-th largest
 *     (ties at the boundary kept); 0 = off; 1 = one-hot at the first largest.
 *   top_p in (0, 1): on the top-k survivors, renormalised, in decreasing
 *     probability, keep the shortest prefix whose mass reaches top_p, plus
 *     every token tied with its last one; 1 = off.
 *   min_p in (0, 1]: keep p >= min_p * max p; 0 = off.
 * p holds the row's temperature softmax (oracle_softmax_row) on entry and the
 * renormalised filtered distribution on exit; T = 0 rows are left one-hot.
 * *margin (may be NULL): the smallest distance of a top-p decision (in units
 * of the top-k mass) or a min-p decision (in units of p / max p) to its
 * boundary.  *kept (may be NULL): the unfiltered probability mass of the
 * survivors.  Returns 0, or 1 when memory runs out.
 */
int oracle_filtered_row(const void* logits, int dt, int64_t V, double T, int top_k, double top_p,
                        double min_p, double* p, double* margin, double* kept);

/*
 * oracle_verify_policy with sampler filters: top_k[2], top_p[2], min_p[2]
 * (index 0 the target rows, 1 the draft rows; all three NULL for none) turn
 * every p_j and q_j into its filtered distribution (oracle_filtered_row)
 * before the rule runs; row_stats then describe the filtered rows (max and
 * log-sum-exp of L/T over the survivors); margin also covers the filter
 * decisions of every row of the sequence, and margin_filter[B] (may be NULL)
 * reports that part alone.
 */
int oracle_verify_filtered(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                           int B, int k, int64_t V, double T,
                           const uint8_t* gate, const double* tau,
                           const double* tau_sched, int n_sched, double min_cum,
                           const int* top_k, const double* top_p, const double* min_p,
                           uint64_t seed, uint64_t seq_offset,
                           const double* u0, const double* u1, int rule,
                           int32_t* accepted_len, int32_t* tokens, double* alpha, int8_t* flags,
                           double* row_stats, double* margin, double* margin_pick,
                           double* margin_filter, int32_t* degenerate, int nthreads);

/*
 * Closed-form acceptance of every draft position [M] "The acceptance ceiling":
 * for a draft drawn from q_j,
 *   min_sum[b, j]  = sum_x min(p_j(x), mu_j(x))  -- modified rejection sampling
 *                    (plain mode mu = q: the maximal-coupling bound 1 - TV);
 *   pq_sum[b, j]   = sum_x p_j(x) q_j(x)         -- sampler-match;
 *   argmax_q[b, j] = q_j(argmax p_j)             -- the argmax rule (first
 *                    largest p_j).
 * mu_j follows the sequence's gate and the policy of oracle_verify_policy
 * (the cumulative floor uses the drafted prefix D_0..D_{j-1}).  Outputs
 * [B, k] (each may be NULL); margin[B] (may be NULL) = the smallest distance
 * of any q_j(x) of a gated sequence to its gate boundaries.  A position whose
 * rows p_j or q_j are invalid (NaN or +inf logit, all -inf), or -- with a
 * cumulative floor -- behind an invalid earlier draft row or drafted token,
 * gets NaN; so does every position of a gated sequence with a threshold
 * outside (0, 1] and no schedule.  top_k / top_p / min_p ([2] each, or NULL)
 * apply the sampler filters of oracle_verify_filtered first; margin then also
 * covers their decisions.  Returns 1 on bad args.
 */
int oracle_diagnostics(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                       int B, int k, int64_t V, double T,
                       const uint8_t* gate, const double* tau,
                       const double* tau_sched, int n_sched, double min_cum,
                       const int* top_k, const double* top_p, const double* min_p,
                       double* min_sum, double* pq_sum, double* argmax_q, double* margin,
                       int nthreads);

/*
 * The interval of token v in the distribution that the stop row of one
 * sequence samples from when its chain stops at position j (j = k: the bonus
 * row p_k; else the residual (p_j - mu_j)+ with mu_j the retained measure of
 * the gate at step j behind the drafted prefix, or p_j when the residual has
 * no mass) -- for judging picks made in lower precision near a boundary.
 * Lt [k+1, V], Ld [k, V] and D [k] are that sequence's rows and drafted
 * tokens; gated / tau its gate; tau_sched, n_sched, min_cum and the filters
 * as in oracle_verify_filtered.  With r those weights, Z = sum r and C the
 * inclusive prefix sums in token order: *weight = r(v) / Z, *lo = C(v-1) / Z,
 * *hi = C(v) / Z; *gate_marg (may be NULL) = the closest q_j(x) of a gated
 * stop row to a gate boundary (INFINITY otherwise).  Returns 0, or 1 on bad
 * arguments or an invalid row.
 */
int oracle_pick_interval(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                         int k, int64_t V, double T, int gated, double tau,
                         const double* tau_sched, int n_sched, double min_cum,
                         const int* top_k, const double* top_p, const double* min_p,
                         int j, int64_t v, double* weight, double* lo, double* hi,
                         double* gate_marg);

#ifdef __cplusplus
}
#endif
#endif
