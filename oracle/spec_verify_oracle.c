/*
 * spec_verify_oracle.c -- plain CPU oracle (fp64) for batched speculative-
 * decoding verification.  TEST INFRASTRUCTURE: see spec_verify_oracle.h for
 * the contract, the sources and who may call it.  Every step is written out
 * the way the pages state it, one sequence at a time, with no fusion.
 */
#include "spec_verify_oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ---------------------------------------------------------------- Philox */

/* Philox4x32-10 [P]: each round multiplies words 0 and 2 by the two round
 * multipliers, mixes the high halves with words 1 and 3 and the key, and the
 * key advances by the two Weyl constants between rounds. */
void oracle_philox4x32_10(const uint32_t ctr[4], const uint32_t key[2], uint32_t out[4]) {
  const uint32_t mult0 = 0xD2511F53u, mult1 = 0xCD9E8D57u;
  const uint32_t weyl0 = 0x9E3779B9u, weyl1 = 0xBB67AE85u;
  uint32_t x0 = ctr[0], x1 = ctr[1], x2 = ctr[2], x3 = ctr[3];
  uint32_t k0 = key[0], k1 = key[1];
  for (int round = 0; round < 10; ++round) {
    if (round > 0) {
      k0 += weyl0;
      k1 += weyl1;
    }
    uint64_t prod0 = (uint64_t)mult0 * (uint64_t)x0;
    uint64_t prod1 = (uint64_t)mult1 * (uint64_t)x2;
    uint32_t hi0 = (uint32_t)(prod0 >> 32), lo0 = (uint32_t)prod0;
    uint32_t hi1 = (uint32_t)(prod1 >> 32), lo1 = (uint32_t)prod1;
    uint32_t y0 = hi1 ^ x1 ^ k0;
    uint32_t y1 = lo1;
    uint32_t y2 = hi0 ^ x3 ^ k1;
    uint32_t y3 = lo0;
    x0 = y0; x1 = y1; x2 = y2; x3 = y3;
  }
  out[0] = x0; out[1] = x1; out[2] = x2; out[3] = x3;
}

double oracle_uniform(uint64_t seed, uint64_t seq, uint32_t pos, uint32_t draw) {
  uint32_t key[2] = {(uint32_t)seed, (uint32_t)(seed >> 32)};
  uint32_t ctr[4] = {(uint32_t)seq, pos, draw, (uint32_t)(seq >> 32)};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  /* 24 high bits, scaled by 2^-24: exact in float and double */
  return (double)(out[0] >> 8) * (1.0 / 16777216.0);
}

/* -------------------------------------------------------------- softmax */

static double logit_at(const void* L, int dt, int64_t i) {
  if (dt == ORACLE_F32) return (double)((const float*)L)[i];
  uint32_t bits = (uint32_t)((const uint16_t*)L)[i] << 16; /* bf16 -> f32 is exact */
  float f;
  memcpy(&f, &bits, sizeof f);
  return (double)f;
}

/* p = softmax(L / T) [M "What changed": the effective distribution is the
 * temperature softmax over the full vocabulary].  Reading: -inf logits are
 * allowed (p = 0); NaN, +inf or an all -inf row make the row invalid, the
 * "non-finite observations fail closed" rule of [R]. */
int oracle_softmax_row(const void* logits, int dt, int64_t V, double T,
                       double* p, double* row_max, double* row_lse) {
  if (T == 0.0) {
    /* Reading for temperature 0 (greedy decoding): the distribution is the
     * T -> 0 limit of the temperature softmax, one-hot at the largest logit;
     * among equal largest logits, the first (smallest index).  Reported row
     * statistics: (max L, max L), the limit of T * (max, lse) of L / T. */
    double m = -INFINITY;
    int64_t best = -1;
    int bad = 0;
    for (int64_t v = 0; v < V; ++v) {
      double x = logit_at(logits, dt, v);
      if (isnan(x) || (isinf(x) && x > 0)) bad = 1;
      if (x > m) {
        m = x;
        best = v;
      }
    }
    if (row_max) *row_max = m;
    if (bad || best < 0) {
      if (row_lse) *row_lse = NAN;
      return 1;
    }
    if (p) {
      for (int64_t v = 0; v < V; ++v) p[v] = 0.0;
      p[best] = 1.0;
    }
    if (row_lse) *row_lse = m;
    return 0;
  }
  double m = -INFINITY;
  int bad = 0;
  for (int64_t v = 0; v < V; ++v) {
    double x = logit_at(logits, dt, v);
    if (isnan(x) || (isinf(x) && x > 0)) bad = 1;
    double xs = x / T;
    if (xs > m) m = xs;
  }
  if (row_max) *row_max = m;
  if (bad || m == -INFINITY) {
    if (row_lse) *row_lse = NAN;
    return 1;
  }
  double s = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    double e = exp(logit_at(logits, dt, v) / T - m);
    if (p) p[v] = e;
    s += e;
  }
  if (p)
    for (int64_t v = 0; v < V; ++v) p[v] /= s;
  if (row_lse) *row_lse = m + log(s);
  return 0;
}

/* ------------------------------------------------------------ filters */

typedef struct {
  double x;   /* logit */
  int64_t v;  /* token */
} ranked_t;

/* decreasing logit, then increasing token */
static int ranked_cmp(const void* a, const void* b) {
  const ranked_t* ra = (const ranked_t*)a;
  const ranked_t* rb = (const ranked_t*)b;
  if (ra->x > rb->x) return -1;
  if (ra->x < rb->x) return 1;
  return ra->v < rb->v ? -1 : (ra->v > rb->v ? 1 : 0);
}

/* The sampler's filter chain after the temperature [M "What changed": the
 * sampler's own chain -- temperature, top-k, top-p, min-p -- whose softmax is
 * the effective distribution; a top_k of 1 is greedy].  p holds the row's
 * temperature softmax on entry and the filtered, renormalised distribution on
 * exit.  Readings: each filter keeps every token tied with its boundary
 * token; top-p works on the top-k survivors renormalised, in decreasing
 * probability, keeping the shortest prefix whose mass reaches top_p; min-p
 * keeps p >= min_p * max p.  *margin: the smallest relative distance of a
 * top-p or min-p decision to its boundary (top-k compares logits exactly). */
int oracle_filtered_row(const void* logits, int dt, int64_t V, double T, int top_k, double top_p,
                        double min_p, double* p, double* margin, double* kept) {
  double marg = INFINITY;
  const int use_k = top_k >= 1 && (int64_t)top_k < V;
  const int use_p = top_p > 0.0 && top_p < 1.0;
  const int use_m = min_p > 0.0;
  if (margin) *margin = marg;
  if (kept) *kept = 1.0;
  if (T == 0.0 || !(use_k || use_p || use_m)) return 0;  /* greedy rows are one-hot already */
  ranked_t* rk = (ranked_t*)malloc((size_t)V * sizeof(ranked_t));
  unsigned char* keep = (unsigned char*)malloc((size_t)V);
  if (!rk || !keep) {
    free(rk); free(keep);
    return 1;
  }
  for (int64_t v = 0; v < V; ++v) {
    rk[v].x = logit_at(logits, dt, v);
    rk[v].v = v;
    keep[v] = 1;
  }
  qsort(rk, (size_t)V, sizeof(ranked_t), ranked_cmp);
  if (top_k == 1) {
    /* greedy: one-hot at the first largest logit */
    if (kept) *kept = p[rk[0].v];
    for (int64_t v = 0; v < V; ++v) p[v] = 0.0;
    p[rk[0].v] = 1.0;
    free(rk); free(keep);
    return 0;
  }
  if (use_k) {
    const double xk = rk[top_k - 1].x;
    for (int64_t i = 0; i < V; ++i) keep[rk[i].v] = rk[i].x >= xk;
  }
  if (use_p) {
    double Sk = 0.0;
    for (int64_t i = 0; i < V; ++i)
      if (keep[rk[i].v]) Sk += p[rk[i].v];
    const double target = top_p * Sk;
    double c = 0.0, before = 0.0;
    int64_t m = -1;
    for (int64_t i = 0; i < V; ++i) {
      if (!keep[rk[i].v]) continue;
      before = c;
      c += p[rk[i].v];
      if (c >= target) {
        m = i;
        break;
      }
    }
    if (m >= 0) {
      marg = fmin(marg, fmin(target - before, c - target) / Sk);
      const double xm = rk[m].x;
      for (int64_t i = 0; i < V; ++i)
        if (rk[i].x < xm) keep[rk[i].v] = 0;
    }
  }
  if (use_m) {
    const double xmax = rk[0].x;
    for (int64_t i = 0; i < V; ++i) {
      if (!keep[rk[i].v]) continue;
      const double ratio = exp((rk[i].x - xmax) / T);  /* p / max p */
      marg = fmin(marg, fabs(ratio - min_p));
      if (!(ratio >= min_p)) keep[rk[i].v] = 0;
    }
  }
  double S = 0.0;
  for (int64_t v = 0; v < V; ++v)
    if (keep[v]) S += p[v];
  for (int64_t v = 0; v < V; ++v) p[v] = keep[v] ? p[v] / S : 0.0;
  free(rk); free(keep);
  if (margin) *margin = marg;
  if (kept) *kept = S;
  return 0;
}

/* ------------------------------------------------------------ sampling */

/* Inverse-CDF pick: the smallest v with prefix(v) > u * Z.  Reading: the
 * strict comparison means a zero-weight token is never picked, so the
 * residual never emits a token with p <= mu ([M] "Where chi-square is
 * blind").  If rounding left no such v, take the last v with weight > 0. */
int64_t oracle_inverse_cdf(const double* r, int64_t V, double u, double* margin) {
  double Z = 0.0;
  for (int64_t v = 0; v < V; ++v) Z += r[v];
  if (!(Z > 0.0)) {
    if (margin) *margin = 0.0;
    return -1;
  }
  double y = u * Z;
  double before = 0.0, upto = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    before = upto;
    upto += r[v];
    if (upto > y) {
      if (margin) *margin = fmin(fabs(u - before / Z), fabs(u - upto / Z));
      return v;
    }
  }
  for (int64_t v = V - 1; v >= 0; --v)
    if (r[v] > 0.0) {
      if (margin) *margin = 0.0;
      return v;
    }
  return -1;
}

static int64_t argmax_first(const double* p, int64_t V) {
  int64_t best = 0;
  for (int64_t v = 1; v < V; ++v)
    if (p[v] > p[best]) best = v;
  return best;
}

/* ------------------------------------------------------ one sequence */

typedef struct {
  const void* Lt; int tdt;
  const void* Ld; int ddt;
  const int32_t* D;
  int B, k;
  int64_t V;
  double T;
  const uint8_t* gate;
  const double* tau;
  uint64_t seed, seq_offset;
  const double* u0;
  const double* u1;
  int rule;
  int32_t* accepted_len; int32_t* tokens; double* alpha; int8_t* flags;
  double* row_stats; double* margin; double* margin_pick; int32_t* degenerate;
  double* margin_filter;  /* the part of margin that comes from the sampler filters */
  const double* tau_sched; int n_sched; /* per-step thresholds (NULL: tau[b] at every step) */
  double min_cum;                       /* cumulative floor (0: no cumulative gate) */
  /* sampler filters of the target [0] and draft [1] rows (NULL: none) */
  const int* top_k; const double* top_p; const double* min_p;
  /* oracle_diagnostics outputs (diagnose = 1 runs diagnose_one instead of verify_one) */
  int diagnose;
  double* diag_min; double* diag_pq; double* diag_argq;
} job_t;

typedef struct {
  double* P;   /* [k+1][V] target distributions p_j */
  double* Q;   /* [k][V]   draft distributions q_j */
  double* mu;  /* [V]      retained measure of one row */
  double* r;   /* [V]      residual weights */
} scratch_t;

static double u_accept(const job_t* J, int b, int j) {
  if (J->u0) return J->u0[(int64_t)b * J->k + j];
  return oracle_uniform(J->seed, J->seq_offset + (uint64_t)b, (uint32_t)j, 0u);
}

static double u_residual(const job_t* J, int b, int jstar) {
  if (J->u1) return J->u1[b];
  return oracle_uniform(J->seed, J->seq_offset + (uint64_t)b, (uint32_t)jstar, 1u);
}

/* The gate threshold of step j of sequence b [R "schedule behavior"]: a
 * supplied schedule overrides the sequence's threshold at every step, its last
 * entry repeating for later steps; without one the sequence's threshold is the
 * floor of every step. */
static double step_threshold(const job_t* J, int b, int j) {
  if (J->tau_sched) return J->tau_sched[j < J->n_sched ? j : J->n_sched - 1];
  return J->tau[b];
}

/* Gate admission of a token with draft probability qv at a step whose
 * threshold is tau_j, behind a drafted prefix whose draft probabilities
 * multiply to cprev [R "schedule behavior"]: the per-step floor qv >= tau_j
 * and, when the cumulative floor is positive, the prefix product including
 * this token, cprev * qv >= min_cum -- both must hold, equality passes.  A zero
 * floor disables the cumulative gate. */
static int admitted(const job_t* J, double tau_j, double cprev, double qv) {
  if (!(qv >= tau_j)) return 0;
  if (J->min_cum > 0.0 && !(cprev * qv >= J->min_cum)) return 0;
  return 1;
}

/* distance of a gate decision to its boundaries: |qv - tau_j| (a zero step
 * floor admits every token whatever the rounding: no boundary) and, with a
 * cumulative floor, |cprev * qv - min_cum| (both in probability units) */
static double gate_margin(const job_t* J, double tau_j, double cprev, double qv) {
  double m = tau_j > 0.0 ? fabs(qv - tau_j) : INFINITY;
  if (J->min_cum > 0.0) m = fmin(m, fabs(cprev * qv - J->min_cum));
  return m;
}

/* mu_j for the rule: plain mode mu = q; gated mode [S "Approach"]: q kept on
 * the tokens the gate would admit at this step (same predicate as the offered
 * token's gate) and NOT renormalised.  The RENORM_MU control renormalises it
 * (the plausible mistake). */
static void retained_measure(const job_t* J, int gated, double tau_j, double cprev, const double* q,
                             double* mu) {
  int64_t V = J->V;
  if (!gated) {
    memcpy(mu, q, (size_t)V * sizeof(double));
    return;
  }
  double kept = 0.0;
  for (int64_t v = 0; v < V; ++v) {
    const int in = J->rule == ORACLE_RULE_MU_STEP_ONLY ? (q[v] >= tau_j) : admitted(J, tau_j, cprev, q[v]);
    mu[v] = in ? q[v] : 0.0;
    kept += mu[v];
  }
  if (J->rule == ORACLE_RULE_RENORM_MU && kept > 0.0)
    for (int64_t v = 0; v < V; ++v) mu[v] /= kept;
}

static void verify_one(const job_t* J, int b, scratch_t* S) {
  const int k = J->k;
  const int64_t V = J->V;
  const int gated = J->gate[b] != 0;
  int32_t* tok = J->tokens + (int64_t)b * (k + 1);
  double* al = J->alpha + (int64_t)b * k;
  int8_t* fl = J->flags + (int64_t)b * k;
  const int32_t* Db = J->D + (int64_t)b * k;
  const int esz_t = J->tdt == ORACLE_BF16 ? 2 : 4, esz_d = J->ddt == ORACLE_BF16 ? 2 : 4;

  /* step 1: the row distributions p_0..p_k and q_0..q_{k-1} (row
   * statistics of the unfiltered L/T), filtered when filters are set */
  int invalid = 0;
  double fmarg = INFINITY;  /* filter decisions near their boundaries */
  for (int j = 0; j <= k; ++j) {
    const char* row = (const char*)J->Lt + ((int64_t)b * (k + 1) + j) * V * esz_t;
    double mx, lse, fm = INFINITY;
    invalid |= oracle_softmax_row(row, J->tdt, V, J->T, S->P + (int64_t)j * V, &mx, &lse);
    double kept = 1.0;
    if (J->top_k && !invalid)
      invalid |= oracle_filtered_row(row, J->tdt, V, J->T, J->top_k[0], J->top_p[0], J->min_p[0],
                                     S->P + (int64_t)j * V, &fm, &kept);
    fmarg = fmin(fmarg, fm);
    lse += log(kept);  /* the statistics of the filtered row (its max is always kept) */
    if (J->row_stats) {
      J->row_stats[((int64_t)b * (2 * k + 1) + j) * 2 + 0] = mx;
      J->row_stats[((int64_t)b * (2 * k + 1) + j) * 2 + 1] = lse;
    }
  }
  for (int j = 0; j < k; ++j) {
    const char* row = (const char*)J->Ld + ((int64_t)b * k + j) * V * esz_d;
    double mx, lse, fm = INFINITY;
    invalid |= oracle_softmax_row(row, J->ddt, V, J->T, S->Q + (int64_t)j * V, &mx, &lse);
    double kept = 1.0;
    if (J->top_k && !invalid)
      invalid |= oracle_filtered_row(row, J->ddt, V, J->T, J->top_k[1], J->top_p[1], J->min_p[1],
                                     S->Q + (int64_t)j * V, &fm, &kept);
    fmarg = fmin(fmarg, fm);
    lse += log(kept);
    if (J->row_stats) {
      J->row_stats[((int64_t)b * (2 * k + 1) + k + 1 + j) * 2 + 0] = mx;
      J->row_stats[((int64_t)b * (2 * k + 1) + k + 1 + j) * 2 + 1] = lse;
    }
  }
  for (int j = 0; j < k; ++j)
    if (Db[j] < 0 || (int64_t)Db[j] >= V) invalid = 1;

  double marg = fmarg;         /* accept tests, gates of tested positions, filters */
  double marg_pick = INFINITY; /* the residual / bonus pick */
  if (J->margin_filter) J->margin_filter[b] = fmarg;
  if (J->degenerate) J->degenerate[b] = 0;
  if (invalid) {
    J->accepted_len[b] = -1;
    for (int j = 0; j <= k; ++j) tok[j] = -1;
    for (int j = 0; j < k; ++j) {
      al[j] = 0.0;
      fl[j] = ORACLE_FLAG_INVALID;
    }
    if (J->margin) J->margin[b] = marg;
    if (J->margin_pick) J->margin_pick[b] = marg_pick;
    return;
  }

  /* the drafted prefix's product of draft probabilities in front of each
   * step, reset to 1 for every verification round [R "schedule behavior"]:
   * cprev[j] = prod_{i<j} q_i(D_i) */
  double cprev[ORACLE_MAX_K + 1];
  cprev[0] = 1.0;
  for (int j = 0; j < k; ++j) cprev[j + 1] = cprev[j] * S->Q[(int64_t)j * V + Db[j]];

  /* step 2: acceptance probability of every position (also past j*).
   * alpha = min(1, p(D)/mu(D)); NULL -> 0; mu(D) = 0 < p(D) -> 1; p(D) = 0 -> 0. */
  for (int j = 0; j < k; ++j) {
    const double pd = S->P[(int64_t)j * V + Db[j]];
    const double qd = S->Q[(int64_t)j * V + Db[j]];
    const double tau = step_threshold(J, b, j);
    const int pass = admitted(J, tau, cprev[j], qd);
    double a;
    if (J->rule == ORACLE_RULE_ORIGINAL_GATE && gated && !pass) {
      a = 0.0; /* failed gate: a target sample, no acceptance */
    } else if (J->rule == ORACLE_RULE_ORIGINAL_GATE || J->rule == ORACLE_RULE_SAMPLER_MATCH ||
               J->rule == ORACLE_RULE_ARGMAX) {
      a = qd > 0.0 ? fmin(1.0, pd / qd) : (pd > 0.0 ? 1.0 : 0.0);
    } else if (gated && !pass) {
      a = 0.0; /* explicit NULL row */
    } else {
      retained_measure(J, gated, tau, cprev[j], S->Q + (int64_t)j * V, S->mu);
      const double md = S->mu[Db[j]];
      a = md > 0.0 ? fmin(1.0, pd / md) : (pd > 0.0 ? 1.0 : 0.0);
    }
    al[j] = a;
    fl[j] = ORACLE_FLAG_UNREACHED;
  }

  /* step 3: walk the chain, stop at the first position not accepted [M] */
  int jstar = k;
  int resid_from_p = 0;   /* stop position samples p itself */
  int resid_argmax = 0;   /* argmax control emits argmax p */
  int64_t direct_token = -1; /* sampler-match control emits its own draw */
  for (int j = 0; j < k; ++j) {
    const double* pj = S->P + (int64_t)j * V;
    const double* qj = S->Q + (int64_t)j * V;
    const int32_t d = Db[j];
    const double u = u_accept(J, b, j);
    const double tau = step_threshold(J, b, j);

    if (J->rule == ORACLE_RULE_SAMPLER_MATCH) {
      /* [M] sampler-match: a fresh target draw; accept iff it equals D */
      double m;
      int64_t x = oracle_inverse_cdf(pj, V, u, &m);
      marg_pick = fmin(marg_pick, m);
      if (x == d) {
        fl[j] = ORACLE_FLAG_ACCEPT;
        continue;
      }
      fl[j] = ORACLE_FLAG_REJECT;
      jstar = j;
      direct_token = x;
      break;
    }
    if (J->rule == ORACLE_RULE_ARGMAX) {
      /* [M] argmax-against-argmax: accept iff D is the target argmax */
      if ((int64_t)d == argmax_first(pj, V)) {
        fl[j] = ORACLE_FLAG_ACCEPT;
        continue;
      }
      fl[j] = ORACLE_FLAG_REJECT;
      jstar = j;
      resid_argmax = 1;
      break;
    }
    if (J->rule == ORACLE_RULE_ORIGINAL_GATE) {
      /* [S "Problem and result"]: the gate filters drafts, acceptance uses
       * the unfiltered q, and a failed gate becomes a plain target sample */
      if (gated) {
        marg = fmin(marg, gate_margin(J, tau, cprev[j], qj[d]));
        if (!admitted(J, tau, cprev[j], qj[d])) {
          fl[j] = ORACLE_FLAG_NULL;
          jstar = j;
          resid_from_p = 1;
          break;
        }
      }
      if (qj[d] > 0.0 && pj[d] < qj[d]) marg = fmin(marg, fabs(u - pj[d] / qj[d]));
      if (pj[d] > 0.0 && u * qj[d] <= pj[d]) {
        fl[j] = ORACLE_FLAG_ACCEPT;
        continue;
      }
      fl[j] = ORACLE_FLAG_REJECT;
      jstar = j;
      break;
    }

    /* the method (and the RESAMPLE_P / RENORM_MU / RESIDUAL_Q controls) */
    if (gated) {
      marg = fmin(marg, gate_margin(J, tau, cprev[j], qj[d]));
      if (!admitted(J, tau, cprev[j], qj[d])) { /* failed gate: explicit NULL row [S "Approach"] */
        fl[j] = ORACLE_FLAG_NULL;
        jstar = j;
        break;
      }
    }
    retained_measure(J, gated, tau, cprev[j], qj, S->mu);
    const double md = S->mu[d];
    if (md > 0.0 && pj[d] < md) marg = fmin(marg, fabs(u - pj[d] / md));
    /* accept test p(D) > 0 && u * mu(D) <= p(D) [M "What changed"] */
    if (pj[d] > 0.0 && u * md <= pj[d]) {
      fl[j] = ORACLE_FLAG_ACCEPT;
      continue;
    }
    fl[j] = ORACLE_FLAG_REJECT;
    jstar = j;
    break;
  }
  if (J->rule == ORACLE_RULE_RESAMPLE_P && jstar < k) resid_from_p = 1;

  /* step 4/5: what the stop row emits */
  int64_t pick;
  if (direct_token >= 0) {
    pick = direct_token;
  } else if (resid_argmax || (J->rule == ORACLE_RULE_ARGMAX && jstar == k)) {
    pick = argmax_first(S->P + (int64_t)jstar * V, V);
  } else {
    const double* pst = S->P + (int64_t)jstar * V;
    const double u = u_residual(J, b, jstar);
    if (jstar == k || resid_from_p) {
      /* ordinary bonus sample of p [S "Approach"] (and the p-resampling controls) */
      memcpy(S->r, pst, (size_t)V * sizeof(double));
    } else {
      /* residual (p - mu)+ [S "Approach"]; plain mode mu = q [M] */
      const double* qst = S->Q + (int64_t)jstar * V;
      const double tau = step_threshold(J, b, jstar);
      if (J->rule == ORACLE_RULE_ORIGINAL_GATE || J->rule == ORACLE_RULE_RESIDUAL_Q) {
        memcpy(S->mu, qst, (size_t)V * sizeof(double));
      } else {
        retained_measure(J, gated, tau, cprev[jstar], qst, S->mu);
      }
      if (gated)
        for (int64_t v = 0; v < V; ++v)
          marg_pick = fmin(marg_pick, gate_margin(J, tau, cprev[jstar], qst[v]));
      double Z = 0.0;
      for (int64_t v = 0; v < V; ++v) {
        double d = pst[v] - S->mu[v];
        S->r[v] = d > 0.0 ? d : 0.0;
        Z += S->r[v];
      }
      if (!(Z > 0.0)) {
        /* reading: a residual with no mass falls back to sampling p */
        memcpy(S->r, pst, (size_t)V * sizeof(double));
        if (J->degenerate) J->degenerate[b] = 1;
      }
    }
    double m;
    pick = oracle_inverse_cdf(S->r, V, u, &m);
    marg_pick = fmin(marg_pick, m);
  }

  /* step 6: outputs */
  J->accepted_len[b] = jstar;
  for (int j = 0; j < jstar; ++j) tok[j] = Db[j];
  tok[jstar] = (int32_t)pick;
  for (int j = jstar + 1; j <= k; ++j) tok[j] = -1;
  if (J->margin) J->margin[b] = fmin(marg, marg_pick);
  if (J->margin_pick) J->margin_pick[b] = marg_pick;
}

/* Closed-form acceptance of every draft position of sequence b [M "The
 * acceptance ceiling"]: when the draft is drawn from q_j, modified rejection
 * sampling accepts with probability sum_x min(p_j(x), mu_j(x)) (plain mode:
 * the maximal-coupling bound sum_x min(p, q) = 1 - TV), sampler-match with
 * sum_x p_j(x) q_j(x), and the argmax rule with q_j(argmax p_j).  mu_j is the
 * retained measure of the gate (its threshold, schedule and cumulative floor
 * with the drafted prefix D_0..D_{j-1}).  A position whose rows p_j, q_j (or,
 * with a cumulative floor, an earlier draft row or drafted token) are invalid
 * gets NaN, as does every position of a gated sequence with a threshold
 * outside (0, 1] and no schedule. */
static void diagnose_one(const job_t* J, int b, scratch_t* S) {
  const int k = J->k;
  const int64_t V = J->V;
  const int gated = J->gate[b] != 0;
  const int32_t* Db = J->D + (int64_t)b * k;
  const int esz_t = J->tdt == ORACLE_BF16 ? 2 : 4, esz_d = J->ddt == ORACLE_BF16 ? 2 : 4;
  int bad_t[ORACLE_MAX_K], bad_d[ORACLE_MAX_K];
  double mx, lse;
  double marg = INFINITY;
  for (int j = 0; j < k; ++j) {
    const char* rt = (const char*)J->Lt + ((int64_t)b * (k + 1) + j) * V * esz_t;
    const char* rd = (const char*)J->Ld + ((int64_t)b * k + j) * V * esz_d;
    bad_t[j] = oracle_softmax_row(rt, J->tdt, V, J->T, S->P + (int64_t)j * V, &mx, &lse);
    bad_d[j] = oracle_softmax_row(rd, J->ddt, V, J->T, S->Q + (int64_t)j * V, &mx, &lse);
    if (J->top_k) {  /* the sampler filters, as in verify_one */
      double fm = INFINITY;
      if (!bad_t[j])
        bad_t[j] = oracle_filtered_row(rt, J->tdt, V, J->T, J->top_k[0], J->top_p[0], J->min_p[0],
                                       S->P + (int64_t)j * V, &fm, NULL);
      marg = fmin(marg, fm);
      fm = INFINITY;
      if (!bad_d[j])
        bad_d[j] = oracle_filtered_row(rd, J->ddt, V, J->T, J->top_k[1], J->top_p[1], J->min_p[1],
                                       S->Q + (int64_t)j * V, &fm, NULL);
      marg = fmin(marg, fm);
    }
  }
  const int cum = gated && J->min_cum > 0.0;
  const int bad_tau = gated && !J->tau_sched && !(J->tau[b] > 0.0 && J->tau[b] <= 1.0);
  double cprev = 1.0;   /* prod_{i<j} q_i(D_i) */
  int prefix_bad = 0;   /* an earlier draft row or drafted token the product needs is invalid */
  for (int j = 0; j < k; ++j) {
    const int64_t o = (int64_t)b * k + j;
    const double* pj = S->P + (int64_t)j * V;
    const double* qj = S->Q + (int64_t)j * V;
    if (bad_t[j] || bad_d[j] || bad_tau || (cum && prefix_bad)) {
      if (J->diag_min) J->diag_min[o] = NAN;
      if (J->diag_pq) J->diag_pq[o] = NAN;
      if (J->diag_argq) J->diag_argq[o] = NAN;
    } else {
      const double tau = step_threshold(J, b, j);
      retained_measure(J, gated, tau, cprev, qj, S->mu);
      double smin = 0.0, spq = 0.0;
      for (int64_t v = 0; v < V; ++v) {
        smin += fmin(pj[v], S->mu[v]);
        spq += pj[v] * qj[v];
        if (gated) marg = fmin(marg, gate_margin(J, tau, cprev, qj[v]));
      }
      if (J->diag_min) J->diag_min[o] = smin;
      if (J->diag_pq) J->diag_pq[o] = spq;
      if (J->diag_argq) J->diag_argq[o] = qj[argmax_first(pj, V)];
    }
    if (bad_d[j] || Db[j] < 0 || (int64_t)Db[j] >= V) prefix_bad = 1;
    else cprev *= qj[Db[j]];
  }
  if (J->margin) J->margin[b] = marg;
}

/* ------------------------------------------- pick intervals (test aid) */

/* Where token v lies in the distribution that a stop row samples from, so
 * that a result computed in lower precision near a decision boundary can be
 * judged: the chain of one sequence stops at position j, and the stop row
 * samples, as in step 5 of verify_one, p_k (j = k, the ordinary bonus sample
 * [S "Approach"]) or the positive part of p_j - mu_j, mu_j the retained
 * measure of the gate at step j behind the drafted prefix D_0..D_{j-1} (plain
 * mode mu_j = q_j [M "What changed"]), or p_j when that part has no mass.
 * The weights are written out here once more, separately from verify_one, so
 * that the two can be checked against each other. */
int oracle_pick_interval(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                         int k, int64_t V, double T, int gated, double tau,
                         const double* tau_sched, int n_sched, double min_cum,
                         const int* top_k, const double* top_p, const double* min_p,
                         int j, int64_t v, double* weight, double* lo, double* hi,
                         double* gate_marg) {
  if (k < 1 || k > ORACLE_MAX_K || V < 1 || !(T >= 0.0) || isinf(T)) return 1;
  if (j < 0 || j > k || v < 0 || v >= V || !Lt || !Ld || !D || !weight || !lo || !hi) return 1;
  if ((tdt != ORACLE_F32 && tdt != ORACLE_BF16) || (ddt != ORACLE_F32 && ddt != ORACLE_BF16)) return 1;
  if ((top_k != NULL) != (top_p != NULL) || (top_k != NULL) != (min_p != NULL)) return 1;
  if (tau_sched && n_sched < 1) return 1;
  const uint8_t g = gated ? 1 : 0;
  job_t J;
  memset(&J, 0, sizeof J);
  J.k = k;
  J.V = V;
  J.T = T;
  J.gate = &g;
  J.tau = &tau;
  J.rule = ORACLE_RULE_MU;
  J.tau_sched = tau_sched;
  J.n_sched = n_sched;
  J.min_cum = min_cum;
  const int esz_t = tdt == ORACLE_BF16 ? 2 : 4, esz_d = ddt == ORACLE_BF16 ? 2 : 4;
  double* pj = (double*)malloc((size_t)V * sizeof(double));
  double* qi = (double*)malloc((size_t)V * sizeof(double));
  double* mu = (double*)malloc((size_t)V * sizeof(double));
  int bad = !pj || !qi || !mu;
  double mx, lse;
  /* the stop row's target distribution (filtered like the rows of verify_one) */
  if (!bad) {
    const char* row = (const char*)Lt + (int64_t)j * V * esz_t;
    bad = oracle_softmax_row(row, tdt, V, T, pj, &mx, &lse);
    if (!bad && top_k) bad = oracle_filtered_row(row, tdt, V, T, top_k[0], top_p[0], min_p[0], pj, NULL, NULL);
  }
  /* the draft rows up to the stop row: the prefix product of the drafted
   * tokens' draft probabilities, and mu_j from q_j */
  double cprev = 1.0;
  for (int i = 0; !bad && i < k && i <= j; ++i) {
    const char* row = (const char*)Ld + (int64_t)i * V * esz_d;
    bad = oracle_softmax_row(row, ddt, V, T, qi, &mx, &lse);
    if (!bad && top_k) bad = oracle_filtered_row(row, ddt, V, T, top_k[1], top_p[1], min_p[1], qi, NULL, NULL);
    if (bad) break;
    if (i < j) {
      if (D[i] < 0 || (int64_t)D[i] >= V) bad = 1;
      else cprev *= qi[D[i]];
    }
  }
  double gm = INFINITY;
  if (!bad) {
    if (j < k) {
      const double tau_j = step_threshold(&J, 0, j);
      retained_measure(&J, gated, tau_j, cprev, qi, mu);
      if (gated)
        for (int64_t x = 0; x < V; ++x) gm = fmin(gm, gate_margin(&J, tau_j, cprev, qi[x]));
      double mass = 0.0;
      for (int64_t x = 0; x < V; ++x) mass += fmax(pj[x] - mu[x], 0.0);
      if (mass > 0.0)
        for (int64_t x = 0; x < V; ++x) mu[x] = fmax(pj[x] - mu[x], 0.0);
      else
        memcpy(mu, pj, (size_t)V * sizeof(double));  /* no residual mass: p itself */
    } else {
      memcpy(mu, pj, (size_t)V * sizeof(double));
    }
    /* mu now holds the stop row's weights; prefix sums in token order */
    double Z = 0.0, below = 0.0;
    for (int64_t x = 0; x < V; ++x) {
      if (x == v) below = Z;
      Z += mu[x];
    }
    *weight = mu[v] / Z;
    *lo = below / Z;
    *hi = (below + mu[v]) / Z;
  }
  if (gate_marg) *gate_marg = gm;
  free(pj); free(qi); free(mu);
  return bad ? 1 : 0;
}

/* ------------------------------------------------------------- batch */

typedef struct {
  const job_t* J;
  int first, stride;
  int err;
} worker_t;

static void* worker_main(void* arg) {
  worker_t* w = (worker_t*)arg;
  const job_t* J = w->J;
  scratch_t S;
  const size_t V = (size_t)J->V;
  S.P = (double*)malloc((size_t)(J->k + 1) * V * sizeof(double));
  S.Q = (double*)malloc((size_t)(J->k > 0 ? J->k : 1) * V * sizeof(double));
  S.mu = (double*)malloc(V * sizeof(double));
  S.r = (double*)malloc(V * sizeof(double));
  if (!S.P || !S.Q || !S.mu || !S.r) {
    w->err = 1;
  } else {
    for (int b = w->first; b < J->B; b += w->stride) {
      if (J->diagnose) diagnose_one(J, b, &S);
      else verify_one(J, b, &S);
    }
  }
  free(S.P); free(S.Q); free(S.mu); free(S.r);
  return NULL;
}

static int run_jobs(const job_t* Jp, int nthreads);

int oracle_verify(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                  int B, int k, int64_t V, double T,
                  const uint8_t* gate, const double* tau,
                  uint64_t seed, uint64_t seq_offset,
                  const double* u0, const double* u1, int rule,
                  int32_t* accepted_len, int32_t* tokens, double* alpha, int8_t* flags,
                  double* row_stats, double* margin, double* margin_pick,
                  int32_t* degenerate, int nthreads) {
  return oracle_verify_policy(Lt, tdt, Ld, ddt, D, B, k, V, T, gate, tau, NULL, 0, 0.0, seed,
                              seq_offset, u0, u1, rule, accepted_len, tokens, alpha, flags,
                              row_stats, margin, margin_pick, degenerate, nthreads);
}

int oracle_verify_policy(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                         int B, int k, int64_t V, double T,
                         const uint8_t* gate, const double* tau,
                         const double* tau_sched, int n_sched, double min_cum,
                         uint64_t seed, uint64_t seq_offset,
                         const double* u0, const double* u1, int rule,
                         int32_t* accepted_len, int32_t* tokens, double* alpha, int8_t* flags,
                         double* row_stats, double* margin, double* margin_pick,
                         int32_t* degenerate, int nthreads) {
  return oracle_verify_filtered(Lt, tdt, Ld, ddt, D, B, k, V, T, gate, tau, tau_sched, n_sched, min_cum,
                                NULL, NULL, NULL, seed, seq_offset, u0, u1, rule, accepted_len, tokens,
                                alpha, flags, row_stats, margin, margin_pick, NULL, degenerate, nthreads);
}

int oracle_verify_filtered(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                           int B, int k, int64_t V, double T,
                           const uint8_t* gate, const double* tau,
                           const double* tau_sched, int n_sched, double min_cum,
                           const int* top_k, const double* top_p, const double* min_p,
                           uint64_t seed, uint64_t seq_offset,
                           const double* u0, const double* u1, int rule,
                           int32_t* accepted_len, int32_t* tokens, double* alpha, int8_t* flags,
                           double* row_stats, double* margin, double* margin_pick,
                           double* margin_filter, int32_t* degenerate, int nthreads) {
  if (B < 0 || k < 1 || k > ORACLE_MAX_K || V < 1 || !(T >= 0.0) || isinf(T)) return 1;
  if ((top_k != NULL) != (top_p != NULL) || (top_k != NULL) != (min_p != NULL)) return 1;
  for (int i = 0; top_k && i < 2; ++i)
    if (top_k[i] < 0 || !(top_p[i] > 0.0 && top_p[i] <= 1.0) || !(min_p[i] >= 0.0 && min_p[i] <= 1.0))
      return 1;
  if (tau_sched && n_sched < 1) return 1;
  if (!(min_cum >= 0.0 && min_cum <= 1.0)) return 1;
  if (B == 0) return 0;
  if (!Lt || !Ld || !D || !gate || !tau || !accepted_len || !tokens || !alpha || !flags) return 1;
  if ((tdt != ORACLE_F32 && tdt != ORACLE_BF16) || (ddt != ORACLE_F32 && ddt != ORACLE_BF16)) return 1;
  if (rule < ORACLE_RULE_MU || rule > ORACLE_RULE_MU_STEP_ONLY) return 1;
  job_t J = {Lt, tdt, Ld, ddt, D, B, k, V, T, gate, tau, seed, seq_offset, u0, u1, rule,
             accepted_len, tokens, alpha, flags, row_stats, margin, margin_pick, degenerate,
             margin_filter, tau_sched, n_sched, min_cum, top_k, top_p, min_p, 0, NULL, NULL, NULL};
  return run_jobs(&J, nthreads);
}

int oracle_diagnostics(const void* Lt, int tdt, const void* Ld, int ddt, const int32_t* D,
                       int B, int k, int64_t V, double T,
                       const uint8_t* gate, const double* tau,
                       const double* tau_sched, int n_sched, double min_cum,
                       const int* top_k, const double* top_p, const double* min_p,
                       double* min_sum, double* pq_sum, double* argmax_q, double* margin,
                       int nthreads) {
  if (B < 0 || k < 1 || k > ORACLE_MAX_K || V < 1 || !(T >= 0.0) || isinf(T)) return 1;
  if (tau_sched && n_sched < 1) return 1;
  if (!(min_cum >= 0.0 && min_cum <= 1.0)) return 1;
  if (B == 0) return 0;
  if (!Lt || !Ld || !D || !gate || !tau) return 1;
  if ((tdt != ORACLE_F32 && tdt != ORACLE_BF16) || (ddt != ORACLE_F32 && ddt != ORACLE_BF16)) return 1;
  job_t J = {Lt, tdt, Ld, ddt, D, B, k, V, T, gate, tau, 0, 0, NULL, NULL, ORACLE_RULE_MU,
             NULL, NULL, NULL, NULL, NULL, margin, NULL, NULL, NULL,
             tau_sched, n_sched, min_cum, top_k, top_p, min_p, 1, min_sum, pq_sum, argmax_q};
  return run_jobs(&J, nthreads);
}

/* the sequences of a job split over nthreads worker threads */
static int run_jobs(const job_t* Jp, int nthreads) {
  const job_t J = *Jp;
  const int B = J.B;
  if (nthreads < 1) nthreads = 1;
  if (nthreads > B) nthreads = B;
  worker_t* ws = (worker_t*)calloc((size_t)nthreads, sizeof(worker_t));
  pthread_t* th = (pthread_t*)calloc((size_t)nthreads, sizeof(pthread_t));
  if (!ws || !th) {
    free(ws); free(th);
    return 1;
  }
  for (int t = 0; t < nthreads; ++t) {
    ws[t].J = &J;
    ws[t].first = t;
    ws[t].stride = nthreads;
  }
  int err = 0;
  if (nthreads == 1) {
    worker_main(&ws[0]);
  } else {
    for (int t = 0; t < nthreads; ++t) pthread_create(&th[t], NULL, worker_main, &ws[t]);
    for (int t = 0; t < nthreads; ++t) pthread_join(th[t], NULL);
  }
  for (int t = 0; t < nthreads; ++t) err |= ws[t].err;
  free(ws); free(th);
  return err ? 1 : 0;
}
