/*
 * Drives every entry point of the CPU oracle over ordinary, edge-case and
 * invalid inputs so that the oracle can be built and run under
 * AddressSanitizer and UndefinedBehaviorSanitizer (tests/test_oracle_sanitized.py).
 *
 * It checks only what must hold for any input -- return codes, token ranges,
 * lengths within [-1, k] -- and leaves the arithmetic to the pinned tests; its
 * job is to make out-of-bounds accesses, leaks, overflow and other undefined
 * behaviour in the oracle visible.  Inputs come from a small xorshift
 * generator of its own.
 */
#include <math.h>
#include <stdint.h>
#include <stdio.h>
#include <stdlib.h>
#include <string.h>

#include "spec_verify_oracle.h"

static uint64_t rng_state = 0x9e3779b97f4a7c15ull;

static double rnd(void) {  /* uniform in [0, 1) */
  rng_state ^= rng_state << 13;
  rng_state ^= rng_state >> 7;
  rng_state ^= rng_state << 17;
  return (double)(rng_state >> 11) * (1.0 / 9007199254740992.0);
}

static double gauss(void) {
  const double u = rnd() + 1e-12, v = rnd();
  return sqrt(-2.0 * log(u)) * cos(6.283185307179586 * v);
}

static int failures = 0;
#define CHECK(cond, ...)                      \
  do {                                        \
    if (!(cond)) {                            \
      fprintf(stderr, "check failed: ");      \
      fprintf(stderr, __VA_ARGS__);           \
      fprintf(stderr, "\n");                  \
      ++failures;                             \
    }                                         \
  } while (0)

/* logits of n entries in element type dt: N(0, s^2), one raised entry per row */
static void* make_logits(int dt, int64_t rows, int64_t V, double s) {
  const int64_t n = rows * V;
  if (dt == ORACLE_F32) {
    float* x = malloc((size_t)(n > 0 ? n : 1) * sizeof(float));
    for (int64_t i = 0; i < n; ++i) x[i] = (float)(s * gauss());
    for (int64_t r = 0; r < rows; ++r) x[r * V + (int64_t)(rnd() * (double)V)] += 4.0f;
    return x;
  }
  uint16_t* x = malloc((size_t)(n > 0 ? n : 1) * sizeof(uint16_t));
  for (int64_t i = 0; i < n; ++i) {
    float f = (float)(s * gauss());
    if (i % V == 0 && rnd() < 0.5) f += 4.0f;
    uint32_t bits;
    memcpy(&bits, &f, 4);
    x[i] = (uint16_t)(bits >> 16);
  }
  return x;
}

static void set_logit(void* L, int dt, int64_t i, float f) {
  if (dt == ORACLE_F32) {
    ((float*)L)[i] = f;
  } else {
    uint32_t bits;
    memcpy(&bits, &f, 4);
    ((uint16_t*)L)[i] = (uint16_t)(bits >> 16);
  }
}

typedef struct {
  int32_t* len;
  int32_t* tok;
  double* alpha;
  int8_t* flags;
  double* stats;
  double* margin;
  double* margin_pick;
  double* margin_filter;
  int32_t* degenerate;
} outputs_t;

static outputs_t alloc_outputs(int B, int k) {
  outputs_t o;
  const size_t b = (size_t)(B > 0 ? B : 1);
  o.len = malloc(b * sizeof(int32_t));
  o.tok = malloc(b * (size_t)(k + 1) * sizeof(int32_t));
  o.alpha = malloc(b * (size_t)k * sizeof(double));
  o.flags = malloc(b * (size_t)k);
  o.stats = malloc(b * (size_t)(2 * k + 1) * 2 * sizeof(double));
  o.margin = malloc(b * sizeof(double));
  o.margin_pick = malloc(b * sizeof(double));
  o.margin_filter = malloc(b * sizeof(double));
  o.degenerate = malloc(b * sizeof(int32_t));
  return o;
}

static void free_outputs(outputs_t* o) {
  free(o->len);
  free(o->tok);
  free(o->alpha);
  free(o->flags);
  free(o->stats);
  free(o->margin);
  free(o->margin_pick);
  free(o->margin_filter);
  free(o->degenerate);
}

static void check_outputs(const outputs_t* o, int B, int k, int64_t V, const char* what) {
  for (int b = 0; b < B; ++b) {
    CHECK(o->len[b] >= -1 && o->len[b] <= k, "%s: accepted_len %d outside [-1, %d]", what, o->len[b], k);
    for (int j = 0; j <= k; ++j) {
      const int32_t t = o->tok[(int64_t)b * (k + 1) + j];
      CHECK(t >= -1 && t < V, "%s: token %d outside [-1, %lld)", what, t, (long long)V);
    }
    for (int j = 0; j < k; ++j) {
      const double a = o->alpha[(int64_t)b * k + j];
      CHECK(a >= 0.0 && a <= 1.0, "%s: alpha %g outside [0, 1]", what, a);
      const int f = o->flags[(int64_t)b * k + j];
      CHECK(f >= ORACLE_FLAG_UNREACHED && f <= ORACLE_FLAG_INVALID, "%s: flag %d", what, f);
    }
  }
}

/* one batch through oracle_verify, oracle_verify_policy, oracle_verify_filtered
 * and oracle_diagnostics */
static void run_batch(int tdt, int ddt, int B, int k, int64_t V, double T, int rule, int nthreads,
                      int explicit_u, int poison) {
  void* Lt = make_logits(tdt, (int64_t)B * (k + 1), V, 2.0);
  void* Ld = make_logits(ddt, (int64_t)B * k, V, 2.0);
  int32_t* D = malloc((size_t)B * (size_t)k * sizeof(int32_t));
  uint8_t* gate = malloc((size_t)B);
  double* tau = malloc((size_t)B * sizeof(double));
  double* u0 = malloc((size_t)B * (size_t)k * sizeof(double));
  double* u1 = malloc((size_t)B * sizeof(double));
  static const double edge_u[4] = {0.0, 0.5, 0.99999994039535522, 0.25};
  for (int b = 0; b < B; ++b) {
    gate[b] = (uint8_t)(b % 2);
    tau[b] = b % 3 == 0 ? 0.5 : (b % 3 == 1 ? 0.3 : 1.0);
    u1[b] = edge_u[b % 4];
    for (int j = 0; j < k; ++j) {
      D[b * k + j] = (int32_t)(rnd() * (double)V);
      u0[b * k + j] = edge_u[(b + j) % 4];
    }
  }
  if (poison && B >= 4 && V >= 2) {
    /* invalid rows and tokens: the oracle must fail those sequences closed */
    set_logit(Lt, tdt, 0 * (int64_t)(k + 1) * V + 1, NAN);          /* NaN in a target row */
    for (int64_t v = 0; v < V; ++v) set_logit(Ld, ddt, 1 * (int64_t)k * V + v, -INFINITY);
    set_logit(Lt, tdt, 2 * (int64_t)(k + 1) * V, INFINITY);        /* +inf logit */
    D[3 * k] = (int32_t)V;                                          /* token out of range */
    if (B >= 5) D[4 * k] = -1;
    if (B >= 6) {
      gate[5] = 1;
      tau[5] = 1.5;                                                 /* threshold outside (0, 1] */
    }
    if (B >= 8) {
      gate[7] = 1;
      tau[7] = 0.0;
    }
  }
  const double* pu0 = explicit_u ? u0 : NULL;
  const double* pu1 = explicit_u ? u1 : NULL;
  char what[160];
  snprintf(what, sizeof what, "tdt %d ddt %d B %d k %d V %lld T %g rule %d threads %d u %d poison %d",
           tdt, ddt, B, k, (long long)V, T, rule, nthreads, explicit_u, poison);

  outputs_t o = alloc_outputs(B, k);
  int rc = oracle_verify(Lt, tdt, Ld, ddt, D, B, k, V, T, gate, tau, 1234u, 7u, pu0, pu1, rule, o.len,
                         o.tok, o.alpha, o.flags, o.stats, o.margin, o.margin_pick, o.degenerate,
                         nthreads);
  CHECK(rc == 0, "%s: oracle_verify returned %d", what, rc);
  if (rc == 0) check_outputs(&o, B, k, V, what);

  static const double sched[3] = {0.25, 0.0, 0.5};
  rc = oracle_verify_policy(Lt, tdt, Ld, ddt, D, B, k, V, T, gate, tau, sched, 3, 0.01, 99u, 0u, pu0,
                            pu1, rule, o.len, o.tok, o.alpha, o.flags, NULL, o.margin, NULL, NULL,
                            nthreads);
  CHECK(rc == 0, "%s: oracle_verify_policy returned %d", what, rc);
  if (rc == 0) check_outputs(&o, B, k, V, what);

  if (rule == ORACLE_RULE_MU) {
    const int top_k[2] = {5, 1};
    const double top_p[2] = {0.9, 0.5};
    const double min_p[2] = {0.05, 0.0};
    rc = oracle_verify_filtered(Lt, tdt, Ld, ddt, D, B, k, V, T, gate, tau, NULL, 0, 0.0, top_k, top_p,
                                min_p, 5u, 0u, pu0, pu1, rule, o.len, o.tok, o.alpha, o.flags, o.stats,
                                o.margin, o.margin_pick, o.margin_filter, o.degenerate, nthreads);
    CHECK(rc == 0, "%s: oracle_verify_filtered returned %d", what, rc);
    if (rc == 0) check_outputs(&o, B, k, V, what);

    double* min_sum = malloc((size_t)B * (size_t)k * sizeof(double));
    double* pq_sum = malloc((size_t)B * (size_t)k * sizeof(double));
    double* argmax_q = malloc((size_t)B * (size_t)k * sizeof(double));
    rc = oracle_diagnostics(Lt, tdt, Ld, ddt, D, B, k, V, T, gate, tau, sched, 3, 0.02, NULL, NULL, NULL,
                            min_sum, pq_sum, argmax_q, o.margin, nthreads);
    CHECK(rc == 0, "%s: oracle_diagnostics returned %d", what, rc);
    rc = oracle_diagnostics(Lt, tdt, Ld, ddt, D, B, k, V, T, gate, tau, NULL, 0, 0.0, top_k, top_p, min_p,
                            min_sum, NULL, argmax_q, NULL, nthreads);
    CHECK(rc == 0, "%s: filtered oracle_diagnostics returned %d", what, rc);
    for (int i = 0; i < B * k; ++i)
      CHECK(isnan(min_sum[i]) || (min_sum[i] >= -1e-12 && min_sum[i] <= 1.0 + 1e-12),
            "%s: min_sum %g", what, min_sum[i]);
    free(min_sum);
    free(pq_sum);
    free(argmax_q);
  }
  free_outputs(&o);
  free(Lt);
  free(Ld);
  free(D);
  free(gate);
  free(tau);
  free(u0);
  free(u1);
}

static void single_row_functions(void) {
  /* Philox and the uniform */
  const uint32_t ctr[4] = {0u, 1u, 2u, 3u}, key[2] = {0xdeadbeefu, 0x12345678u};
  uint32_t out[4];
  oracle_philox4x32_10(ctr, key, out);
  for (uint32_t d = 0; d < 4; ++d) {
    const double u = oracle_uniform(0xffffffffffffffffull, 0xfffffffffull, 0xffffffffu, d);
    CHECK(u >= 0.0 && u < 1.0, "uniform %g outside [0, 1)", u);
  }
  /* softmax rows: V = 1, all -inf, NaN, greedy, no output array */
  float row[5] = {0.f, -INFINITY, 3.f, 3.f, -1.f};
  double p[5], m, lse;
  CHECK(oracle_softmax_row(row, ORACLE_F32, 5, 0.8, p, &m, &lse) == 0, "softmax of a valid row");
  CHECK(oracle_softmax_row(row, ORACLE_F32, 5, 0.0, p, &m, &lse) == 0, "greedy softmax");
  CHECK(p[2] == 1.0 && p[3] == 0.0, "greedy keeps the first largest logit");
  CHECK(oracle_softmax_row(row, ORACLE_F32, 1, 1.0, NULL, &m, &lse) == 0, "softmax of V = 1");
  float bad[3] = {-INFINITY, -INFINITY, -INFINITY};
  CHECK(oracle_softmax_row(bad, ORACLE_F32, 3, 1.0, p, &m, &lse) == 1, "an all -inf row is invalid");
  bad[1] = NAN;
  CHECK(oracle_softmax_row(bad, ORACLE_F32, 3, 1.0, p, &m, &lse) == 1, "a NaN row is invalid");
  /* inverse CDF: no mass, one entry, u at both ends */
  const double zeros[4] = {0.0, 0.0, 0.0, 0.0}, one[4] = {0.0, 0.0, 2.0, 0.0};
  double margin;
  CHECK(oracle_inverse_cdf(zeros, 4, 0.5, &margin) == -1, "no mass gives -1");
  CHECK(oracle_inverse_cdf(one, 4, 0.0, &margin) == 2, "u = 0 picks the only positive weight");
  CHECK(oracle_inverse_cdf(one, 4, 0.99999994039535522, NULL) == 2, "u near 1 picks it too");
  CHECK(oracle_inverse_cdf(one, 1, 0.5, NULL) == -1, "a prefix without mass gives -1");
  /* filtered rows: every filter, each off, top_k beyond V */
  double kept;
  for (int t = 0; t < 4; ++t) {
    oracle_softmax_row(row, ORACLE_F32, 5, 1.0, p, &m, &lse);
    const int tk[4] = {2, 0, 1, 9};
    const double tp[4] = {0.7, 1.0, 0.3, 0.999};
    const double mp[4] = {0.0, 0.5, 0.0, 1.0};
    CHECK(oracle_filtered_row(row, ORACLE_F32, 5, 1.0, tk[t], tp[t], mp[t], p, &margin, &kept) == 0,
          "filtered row %d", t);
  }
}

int main(void) {
  single_row_functions();
  static const int64_t Vs[5] = {1, 2, 7, 67, 300};
  static const double Ts[3] = {1.0, 0.7, 0.0};
  static const int dts[3][2] = {{ORACLE_F32, ORACLE_F32}, {ORACLE_BF16, ORACLE_BF16}, {ORACLE_F32, ORACLE_BF16}};
  int cases = 0;
  for (int d = 0; d < 3; ++d)
    for (int vi = 0; vi < 5; ++vi)
      for (int ti = 0; ti < 3; ++ti) {
        const int k = 1 + (vi + ti) % 4;
        run_batch(dts[d][0], dts[d][1], 8, k, Vs[vi], Ts[ti], ORACLE_RULE_MU, 1 + (ti % 3), vi % 2, 0);
        run_batch(dts[d][0], dts[d][1], 8, k, Vs[vi], Ts[ti], ORACLE_RULE_MU, 2, 1, 1);
        cases += 2;
      }
  /* every control rule, plain and gated sequences */
  for (int rule = ORACLE_RULE_MU; rule <= ORACLE_RULE_MU_STEP_ONLY; ++rule) {
    run_batch(ORACLE_F32, ORACLE_F32, 6, 3, 8, 1.0, rule, 1, 0, 0);
    run_batch(ORACLE_BF16, ORACLE_F32, 6, 2, 67, 0.7, rule, 3, 1, 0);
    cases += 2;
  }
  /* the largest k, and an empty batch */
  run_batch(ORACLE_F32, ORACLE_F32, 2, ORACLE_MAX_K, 3, 1.0, ORACLE_RULE_MU, 2, 0, 0);
  {
    outputs_t o = alloc_outputs(1, 2);
    float one = 0.f;
    const int rc = oracle_verify(&one, ORACLE_F32, &one, ORACLE_F32, NULL, 0, 2, 1, 1.0, NULL, NULL, 0u,
                                 0u, NULL, NULL, ORACLE_RULE_MU, o.len, o.tok, o.alpha, o.flags, NULL,
                                 NULL, NULL, NULL, 1);
    CHECK(rc == 0 || rc == 1, "empty batch returned %d", rc);
    free_outputs(&o);
  }
  printf("%d batches, %d failed checks\n", cases + 2, failures);
  return failures == 0 ? 0 : 1;
}
