"""Pins of the CPU oracle against what the pages and the mathematics fix.

None of these tests compares the oracle with a retyped copy of itself: each
checks a printed value (the gated worked example, the Philox known answers,
the chi-square threshold), a closed form (sum min(p, q) = 1 - TV, sum p*q), a
library routine (scipy's logsumexp), an exact law obtained by enumeration, or
a zero-tolerance support property.  Known-wrong control rules show that each
law test has the power to reject a plausible mistake.
"""
import os

import numpy as np
import pytest
from scipy.special import logsumexp, softmax
from scipy.stats import chi2

from oracle import oracle as O
from tests.law import distributions, exact_law, position_marginals

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _golden_rows(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


# ------------------------------------------------------------------ Philox

def test_philox_known_answers():
    for row in _golden_rows("philox4x32_10_kat.txt"):
        w = [int(x, 16) for x in row]
        out = O.philox4x32_10(w[0:4], w[4:6])
        assert [int(x) for x in out] == w[6:10]


def test_uniform_maps_seed_sequence_position_draw_onto_key_and_counter():
    # key = (seed lo, seed hi), counter = (seq lo, pos, draw, seq hi), u = (out0 >> 8) 2^-24
    rows = [[int(x, 16) for x in r] for r in _golden_rows("philox4x32_10_kat.txt")]
    for c0, c1, c2, c3, k0, k1, o0, *_ in rows:
        seed = k0 | (k1 << 32)
        seq = c0 | (c3 << 32)
        assert O.uniform(seed, seq, c1, c2) == (o0 >> 8) / 2.0 ** 24


def test_uniforms_are_24_bit_grid_points_and_look_uniform():
    u = np.array([O.uniform(12345, b, j, d) for b in range(200) for j in range(5) for d in range(2)])
    assert np.all((u >= 0) & (u < 1))
    assert np.all(u * 2 ** 24 == np.floor(u * 2 ** 24))
    # Kolmogorov-Smirnov distance against U[0,1) for 2000 draws: 1.95/sqrt(n) is alpha ~ 1e-3
    s = np.sort(u)
    n = len(s)
    ks = max(np.max(np.arange(1, n + 1) / n - s), np.max(s - np.arange(n) / n))
    assert ks < 1.95 / np.sqrt(n)


# ------------------------------------------------------------------ softmax

@pytest.mark.parametrize("T", [0.7, 1.0, 1.5])
@pytest.mark.parametrize("bf16", [False, True])
def test_softmax_row_matches_library_logsumexp(T, bf16):
    rng = np.random.default_rng(3)
    x = (rng.standard_normal(1000) * 4).astype(np.float32)
    if bf16:
        bits = x.view(np.uint32) >> 16
        arr = bits.astype(np.uint16)
        x = (bits << 16).astype(np.uint32).view(np.float32)
    else:
        arr = x
    p, mx, lse, ok = O.softmax_row(arr, T)
    xs = x.astype(np.float64) / T
    assert ok
    assert mx == np.max(xs)
    assert abs(lse - logsumexp(xs)) <= 1e-12 * abs(logsumexp(xs))
    np.testing.assert_allclose(p, softmax(xs), rtol=1e-12, atol=0)


def test_softmax_row_invalid_and_minus_inf():
    x = np.array([0.0, -np.inf, 1.0], dtype=np.float32)
    p, _, _, ok = O.softmax_row(x, 1.0)
    assert ok and p[1] == 0.0 and abs(p.sum() - 1) < 1e-15
    for bad in ([0.0, np.nan, 1.0], [0.0, np.inf, 1.0], [-np.inf, -np.inf]):
        _, _, _, ok = O.softmax_row(np.array(bad, dtype=np.float32), 1.0)
        assert not ok


# ------------------------------------------------------------- inverse CDF

def test_inverse_cdf_law_and_zero_weights():
    r = np.array([0.0, 0.2, 0.0, 0.5, 0.3, 0.0])
    # law over a fine u grid equals r / Z; zero-weight tokens never picked
    us = (np.arange(100000) + 0.5) / 100000
    picks = np.array([O.inverse_cdf(r, u)[0] for u in us[::10]])
    freq = np.bincount(picks, minlength=6) / len(picks)
    np.testing.assert_allclose(freq, r / r.sum(), atol=2e-4)
    assert O.inverse_cdf(r, 0.0)[0] == 1  # u = 0 must not pick the leading zero-weight token
    assert O.inverse_cdf(r, 1.0 - 2.0 ** -24)[0] == 4
    assert O.inverse_cdf(np.zeros(4), 0.3)[0] == -1


# ---------------------------------------------------------- exact laws

def _check_lossless(law, P, Q, gated, tau, tol=1e-10):
    k = Q.shape[0]
    V = P.shape[1]
    reach, emit, passed = position_marginals(law, k, V)
    assert abs(sum(law.values()) - 1.0) < tol
    for j in range(k + 1):
        if reach[j] > 1e-9:
            np.testing.assert_allclose(emit[j] / reach[j], P[j], atol=tol / reach[j])
    for j in range(k):
        if reach[j] > 1e-9:
            mu = Q[j] * (Q[j] >= tau) if gated else Q[j]
            assert abs(passed[j] / reach[j] - np.minimum(P[j], mu).sum()) < tol / reach[j]


def _worked_example():
    g = {r[0]: [float(x) for x in r[1:]] for r in _golden_rows("gated_worked_example.txt")}
    p, q = np.array(g["p"]), np.array(g["q"])
    Lt = np.log(np.stack([p, p])).astype(np.float32)  # k = 1: position 0 and the bonus row
    Ld = np.log(q)[None, :].astype(np.float32)
    return g, Lt, Ld


def test_worked_example_mu_rule_emits_p():
    g, Lt, Ld = _worked_example()
    law = exact_law(Lt, Ld, 1.0, True, g["threshold"][0], rule=O.RULE_MU)
    _, emit, _ = position_marginals(law, 1, 2)
    # the first emitted token's law is printed on the page; exact up to fp32 logits
    np.testing.assert_allclose(emit[0], g["emitted_mu_rule"], atol=1e-12)


def test_worked_example_original_gate_is_biased_as_printed():
    g, Lt, Ld = _worked_example()
    law = exact_law(Lt, Ld, 1.0, True, g["threshold"][0], rule=O.RULE_ORIGINAL_GATE)
    _, emit, _ = position_marginals(law, 1, 2)
    # fp32 logits move q by ~1e-8 from (0.875, 0.125); the biased law moves with it
    np.testing.assert_allclose(emit[0], g["emitted_original_gate"], atol=1e-7)


def _random_case(rng, V, k, scale=2.0, noise=1.0):
    Lt = (rng.standard_normal((k + 1, V)) * scale).astype(np.float32)
    Ld = (Lt[:k] + rng.standard_normal((k, V)) * noise).astype(np.float32)
    return Lt, Ld


@pytest.mark.parametrize("V,k", [(2, 1), (3, 2), (5, 2), (8, 3)])
@pytest.mark.parametrize("gated,tau", [(False, 0.5), (True, 0.5), (True, 0.3)])
def test_exact_law_is_lossless(V, k, gated, tau):
    rng = np.random.default_rng(100 * V + 10 * k + int(gated) + int(tau * 10))
    for trial in range(2):
        Lt, Ld = _random_case(rng, V, k, scale=2.0 + trial)
        T = 1.0 if trial == 0 else 0.7
        law = exact_law(Lt, Ld, T, gated, tau)
        P, Q = distributions(Lt, Ld, T)
        _check_lossless(law, P, Q, gated, tau)


def test_exact_law_plain_pass_rate_is_one_minus_tv():
    rng = np.random.default_rng(7)
    Lt, Ld = _random_case(rng, 6, 2)
    law = exact_law(Lt, Ld, 1.0, False, 0.5)
    P, Q = distributions(Lt, Ld, 1.0)
    reach, _, passed = position_marginals(law, 2, 6)
    for j in range(2):
        tv = 0.5 * np.abs(P[j] - Q[j]).sum()
        assert abs(passed[j] / reach[j] - (1.0 - tv)) < 1e-10
        assert passed[j] / reach[j] >= (P[j] * Q[j]).sum()


@pytest.mark.parametrize("rule", [O.RULE_ORIGINAL_GATE, O.RULE_RESAMPLE_P, O.RULE_ARGMAX,
                                  O.RULE_RENORM_MU, O.RULE_RESIDUAL_Q])
def test_exact_law_rejects_known_wrong_rules(rule):
    # p = (0.5, 0.25, 0.25), q = (0.6, 0.35, 0.05), tau = 0.5: each mistake moves the law
    p = np.array([0.5, 0.25, 0.25])
    q = np.array([0.6, 0.35, 0.05])
    Lt = np.log(np.stack([p, p])).astype(np.float32)
    Ld = np.log(q)[None, :].astype(np.float32)
    law = exact_law(Lt, Ld, 1.0, True, 0.5, rule=rule)
    _, emit, _ = position_marginals(law, 1, 3)
    assert np.max(np.abs(emit[0] - p)) > 1e-2


def test_exact_law_sampler_match_control_is_lossless_with_sum_pq():
    # sampler-match: accept iff a fresh target draw equals D; acceptance sum p*q [mlxcel #992]
    rng = np.random.default_rng(11)
    V, k, n = 5, 1, 200000
    Lt, Ld = _random_case(rng, V, k)
    P, Q = distributions(Lt, Ld, 1.0)
    D = rng.choice(V, size=(n, k), p=Q[0])
    out = O.verify(np.broadcast_to(Lt, (n, k + 1, V)), np.broadcast_to(Ld, (n, k, V)), D, 1.0, 0, 0.5,
                   seed=5, rule=O.RULE_SAMPLER_MATCH, nthreads=4)
    acc = (out["accepted_len"] >= 1).mean()
    spq = (P[0] * Q[0]).sum()
    assert abs(acc - spq) < 4 * np.sqrt(spq * (1 - spq) / n)
    assert spq <= np.minimum(P[0], Q[0]).sum()
    counts = np.bincount(out["tokens"][:, 0], minlength=V)
    stat = ((counts - n * P[0]) ** 2 / (n * P[0])).sum()
    assert stat < chi2.ppf(1 - 1e-4, V - 1)


def test_alpha_averages_to_sum_min_closed_form():
    # E_{D~q}[alpha(D)] = sum_x min(p, mu): pins alpha = min(1, p/mu) on every token
    rng = np.random.default_rng(5)
    V = 7
    Lt, Ld = _random_case(rng, V, 1)
    P, Q = distributions(Lt, Ld, 1.0)
    D = np.arange(V, dtype=np.int32)[:, None]
    for gated, tau in [(False, 0.5), (True, 0.2), (True, 0.45)]:
        out = O.verify(np.broadcast_to(Lt, (V, 2, V)), np.broadcast_to(Ld, (V, 1, V)), D, 1.0,
                       int(gated), tau, seed=1)
        mu = Q[0] * (Q[0] >= tau) if gated else Q[0]
        assert abs((Q[0] * out["alpha"][:, 0]).sum() - np.minimum(P[0], mu).sum()) < 1e-14


# ---------------------------------------------------------------- chi-square

def test_page_chi_square_threshold_is_the_library_quantile():
    g = {r[0]: float(r[1]) for r in _golden_rows("chi_square_threshold.txt")}
    assert abs(chi2.ppf(1 - g["alpha"], int(g["dof"])) - g["threshold"]) < 1e-4


def _tiny_config(rng, n):
    # tiny config: V=8, k=3, target ~ N(0, 2^2), draft = target + N(0, 1), T = 1
    V, k = 8, 3
    Lt, Ld = _random_case(rng, V, k)
    _, Q = distributions(Lt, Ld, 1.0)
    D = np.stack([rng.choice(V, size=n, p=Q[j]) for j in range(k)], axis=1).astype(np.int32)
    return Lt, Ld, D


def _chi_square_position0(out, P0):
    n = out["tokens"].shape[0]
    counts = np.bincount(out["tokens"][:, 0], minlength=len(P0))
    return ((counts - n * P0) ** 2 / (n * P0)).sum()


@pytest.mark.parametrize("gated", [False, True])
def test_chi_square_emitted_tokens_follow_p(gated):
    rng = np.random.default_rng(21 + gated)
    n = 100000
    Lt, Ld, D = _tiny_config(rng, n)
    P, Q = distributions(Lt, Ld, 1.0)
    out = O.verify(np.broadcast_to(Lt, (n, 4, 8)), np.broadcast_to(Ld, (n, 3, 8)), D, 1.0, int(gated),
                   0.5, seed=2024, nthreads=4)
    thr = chi2.ppf(1 - 1e-4, 7)
    assert _chi_square_position0(out, P[0]) < thr
    # every later position, conditional on being reached, also follows p_j
    for j in range(1, 4):
        sel = out["accepted_len"] >= j
        if sel.sum() > 2000:
            counts = np.bincount(out["tokens"][sel, j], minlength=8)
            m = sel.sum()
            assert ((counts - m * P[j]) ** 2 / (m * P[j])).sum() < thr


@pytest.mark.parametrize("rule", [O.RULE_RESAMPLE_P, O.RULE_ARGMAX, O.RULE_ORIGINAL_GATE])
def test_chi_square_rejects_known_wrong_rules(rule):
    rng = np.random.default_rng(40 + rule)
    n = 100000
    if rule == O.RULE_ORIGINAL_GATE:
        p, q = np.array([0.5, 0.5]), np.array([0.875, 0.125])
        Lt = np.log(np.stack([p, p])).astype(np.float32)
        Ld = np.log(q)[None, :].astype(np.float32)
        D = rng.choice(2, size=(n, 1), p=q).astype(np.int32)
        k, V = 1, 2
    else:
        Lt, Ld, D = _tiny_config(rng, n)
        k, V = 3, 8
    P, _ = distributions(Lt, Ld, 1.0)
    out = O.verify(np.broadcast_to(Lt, (n, k + 1, V)), np.broadcast_to(Ld, (n, k, V)), D, 1.0, 1,
                   0.5, seed=7, rule=rule, nthreads=4)
    with np.errstate(divide="ignore", invalid="ignore"):
        assert _chi_square_position0(out, P[0]) > chi2.ppf(1 - 1e-4, V - 1)


# ----------------------------------------------------------- support, edges

def test_zero_target_mass_is_never_accepted_or_emitted():
    # token 0 has p = 0 (target logit -inf); the drafter offers it, sometimes with q = 0 too
    rng = np.random.default_rng(9)
    n, V = 4000, 4
    Lt = np.tile(np.array([-np.inf, 0.0, 0.5, -1.0], dtype=np.float32), (n, 2, 1))
    Ld = np.tile(np.array([1.0, 0.0, 0.0, 0.0], dtype=np.float32), (n, 1, 1))
    Ld[: n // 2, 0, 0] = -np.inf  # underflowed proposal mass: u * 0 <= 0 must not accept
    D = np.zeros((n, 1), dtype=np.int32)
    for gated in (0, 1):
        out = O.verify(Lt, Ld, D, 1.0, gated, 0.3, seed=rng.integers(1 << 60))
        assert np.all(out["accepted_len"] == 0)
        assert np.all(out["tokens"][:, 0] != 0)
        assert np.all(out["alpha"][:, 0] == 0.0)


def test_residual_never_emits_tokens_where_p_le_mu():
    rng = np.random.default_rng(13)
    n, V = 20000, 6
    Lt, Ld = _random_case(rng, V, 1, scale=1.5, noise=1.5)
    P, Q = distributions(Lt, Ld, 1.0)
    D = rng.choice(V, size=(n, 1), p=Q[0]).astype(np.int32)
    for gated, tau in [(0, 0.5), (1, 0.25)]:
        out = O.verify(np.broadcast_to(Lt, (n, 2, V)), np.broadcast_to(Ld, (n, 1, V)), D, 1.0, gated,
                       tau, seed=3)
        mu = Q[0] * (Q[0] >= tau) if gated else Q[0]
        stopped = out["accepted_len"] == 0
        assert stopped.any()
        assert np.all(P[0][out["tokens"][stopped, 0]] > mu[out["tokens"][stopped, 0]])


def test_gate_equality_passes():
    # q = (0.5, 0.5) exactly (equal logits); threshold 0.5: the offered token is admitted, not NULL
    Lt = np.zeros((1, 2, 2), dtype=np.float32)
    Ld = np.zeros((1, 1, 2), dtype=np.float32)
    out = O.verify(Lt, Ld, np.array([[1]]), 1.0, 1, 0.5, u0=np.array([[0.999]]), u1=np.array([0.1]))
    assert out["flags"][0, 0] == O.FLAG_ACCEPT and out["alpha"][0, 0] == 1.0


def test_null_row_ends_the_chain_and_samples_the_residual():
    # gated, q(D) < tau: flag NULL, alpha 0, later positions unreached
    p = np.array([0.5, 0.5])
    q = np.array([0.875, 0.125])
    Lt = np.log(np.stack([p, p, p])).astype(np.float32)[None]
    Ld = np.log(np.stack([q, q])).astype(np.float32)[None]
    out = O.verify(Lt, Ld, np.array([[1, 0]]), 1.0, 1, 0.5, u0=np.array([[0.0, 0.0]]),
                   u1=np.array([0.0]))
    assert out["accepted_len"][0] == 0
    assert list(out["flags"][0]) == [O.FLAG_NULL, O.FLAG_UNREACHED]
    assert out["tokens"][0, 0] == 1  # residual (p - mu)+ = (0, 0.5): only token 1
    assert list(out["tokens"][0, 1:]) == [-1, -1]
    assert out["alpha"][0, 0] == 0.0 and out["alpha"][0, 1] > 0.5


def test_residual_without_mass_samples_p_and_is_reported():
    # [M] names a fallback for a degenerate residual without defining it; the
    # reading: when (p - mu)+ has no mass (mu = p), sample p with the same u1
    # and report the sequence as degenerate.  Here p = q = mu = (1, 0) at
    # threshold 1/2 and the offered token 1 has q = 0: a NULL row whose
    # residual is empty, so token 0 (all of p) is emitted.
    Lt = np.array([[[0.0, -np.inf], [0.0, -np.inf]]], dtype=np.float32)
    Ld = np.array([[[0.0, -np.inf]]], dtype=np.float32)
    out = O.verify(Lt, Ld, np.array([[1]], dtype=np.int32), 1.0, 1, 0.5)
    assert out["accepted_len"][0] == 0 and out["flags"][0, 0] == O.FLAG_NULL
    assert list(out["tokens"][0]) == [0, -1]
    assert out["degenerate"][0] == 1
    # an ordinary stop row is not degenerate
    p = np.array([0.5, 0.5])
    q = np.array([0.875, 0.125])
    Lt = np.log(np.stack([p, p])).astype(np.float32)[None]
    Ld = np.log(q).astype(np.float32)[None, None]
    out = O.verify(Lt, Ld, np.array([[1]], dtype=np.int32), 1.0, 1, 0.5)
    assert out["accepted_len"][0] == 0 and out["degenerate"][0] == 0


def test_invalid_sequences_fail_closed():
    rng = np.random.default_rng(1)
    Lt, Ld = _random_case(rng, 5, 2)
    Lt = np.stack([Lt] * 4)
    Ld = np.stack([Ld] * 4)
    D = np.zeros((4, 2), dtype=np.int32)
    Lt[1, 2, 3] = np.nan       # NaN in the bonus row
    Ld[2, 0, :] = -np.inf      # all -inf draft row
    D[3, 1] = 5                # token out of range
    out = O.verify(Lt, Ld, D, 1.0, 0, 0.5, seed=1)
    assert out["accepted_len"][0] >= 0
    for b in (1, 2, 3):
        assert out["accepted_len"][b] == -1
        assert np.all(out["tokens"][b] == -1)
        assert np.all(out["flags"][b] == O.FLAG_INVALID)


def test_sequence_offset_and_threads_do_not_change_results():
    rng = np.random.default_rng(8)
    B, k, V = 24, 3, 16
    Lt = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    Ld = (Lt[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    D = rng.integers(0, V, size=(B, k)).astype(np.int32)
    gate = (np.arange(B) % 2).astype(np.uint8)
    full = O.verify(Lt, Ld, D, 0.8, gate, 0.3, seed=99, nthreads=1)
    thr = O.verify(Lt, Ld, D, 0.8, gate, 0.3, seed=99, nthreads=5)
    for key in full:
        np.testing.assert_array_equal(full[key], thr[key])
    half = O.verify(Lt[12:], Ld[12:], D[12:], 0.8, gate[12:], 0.3, seed=99, seq_offset=12)
    for key in full:
        np.testing.assert_array_equal(full[key][12:], half[key])


def test_margin_reports_draws_near_a_boundary():
    p = np.array([0.5, 0.5])
    q = np.array([0.8, 0.2])
    Lt = np.log(np.stack([p, p])).astype(np.float32)[None]
    Ld = np.log(q).astype(np.float32)[None, None]
    P, Q = distributions(Lt[0], Ld[0], 1.0)
    ratio = P[0, 0] / Q[0, 0]
    near = O.verify(Lt, Ld, np.array([[0]]), 1.0, 0, 0.5, u0=np.array([[ratio + 3e-7]]),
                    u1=np.array([0.5]))
    far = O.verify(Lt, Ld, np.array([[0]]), 1.0, 0, 0.5, u0=np.array([[ratio + 0.1]]),
                   u1=np.array([0.5]))
    assert near["margin"][0] < 1e-6 and far["margin"][0] > 1e-3


# --------------------------------------------------- temperature 0 (greedy)

def _greedy_case(rng, B, k, V, ties=True):
    """Integer-valued logits (many exact ties) and drafted tokens that often
    equal a row's argmax."""
    Lt = rng.integers(-3, 4, size=(B, k + 1, V)).astype(np.float32)
    Ld = (Lt[:, :k] + rng.integers(-1, 2, size=(B, k, V))).astype(np.float32)
    if not ties:
        Lt += rng.permutation(V)[None, None, :].astype(np.float32) * 1e-3
        Ld += rng.permutation(V)[None, None, :].astype(np.float32) * 1e-3
    D = np.where(rng.random((B, k)) < 0.7, np.argmax(Lt[:, :k], axis=2),
                 np.where(rng.random((B, k)) < 0.5, np.argmax(Ld, axis=2),
                          rng.integers(0, V, size=(B, k)))).astype(np.int32)
    return Lt, Ld, D


@pytest.mark.parametrize("gated", [0, 1])
def test_greedy_is_the_argmax_chain(gated):
    # T = 0: p and q are one-hot at the first largest logit (numpy's argmax
    # convention), so the rule reduces to: NULL (gated) where D differs from
    # the draft argmax, reject where it differs from the target argmax, and
    # emit the target argmax of the stop row
    rng = np.random.default_rng(41 + gated)
    B, k, V = 400, 4, 9
    Lt, Ld, D = _greedy_case(rng, B, k, V)
    out = O.verify(Lt, Ld, D, 0.0, gated, 0.5, seed=5)
    tstar = np.argmax(Lt, axis=2)
    dstar = np.argmax(Ld, axis=2)
    for b in range(B):
        j = 0
        flags = []
        while j < k:
            if gated and D[b, j] != dstar[b, j]:
                flags.append(O.FLAG_NULL)
                break
            if D[b, j] != tstar[b, j]:
                flags.append(O.FLAG_REJECT)
                break
            flags.append(O.FLAG_ACCEPT)
            j += 1
        assert out["accepted_len"][b] == j
        assert list(out["tokens"][b, :j]) == list(D[b, :j])
        assert out["tokens"][b, j] == tstar[b, j]
        assert all(t == -1 for t in out["tokens"][b, j + 1:])
        assert list(out["flags"][b, :len(flags)]) == flags
        admitted = (D[b] == dstar[b]) if gated else np.ones(k, bool)
        assert np.array_equal(out["alpha"][b], (admitted & (D[b] == tstar[b, :k])).astype(float))


def test_greedy_ties_take_the_first_maximum():
    Lt = np.array([[[1.0, 3.0, 3.0, 2.0], [0.0, 5.0, 0.0, 5.0]]], dtype=np.float32)
    Ld = np.array([[[3.0, 3.0, 0.0, 0.0]]], dtype=np.float32)
    out = O.verify(Lt, Ld, np.array([[1]]), 0.0, 0, 0.5)
    assert out["accepted_len"][0] == 1 and list(out["tokens"][0]) == [1, 1]
    out = O.verify(Lt, Ld, np.array([[2]]), 0.0, 0, 0.5)
    assert out["accepted_len"][0] == 0 and list(out["tokens"][0]) == [1, -1]
    out = O.verify(Lt, Ld, np.array([[1]]), 0.0, 1, 0.5)  # draft argmax is token 0: NULL
    assert out["flags"][0, 0] == O.FLAG_NULL and list(out["tokens"][0]) == [1, -1]


@pytest.mark.parametrize("gated", [0, 1])
def test_greedy_is_the_low_temperature_limit(gated):
    # with every maximum ahead of the runner-up by at least 1e-3, T = 1e-7
    # makes every probability but the largest exp(-1e4): zero in double, so
    # the ordinary rule at that temperature must do what the greedy rule does
    rng = np.random.default_rng(7 + gated)
    Lt, Ld, D = _greedy_case(rng, 300, 3, 12, ties=False)
    g = O.verify(Lt, Ld, D, 0.0, gated, 0.5, seed=11)
    t = O.verify(Lt, Ld, D, 1e-7, gated, 0.5, seed=11)
    for key in ("accepted_len", "tokens", "flags"):
        assert np.array_equal(g[key], t[key]), key
    assert np.allclose(g["alpha"], t["alpha"], atol=1e-12)


# ------------------------------------------- gate policy: schedules, cumulative floor

def _policy_rows(qs, V=10):
    """One gated sequence whose drafted token at step j has draft probability
    exactly qs[j] (1/n for n equal logits, the rest -inf) and whose target rows
    equal its draft rows, so every admitted draft is accepted (alpha = 1) and
    the accepted length counts the drafts the gate retains."""
    k = len(qs)
    Ld = np.full((1, k, V), -np.inf, dtype=np.float32)
    for j, q in enumerate(qs):
        n = int(round(1.0 / q))
        assert abs(n * q - 1.0) < 1e-12
        Ld[0, j, :n] = 0.0
    Lt = np.concatenate([Ld, Ld[:, :1]], axis=1)  # bonus row: any valid row
    D = np.zeros((1, k), dtype=np.int32)
    return Lt, Ld, D


def _floats(text):
    return [float(x) for x in text.split(",")]


@pytest.mark.parametrize("row", range(8))
def test_gate_policy_worked_examples_retain_as_printed(row):
    rows = _golden_rows("gate_schedule_example.txt")
    kind, qs, sched, cum, want = rows[row]
    Lt, Ld, D = _policy_rows(_floats(qs))
    out = O.verify(Lt, Ld, D, 1.0, 1, 0.99, seed=3, tau_sched=_floats(sched), min_cum=float(cum))
    got = int(out["accepted_len"][0])
    if want.startswith(">="):
        assert got >= int(want[2:])
    else:
        assert got == int(want), (kind, qs, sched, cum)
    k = len(_floats(qs))
    if got < k:  # the failed gate is an explicit NULL row that ends the prefix
        assert out["flags"][0, got] == O.FLAG_NULL
        assert np.all(out["flags"][0, got + 1:] == O.FLAG_UNREACHED)
        assert out["alpha"][0, got] == 0.0
    assert np.all(out["flags"][0, :got] == O.FLAG_ACCEPT)


def test_gate_policy_cumulative_floor_just_above_a_product_fails():
    # the survival rows meet their floors exactly; the next double up fails
    Lt, Ld, D = _policy_rows([0.5, 0.5, 0.5])
    for floor, want in ((0.5, 0), (0.25, 1), (0.125, 2)):
        out = O.verify(Lt, Ld, D, 1.0, 1, 0.5, tau_sched=[0.0], min_cum=np.nextafter(floor, 1.0))
        assert out["accepted_len"][0] == want


def test_gate_policy_last_threshold_repeats():
    # schedule (0.1, 0.6): steps 2 and 3 use 0.6 as well
    Lt, Ld, D = _policy_rows([0.5, 1.0, 1.0, 0.5])
    out = O.verify(Lt, Ld, D, 1.0, 1, 0.99, tau_sched=[0.1, 0.6])
    assert out["accepted_len"][0] == 3 and out["flags"][0, 3] == O.FLAG_NULL
    out = O.verify(Lt, Ld, D, 1.0, 1, 0.99, tau_sched=[0.1, 0.6, 0.6, 0.5])
    assert out["accepted_len"][0] == 4


def test_gate_policy_floors_compose_by_logical_and():
    Lt, Ld, D = _policy_rows([0.5, 0.5, 0.5])
    # the step floor passes every step, the cumulative floor fails step 2
    assert O.verify(Lt, Ld, D, 1.0, 1, 0.5, tau_sched=[0.35], min_cum=0.2)["accepted_len"][0] == 2
    # the cumulative floor passes step 0 (0.25 >= 0.2), the step floor fails it
    Lt, Ld, D = _policy_rows([0.25, 1.0])
    assert O.verify(Lt, Ld, D, 1.0, 1, 0.5, tau_sched=[0.35], min_cum=0.2)["accepted_len"][0] == 0
    assert O.verify(Lt, Ld, D, 1.0, 1, 0.5, tau_sched=[0.2], min_cum=0.2)["accepted_len"][0] == 2


def test_gate_policy_cumulative_product_uses_draft_probabilities():
    # [R "schedule behavior"]: the prefix product is of the draft's own
    # probabilities of its drafted tokens; the target rows play no part in the
    # gate.  q_0(D_0) = q_1(D_1) = 1/2 while p_0(D_0) = 1/8: the floor 1/4 is
    # met exactly by the draft product at step 1 (equality passes) and would
    # be missed by the target's (1/16).  u0 = 0 accepts every admitted draft.
    V = 8
    Ld = np.full((1, 2, V), -np.inf, dtype=np.float32)
    Ld[0, :, :2] = 0.0
    Lt = np.zeros((1, 3, V), dtype=np.float32)
    D = np.zeros((1, 2), dtype=np.int32)
    out = O.verify(Lt, Ld, D, 1.0, 1, 0.5, tau_sched=[0.0], min_cum=0.25, u0=np.zeros((1, 2)),
                   u1=np.full(1, 0.5))
    assert out["accepted_len"][0] == 2
    assert list(out["flags"][0]) == [O.FLAG_ACCEPT, O.FLAG_ACCEPT]
    np.testing.assert_allclose(out["alpha"][0], [0.25, 0.25], rtol=0, atol=1e-15)


def test_gate_policy_special_cases_reduce_to_the_plain_and_flat_rules():
    rng = np.random.default_rng(77)
    B, k, V = 300, 4, 40
    Lt = (rng.standard_normal((B, k + 1, V)) * 2.5).astype(np.float32)
    Ld = (Lt[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    D = np.argmax(Ld + rng.gumbel(size=Ld.shape), axis=2).astype(np.int32)
    keys = ("accepted_len", "tokens", "flags", "alpha")
    # schedule 0 and floor 0: every token is admitted, mu = q -- plain mode
    a = O.verify(Lt, Ld, D, 1.0, 1, 0.9, seed=9, tau_sched=[0.0], min_cum=0.0)
    b = O.verify(Lt, Ld, D, 1.0, 0, 0.9, seed=9)
    for key in keys:
        assert np.array_equal(a[key], b[key]), key
    # a flat one-entry schedule overrides every sequence's own threshold
    a = O.verify(Lt, Ld, D, 1.0, 1, rng.uniform(0.05, 1.0, B), seed=9, tau_sched=[0.3])
    b = O.verify(Lt, Ld, D, 1.0, 1, 0.3, seed=9)
    for key in keys:
        assert np.array_equal(a[key], b[key]), key
    # a cumulative floor never admits more than the step floor alone
    a = O.verify(Lt, Ld, D, 1.0, 1, 0.3, seed=9, min_cum=0.05)
    assert np.all(a["accepted_len"] <= b["accepted_len"])
    # plain sequences ignore the policy
    a = O.verify(Lt, Ld, D, 1.0, 0, 0.3, seed=9, tau_sched=[0.9, 0.1], min_cum=0.5)
    c = O.verify(Lt, Ld, D, 1.0, 0, 0.3, seed=9)
    for key in keys:
        assert np.array_equal(a[key], c[key]), key


def _check_emits_p(law, P, tol=1e-10):
    k = P.shape[0] - 1
    reach, emit, _ = position_marginals(law, k, P.shape[1])
    assert abs(sum(law.values()) - 1.0) < tol
    for j in range(k + 1):
        if reach[j] > 1e-9:
            np.testing.assert_allclose(emit[j] / reach[j], P[j], atol=tol / reach[j])


@pytest.mark.parametrize("V,k,sched,cum", [(3, 2, [0.0], 0.2), (4, 3, [0.1, 0.3], 0.05),
                                           (4, 2, [0.25], 0.1), (5, 2, [0.3, 0.0], 0.0)])
def test_exact_law_is_lossless_under_gate_policy(V, k, sched, cum):
    # [S "Approach"]: keeping q on the admitted set, the failed gate as a NULL
    # row and the residual (p - mu)+ preserve p whatever the admitted set, as
    # long as it depends on the committed prefix only -- here the schedule and
    # the prefix product
    rng = np.random.default_rng(1000 * V + 100 * k + int(100 * cum))
    for trial in range(2):
        Lt, Ld = _random_case(rng, V, k, scale=1.5 + trial)
        law = exact_law(Lt, Ld, 1.0, True, 0.99, tau_sched=sched, min_cum=cum)
        P, _ = distributions(Lt, Ld, 1.0)
        _check_emits_p(law, P)


def test_exact_law_rejects_mu_without_the_cumulative_floor():
    # p = q on step 0 and step 1; step 1's admitted set shrinks when the
    # prefix product is low, and a mu that ignores it is no longer lossless
    p0 = np.array([0.45, 0.35, 0.2])
    p1 = np.array([0.6, 0.3, 0.1])
    q1 = np.array([0.7, 0.2, 0.1])
    Lt = np.log(np.stack([p0, p1, p1])).astype(np.float32)
    Ld = np.log(np.stack([p0, q1])).astype(np.float32)
    P, _ = distributions(Lt, Ld, 1.0)
    good = exact_law(Lt, Ld, 1.0, True, 0.99, tau_sched=[0.0], min_cum=0.2)
    _check_emits_p(good, P)
    bad = exact_law(Lt, Ld, 1.0, True, 0.99, tau_sched=[0.0], min_cum=0.2, rule=O.RULE_MU_STEP_ONLY)
    _, emit, _ = position_marginals(bad, 2, 3)
    reach, _, _ = position_marginals(bad, 2, 3)
    assert np.max(np.abs(emit[1] / reach[1] - P[1])) > 1e-3


def test_gate_policy_margin_covers_the_cumulative_decision():
    Lt, Ld, D = _policy_rows([0.5, 0.5])
    out = O.verify(Lt, Ld, D, 1.0, 1, 0.5, tau_sched=[0.0], min_cum=0.25 + 3e-7)
    assert out["margin"][0] < 1e-6 and out["accepted_len"][0] == 1
    out = O.verify(Lt, Ld, D, 1.0, 1, 0.5, tau_sched=[0.0], min_cum=0.3)
    assert out["margin"][0] > 1e-3


def test_gate_policy_bad_arguments_are_rejected():
    Lt, Ld, D = _policy_rows([0.5])
    for kw in (dict(tau_sched=[]), dict(min_cum=-0.1), dict(min_cum=1.5), dict(min_cum=np.nan)):
        with pytest.raises(ValueError):
            O.verify(Lt, Ld, D, 1.0, 1, 0.5, **kw)


# ------------------------------------------------- closed-form acceptance diagnostics

def test_diagnostics_reproduce_the_printed_ceiling_example():
    g = {r[0]: [float(x) for x in r[1:]] for r in _golden_rows("acceptance_ceiling_example.txt")}
    p, q = np.array(g["p"]), np.array(g["q"])
    with np.errstate(divide="ignore"):
        Lt = np.log(np.stack([p, p]))[None].astype(np.float32)
        Ld = np.log(q)[None, None].astype(np.float32)
    d = O.diagnostics(Lt, Ld, np.zeros((1, 1)), 1.0, 0, 0.5)
    assert abs(d["argmax_q"][0, 0] - g["argmax_q"][0]) < 1e-7
    assert abs(d["min_sum"][0, 0] - g["ceiling"][0]) < 1e-7
    assert abs(d["pq_sum"][0, 0] - g["sampler_match"][0]) < 1e-7


@pytest.mark.parametrize("gated,tau,sched", [(False, 0.5, None), (True, 0.3, None), (True, 0.99, [0.2, 0.0])])
def test_diagnostics_are_the_exact_pass_rates_of_the_three_rules(gated, tau, sched):
    # without a cumulative floor mu_j does not depend on the prefix, so the
    # enumerated law's pass rate at every reached position is the closed form
    rng = np.random.default_rng(31 + int(gated) + (sched is not None))
    V, k = 4, 2
    Lt, Ld = _random_case(rng, V, k, scale=1.5)
    d = O.diagnostics(Lt[None], Ld[None], np.zeros((1, k)), 1.0, int(gated), tau, tau_sched=sched)
    for rule, key in ((O.RULE_MU, "min_sum"), (O.RULE_ARGMAX, "argmax_q")):
        g, t = (gated, tau) if rule == O.RULE_MU else (False, 0.5)
        law = exact_law(Lt, Ld, 1.0, g, t, rule=rule, tau_sched=sched if rule == O.RULE_MU else None)
        reach, _, passed = position_marginals(law, k, V)
        for j in range(k):
            assert abs(passed[j] / reach[j] - d[key][0, j]) < 1e-9, (key, j)
    # sampler-match draws a fresh target token with u0: its pass rate at step 0
    # over the cells of u0 cut at p_0's cumulative sums, for every draft D_0
    P, Q = distributions(Lt, Ld, 1.0)
    edges = np.concatenate([[0.0], np.cumsum(P[0])])
    edges[-1] = 1.0
    mids, vols = 0.5 * (edges[:-1] + edges[1:]), np.diff(edges)
    keep = vols > 0
    mids, vols = mids[keep], vols[keep]
    n = V * len(mids)
    D = np.zeros((n, k), dtype=np.int32)
    D[:, 0] = np.repeat(np.arange(V), len(mids))
    u0 = np.full((n, k), 0.5)
    u0[:, 0] = np.tile(mids, V)
    out = O.verify(np.broadcast_to(Lt, (n, k + 1, V)), np.broadcast_to(Ld, (n, k, V)), D, 1.0, 0, 0.5,
                   u0=u0, u1=np.full(n, 0.5), rule=O.RULE_SAMPLER_MATCH)
    acc = (out["accepted_len"] >= 1).astype(float)
    rate = float((acc * np.tile(vols, V) * np.repeat(Q[0], len(mids))).sum())
    assert abs(rate - d["pq_sum"][0, 0]) < 1e-12


@pytest.mark.parametrize("sched,cum", [([0.0], 0.2), ([0.1, 0.3], 0.1), (None, 0.3)])
def test_diagnostics_min_sum_is_the_mean_acceptance_probability(sched, cum):
    # E over D_j ~ q_j of the oracle's alpha_j, the drafted prefix held fixed,
    # is sum_x min(p_j, mu_j) -- also with a cumulative floor, whose mu_j
    # depends on the prefix
    rng = np.random.default_rng(int(100 * cum) + len(sched or []))
    V, k = 6, 3
    Lt, Ld = _random_case(rng, V, k, scale=1.5)
    _, Q = distributions(Lt, Ld, 1.0)
    prefix = rng.integers(0, V, size=k)
    d = O.diagnostics(Lt[None], Ld[None], prefix[None], 1.0, 1, 0.4, tau_sched=sched, min_cum=cum)
    for j in range(k):
        D = np.broadcast_to(prefix, (V, k)).copy()
        D[:, j] = np.arange(V)
        a = O.verify(np.broadcast_to(Lt, (V, k + 1, V)), np.broadcast_to(Ld, (V, k, V)), D, 1.0, 1, 0.4,
                     tau_sched=sched, min_cum=cum)["alpha"][:, j]
        assert abs((Q[j] * a).sum() - d["min_sum"][0, j]) < 1e-12


def test_diagnostics_plain_ceiling_is_one_minus_total_variation():
    rng = np.random.default_rng(3)
    B, k, V = 20, 3, 50
    Lt = (rng.standard_normal((B, k + 1, V)) * 2).astype(np.float32)
    Ld = (Lt[:, :k] + rng.standard_normal((B, k, V))).astype(np.float32)
    d = O.diagnostics(Lt, Ld, np.zeros((B, k)), 0.8, 0, 0.5, nthreads=4)
    P = softmax(Lt[:, :k].astype(np.float64) / 0.8, axis=-1)
    Q = softmax(Ld.astype(np.float64) / 0.8, axis=-1)
    np.testing.assert_allclose(d["min_sum"], 1.0 - 0.5 * np.abs(P - Q).sum(-1), atol=1e-12)
    # min(a, b) >= a b on [0, 1]: rejection sampling accepts at least as often as sampler-match
    assert np.all(d["min_sum"] >= d["pq_sum"] - 1e-15)
    assert np.all(d["min_sum"] <= 1.0 + 1e-12)


def test_diagnostics_argmax_rule_takes_the_first_largest_target_probability():
    # [M] "The acceptance ceiling": the argmax rule accepts with q(argmax p);
    # among equal largest p the first token is its argmax (the greedy tie rule)
    with np.errstate(divide="ignore"):
        Lt = np.log(np.array([[0.4, 0.4, 0.2], [0.4, 0.4, 0.2]]))[None].astype(np.float32)
        Ld = np.log(np.array([[0.1, 0.6, 0.3]]))[None].astype(np.float32)
    d = O.diagnostics(Lt, Ld, np.zeros((1, 1), dtype=np.int32), 1.0, 0, 0.5)
    assert abs(d["argmax_q"][0, 0] - 0.1) < 1e-7
    # the argmax control rule accepts only the first largest token
    out = O.verify(Lt, Ld, np.array([[1]], dtype=np.int32), 1.0, 0, 0.5, rule=O.RULE_ARGMAX)
    assert out["accepted_len"][0] == 0 and out["tokens"][0, 0] == 0
    out = O.verify(Lt, Ld, np.array([[0]], dtype=np.int32), 1.0, 0, 0.5, rule=O.RULE_ARGMAX)
    assert out["accepted_len"][0] == 1 and list(out["tokens"][0]) == [0, 0]


def test_diagnostics_greedy_and_invalid_rows():
    Lt = np.array([[[0.0, 2.0, 1.0], [1.0, 0.0, 0.0], [0.0, 0.0, 0.0]]], dtype=np.float32)
    Ld = np.array([[[0.0, 3.0, 0.0], [0.0, 1.0, 0.0]]], dtype=np.float32)
    d = O.diagnostics(Lt, Ld, np.array([[1, 0]]), 0.0, 0, 0.5)
    # one-hot p and q: the argmaxes agree at step 0 (token 1), differ at step 1
    assert list(d["min_sum"][0]) == [1.0, 0.0] and list(d["pq_sum"][0]) == [1.0, 0.0]
    assert list(d["argmax_q"][0]) == [1.0, 0.0]
    bad = Lt.copy()
    bad[0, 1, 2] = np.nan
    d = O.diagnostics(bad, Ld, np.array([[1, 0]]), 1.0, 1, 0.3, tau_sched=[0.0], min_cum=0.1)
    assert np.isfinite(d["min_sum"][0, 0]) and np.isnan(d["min_sum"][0, 1])
    # a drafted token out of range poisons the cumulative product behind it
    d = O.diagnostics(Lt, Ld, np.array([[7, 0]]), 1.0, 1, 0.3, tau_sched=[0.0], min_cum=0.1)
    assert np.isfinite(d["pq_sum"][0, 0]) and np.isnan(d["pq_sum"][0, 1])
    d = O.diagnostics(Lt, Ld, np.array([[7, 0]]), 1.0, 1, 0.3)
    assert np.all(np.isfinite(d["pq_sum"]))


# ------------------------------------------------------------ sampler filters

def test_filter_examples_worked_by_hand():
    p = np.array([0.5, 0.3, 0.15, 0.05])
    L = np.log(p).astype(np.float32)
    rows = _golden_rows("filter_examples.txt")
    assert len(rows) == 10
    for r in rows:
        top_k, top_p, min_p = int(r[0]), float(r[1]), float(r[2])
        want = np.array([float(x) for x in r[3:]])
        got, margin = O.filtered_row(L, 1.0, top_k, top_p, min_p)
        np.testing.assert_allclose(got, want, atol=1e-6, err_msg=str(r[:3]))
        assert margin > 1e-3  # no example sits on a boundary


def test_filters_keep_ties_and_follow_the_chain_order():
    # ties at the top-k boundary are kept
    L = np.array([2.0, 1.0, 1.0, 0.0], dtype=np.float32)
    got, _ = O.filtered_row(L, 1.0, 2, 1.0, 0.0)
    e = np.exp([2.0, 1.0, 1.0])
    np.testing.assert_allclose(got, np.append(e / e.sum(), 0.0), atol=1e-12)
    # top-p sees the top-k survivors renormalised: p = (0.5, 0.3, 0.15, 0.05)
    # with top_k = 2 gives (0.625, 0.375), so top_p = 0.6 keeps one token,
    # while on the full row 0.6 would keep two
    L = np.log(np.array([0.5, 0.3, 0.15, 0.05])).astype(np.float32)
    assert np.count_nonzero(O.filtered_row(L, 1.0, 2, 0.6, 0.0)[0]) == 1
    assert np.count_nonzero(O.filtered_row(L, 1.0, 0, 0.6, 0.0)[0]) == 2
    # min_p = 1 keeps the largest only; filters off leave the softmax as is
    assert np.count_nonzero(O.filtered_row(L, 1.0, 0, 1.0, 1.0)[0]) == 1
    p0, _, _, _ = O.softmax_row(L, 1.3)
    np.testing.assert_array_equal(O.filtered_row(L, 1.3, 0, 1.0, 0.0)[0], p0)


def test_top_p_keeps_the_prefix_whose_mass_reaches_top_p_exactly():
    # [M] "What changed", as read here: top-p keeps the shortest prefix, in decreasing
    # probability, whose mass reaches top_p.  With top_p chosen so that
    # top_p * (total mass) equals the first token's probability exactly in
    # double, the first token alone reaches it; the next top_p up needs two.
    L = np.array([1.5, 0.25, -0.5, -2.0], dtype=np.float32)
    p, _, _, _ = O.softmax_row(L, 1.0)
    total = 0.0
    for v in np.argsort(-L, kind="stable"):  # decreasing logit, the filter's order
        total += p[v]
    tp = p[0] / total
    for _ in range(8):  # a few ulps either way until the product is exact
        if tp * total == p[0]:
            break
        tp = np.nextafter(tp, 1.0 if tp * total < p[0] else 0.0)
    assert tp * total == p[0]
    got, margin = O.filtered_row(L, 1.0, 0, tp, 0.0)
    assert np.count_nonzero(got) == 1 and got[0] == 1.0
    assert margin == 0.0  # the decision sits on its boundary
    up = np.nextafter(tp, 1.0)
    while up * total <= p[0]:
        up = np.nextafter(up, 1.0)
    assert np.count_nonzero(O.filtered_row(L, 1.0, 0, up, 0.0)[0]) == 2


def test_filtered_target_support_is_never_violated():
    # [M "Where chi-square is blind"]: a top_k = 2 target against an
    # unfiltered drafter must never emit (or accept) a token outside the
    # target's two-token support
    rng = np.random.default_rng(12)
    n, k, V = 3000, 3, 6
    Lt = (rng.standard_normal((k + 1, V)) * 1.5).astype(np.float32)
    Ld = (rng.standard_normal((k, V)) * 1.5).astype(np.float32)
    _, Q = distributions(Lt, Ld, 1.0)
    D = np.stack([rng.choice(V, size=n, p=Q[j]) for j in range(k)], axis=1).astype(np.int32)
    filt = ((2, 1.0, 0.0), (0, 1.0, 0.0))
    out = O.verify(np.broadcast_to(Lt, (n, k + 1, V)), np.broadcast_to(Ld, (n, k, V)), D, 1.0, 0, 0.5,
                   seed=3, nthreads=4, filters=filt)
    support = [set(np.argsort(-Lt[j])[:2]) for j in range(k + 1)]
    for b in range(n):
        a = out["accepted_len"][b]
        for j in range(a + 1):
            assert out["tokens"][b, j] in support[j], (b, j)


@pytest.mark.parametrize("filt", [((2, 1.0, 0.0), (0, 1.0, 0.0)), ((0, 0.7, 0.0), (3, 1.0, 0.0)),
                                  ((3, 0.9, 0.1), (2, 0.8, 0.0)), ((0, 1.0, 0.3), (0, 1.0, 0.2))])
@pytest.mark.parametrize("gated", [False, True])
def test_exact_law_is_lossless_with_filtered_distributions(filt, gated):
    # modified rejection sampling preserves whatever p it is given: the
    # emitted marginals equal the filtered target rows, drafts drawn from the
    # filtered draft rows
    rng = np.random.default_rng(5 + int(gated) + 10 * filt[0][0])
    Lt, Ld = _random_case(rng, 5, 2, scale=1.5)
    law = exact_law(Lt, Ld, 1.0, gated, 0.3, filters=filt)
    P, _ = distributions(Lt, Ld, 1.0, filt)
    _check_emits_p(law, P)


def test_top_k_one_is_greedy_and_filters_off_change_nothing():
    rng = np.random.default_rng(8)
    B, k, V = 200, 3, 12
    Lt, Ld, D = _greedy_case(rng, B, k, V, ties=False)
    for gated in (0, 1):
        g = O.verify(Lt, Ld, D, 0.0, gated, 0.5, seed=4)
        f = O.verify(Lt, Ld, D, 0.9, gated, 0.5, seed=4, filters=((1, 1.0, 0.0), (1, 1.0, 0.0)))
        for key in ("accepted_len", "tokens", "flags", "alpha"):
            assert np.array_equal(g[key], f[key]), key
    a = O.verify(Lt, Ld, D, 0.9, 1, 0.5, seed=4)
    b = O.verify(Lt, Ld, D, 0.9, 1, 0.5, seed=4, filters=((0, 1.0, 0.0), (0, 1.0, 0.0)))
    for key in ("accepted_len", "tokens", "flags", "alpha", "margin"):
        assert np.array_equal(a[key], b[key]), key


def test_filter_margin_reports_top_p_and_min_p_boundaries():
    L = np.log(np.array([0.5, 0.3, 0.15, 0.05])).astype(np.float32)
    assert O.filtered_row(L, 1.0, 0, 0.8 + 1e-8, 0.0)[1] < 1e-6   # 0.5 + 0.3 reaches 0.8
    assert O.filtered_row(L, 1.0, 0, 1.0, 0.3 + 1e-8)[1] < 1e-6   # 0.15 / 0.5 = 0.3
    with pytest.raises(ValueError):
        O.verify(L[None, None].repeat(2, 1), L[None, None], np.zeros((1, 1)), 1.0, 0, 0.5,
                 filters=((0, 0.0, 0.0), (0, 1.0, 0.0)))


def test_filtered_row_statistics_and_diagnostics():
    # row_stats of a filtered row: max and log-sum-exp of L/T over the
    # survivors (scipy's logsumexp); the diagnostics' sum min(p, q) is the
    # mean acceptance probability over drafts drawn from the filtered q
    rng = np.random.default_rng(21)
    V, k = 7, 2
    Lt, Ld = _random_case(rng, V, k, scale=1.5)
    filt = ((3, 0.9, 0.0), (0, 0.8, 0.05))
    out = O.verify(Lt[None], Ld[None], np.zeros((1, k), np.int32), 0.8, 0, 0.5, filters=filt)
    for j in range(k + 1):
        p, _ = O.filtered_row(Lt[j], 0.8, *filt[0])
        kept = p > 0
        assert abs(out["row_stats"][0, j, 1] - logsumexp(Lt[j][kept].astype(np.float64) / 0.8)) < 1e-12
    P, Q = distributions(Lt, Ld, 0.8, filt)
    prefix = np.array([int(np.argmax(Q[0])), 0])
    d = O.diagnostics(Lt[None], Ld[None], prefix[None], 0.8, 0, 0.5, filters=filt)
    for j in range(k):
        D = np.broadcast_to(prefix, (V, k)).copy()
        D[:, j] = np.arange(V)
        a = O.verify(np.broadcast_to(Lt, (V, k + 1, V)), np.broadcast_to(Ld, (V, k, V)), D, 0.8, 0, 0.5,
                     filters=filt)["alpha"][:, j]
        assert abs((Q[j] * a).sum() - d["min_sum"][0, j]) < 1e-12


# ------------------------------------------- pick intervals (judging near-boundary picks)

def test_pick_interval_of_the_worked_example():
    # Strata PR #3416, "Problem and result": p = (1/2, 1/2), q = (7/8, 1/8),
    # threshold 1/2.  Stopping at position 0 the residual (p - mu)+ with
    # mu = (7/8, 0) is (0, 1/2): token 1 takes all of [0, 1), token 0 nothing;
    # the bonus row is p itself.
    Lt, Ld = _worked_example_rows()
    w0, lo0, hi0, _ = O.pick_interval(Lt, Ld, np.array([0]), 1.0, 1, 0.5, 0, 0)
    w1, lo1, hi1, gm = O.pick_interval(Lt, Ld, np.array([0]), 1.0, 1, 0.5, 0, 1)
    assert (w0, w1) == (0.0, 1.0) and (lo1, hi1) == (0.0, 1.0) and lo0 == hi0 == 0.0
    assert abs(gm - 0.375) < 1e-9  # the closer of q = 7/8 and 1/8 to the threshold 1/2
    wb, lob, hib, gmb = O.pick_interval(Lt, Ld, np.array([0]), 1.0, 1, 0.5, 1, 1)
    assert abs(wb - 0.5) < 1e-12 and abs(lob - 0.5) < 1e-12 and hib == 1.0 and gmb == np.inf


def _worked_example_rows():
    p = np.array([0.5, 0.5])
    q = np.array([0.875, 0.125])
    return np.log(np.stack([p, p])).astype(np.float32), np.log(q)[None].astype(np.float32)


PICK_CASES = [
    # (V, k, T, gate, tau, sched, cum, filters)
    (40, 3, 1.0, 0, 0.5, None, 0.0, None),
    (40, 3, 0.7, 1, 0.3, None, 0.0, None),
    (9, 2, 1.3, 1, 0.2, None, 0.0, None),
    (60, 4, 1.0, 1, 0.5, [0.25, 0.1], 0.02, None),
    (50, 2, 0.8, 0, 0.5, None, 0.0, ((5, 0.9, 0.0), (0, 0.95, 0.05))),
    (30, 3, 0.0, 1, 0.5, None, 0.0, None),
]


@pytest.mark.parametrize("case", range(len(PICK_CASES)))
def test_pick_interval_holds_the_oracles_own_pick(case):
    # A separately written restatement of the stop row's weights: for every
    # sequence the emitted token's interval has weight and holds u1 (the same
    # u1 the oracle drew), at the oracle's own stop position.
    V, k, T, gate, tau, sched, cum, filt = PICK_CASES[case]
    rng = np.random.default_rng(100 + case)
    B = 60
    Lt = (rng.normal(size=(B, k + 1, V)) * 2.0).astype(np.float32)
    Ld = (Lt[:, :k] + rng.normal(size=(B, k, V))).astype(np.float32)
    if T == 0.0:
        Lt = np.round(Lt).astype(np.float32)
        Ld = np.round(Ld).astype(np.float32)
    D = rng.integers(0, V, size=(B, k)).astype(np.int32)
    # drafts often at a row's largest draft logit, so that gates pass and chains run on
    D = np.where(rng.random((B, k)) < 0.6, np.argmax(Ld, axis=2), D).astype(np.int32)
    out = O.verify(Lt, Ld, D, T, gate, tau, seed=77, tau_sched=sched, min_cum=cum, filters=filt)
    for b in range(B):
        j = int(out["accepted_len"][b])
        v = int(out["tokens"][b, j])
        u1 = O.uniform(77, b, j, 1)
        w, lo, hi, _ = O.pick_interval(Lt[b], Ld[b], D[b], T, gate, tau, j, v, tau_sched=sched,
                                       min_cum=cum, filters=filt)
        assert w > 0.0, (b, j, v)
        if T > 0.0:
            assert lo - 1e-12 <= u1 < hi + 1e-12, (b, j, v, u1, lo, hi)


@pytest.mark.parametrize("gate,j", [(0, 0), (1, 1), (1, 3)])
def test_pick_intervals_tile_the_unit_interval(gate, j):
    rng = np.random.default_rng(5 + j)
    V, k = 25, 3
    Lt = (rng.normal(size=(k + 1, V)) * 2.0).astype(np.float32)
    Ld = (Lt[:k] + rng.normal(size=(k, V))).astype(np.float32)
    D = np.argmax(Ld, axis=1).astype(np.int32)
    iv = [O.pick_interval(Lt, Ld, D, 1.0, gate, 0.2, j, v) for v in range(V)]
    w = np.array([x[0] for x in iv])
    lo = np.array([x[1] for x in iv])
    hi = np.array([x[2] for x in iv])
    assert abs(w.sum() - 1.0) < 1e-12 and lo[0] == 0.0 and abs(hi[-1] - 1.0) < 1e-12
    np.testing.assert_allclose(lo[1:], hi[:-1], rtol=0, atol=1e-15)
    np.testing.assert_allclose(hi - lo, w, rtol=0, atol=1e-15)
    if j == k:  # the bonus row: the weights are p_k itself
        np.testing.assert_allclose(w, softmax(Lt[k].astype(np.float64)), rtol=1e-12, atol=1e-15)


def test_pick_interval_rejects_bad_arguments():
    Lt, Ld = _worked_example_rows()
    for j, v in ((-1, 0), (2, 0), (0, 2), (0, -1)):
        with pytest.raises(ValueError):
            O.pick_interval(Lt, Ld, np.array([0]), 1.0, 1, 0.5, j, v)
    bad = Lt.copy()
    bad[0, 0] = np.nan
    with pytest.raises(ValueError):
        O.pick_interval(bad, Ld, np.array([0]), 1.0, 1, 0.5, 0, 1)
