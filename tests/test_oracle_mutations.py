"""Do the oracle's pins catch plausible mistakes?

Each case below plants one mistake in a copy of ``oracle/spec_verify_oracle.c``
(a dropped term, a wrong comparison, a transposed operand, a wrong row or
constant), builds the copy, and runs the oracle pin suite (``test_oracle.py``
and ``test_metrics.py``) against it in a fresh process; at least one pin must
fail.  The unmutated copy, built the same way, must pass them all, so a
mutant's failure comes from its mistake and not from the harness.  Nothing
here touches the committed oracle or the CUDA library.
"""
from __future__ import annotations

import os
import shutil
import subprocess
import sys
from concurrent.futures import ThreadPoolExecutor

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
ORACLE = os.path.join(ROOT, "oracle")
SOURCE = os.path.join(ORACLE, "spec_verify_oracle.c")

# name -> [(text in the oracle source, replacement), ...]; every text occurs once
MUTATIONS = {
    # the gate: equality must pass (admit iff q(D) >= tau)
    "gate_strict": [("if (!(qv >= tau_j)) return 0;", "if (!(qv > tau_j)) return 0;")],
    # the accept test: the p(D) > 0 conjunct dropped
    "accept_without_support": [("if (pj[d] > 0.0 && u * md <= pj[d]) {", "if (u * md <= pj[d]) {")],
    # the accept test with p and mu transposed
    "accept_transposed": [("if (pj[d] > 0.0 && u * md <= pj[d]) {",
                           "if (pj[d] > 0.0 && u * pj[d] <= md) {")],
    # mu renormalised over the admitted set for the method itself
    "mu_renormalised": [("if (J->rule == ORACLE_RULE_RENORM_MU && kept > 0.0)", "if (kept > 0.0)")],
    # the gated residual built from q instead of mu
    "residual_from_q": [("if (J->rule == ORACLE_RULE_ORIGINAL_GATE || J->rule == ORACLE_RULE_RESIDUAL_Q) {",
                         "if (1) {")],
    # the residual keeps the negative part of p - mu
    "residual_abs": [("S->r[v] = d > 0.0 ? d : 0.0;", "S->r[v] = fabs(d);")],
    # a NULL row that does not end the chain
    "null_continues": [("        fl[j] = ORACLE_FLAG_NULL;\n        jstar = j;\n        break;\n      }\n    }\n"
                        "    retained_measure",
                        "        fl[j] = ORACLE_FLAG_NULL;\n        continue;\n      }\n    }\n"
                        "    retained_measure")],
    # the bonus (and p-resampling) sample taken from target row 0
    "bonus_from_row0": [("(and the p-resampling controls) */\n      memcpy(S->r, pst, (size_t)V * sizeof(double));",
                         "(and the p-resampling controls) */\n      memcpy(S->r, S->P, (size_t)V * sizeof(double));")],
    # a NULL position reports the unfiltered ratio instead of 0
    "null_alpha": [("a = 0.0; /* explicit NULL row */", "a = qd > 0.0 ? fmin(1.0, pd / qd) : 0.0;")],
    # the cumulative gate multiplies target instead of draft probabilities
    "cumulative_uses_p": [("cprev[j + 1] = cprev[j] * S->Q[(int64_t)j * V + Db[j]];",
                           "cprev[j + 1] = cprev[j] * S->P[(int64_t)j * V + Db[j]];")],
    # the inverse CDF with a non-strict comparison (zero-weight tokens pickable)
    "inverse_cdf_nonstrict": [("if (upto > y) {", "if (upto >= y) {")],
    # the temperature left out of the softmax
    "no_temperature": [("double xs = x / T;", "double xs = x;"),
                       ("double e = exp(logit_at(logits, dt, v) / T - m);",
                        "double e = exp(logit_at(logits, dt, v) - m);")],
    # Philox with nine rounds
    "philox_9_rounds": [("for (int round = 0; round < 10; ++round) {", "for (int round = 0; round < 9; ++round) {")],
    # Philox with the first Weyl constant on both key words
    "philox_key_schedule": [("k1 += weyl1;", "k1 += weyl0;")],
    # the uniform from 23 bits
    "uniform_23_bits": [("(double)(out[0] >> 8) * (1.0 / 16777216.0)", "(double)(out[0] >> 9) * (1.0 / 8388608.0)")],
    # the diagnostics' ceiling as sum max instead of sum min
    "diagnostics_sum_max": [("smin += fmin(pj[v], S->mu[v]);", "smin += fmax(pj[v], S->mu[v]);")],
    # top-p keeping the prefix that passes top_p strictly
    "top_p_strict": [("if (c >= target) {", "if (c > target) {")],
    # greedy rows one-hot at the last of equal largest logits
    "greedy_last_max": [("      if (x > m) {\n        m = x;\n        best = v;",
                         "      if (x >= m) {\n        m = x;\n        best = v;")],
    # the argmax rule and diagnostics taking the last largest p
    "argmax_last": [("if (p[v] > p[best]) best = v;", "if (p[v] >= p[best]) best = v;")],
    # the argmax rule's acceptance read from p instead of q
    "diagnostics_argmax_reads_p": [("J->diag_argq[o] = qj[argmax_first(pj, V)];",
                                    "J->diag_argq[o] = pj[argmax_first(pj, V)];")],
    # sampler-match's acceptance summed against mu instead of q
    "diagnostics_pq_uses_mu": [("spq += pj[v] * qj[v];", "spq += pj[v] * S->mu[v];")],
    # top-k dropping the tokens tied with its boundary token
    "top_k_drops_ties": [("keep[rk[i].v] = rk[i].x >= xk;", "keep[rk[i].v] = i < top_k;")],
    # min-p with a strict comparison
    "min_p_strict": [("if (!(ratio >= min_p)) keep[rk[i].v] = 0;", "if (!(ratio > min_p)) keep[rk[i].v] = 0;")],
    # a residual with no mass not reported as degenerate
    "degenerate_unreported": [("if (J->degenerate) J->degenerate[b] = 1;", "if (J->degenerate) J->degenerate[b] = 0;")],
    # the accept uniforms keyed on the local sequence index, without the offset
    "sequence_offset_ignored": [("return oracle_uniform(J->seed, J->seq_offset + (uint64_t)b, (uint32_t)j, 0u);",
                                 "return oracle_uniform(J->seed, (uint64_t)b, (uint32_t)j, 0u);")],
    # the pick interval's upper end without the token's own weight
    "pick_interval_without_own_weight": [("*hi = (below + mu[v]) / Z;", "*hi = below / Z;")],
    # the pick interval's gated residual built from q instead of mu
    "pick_interval_residual_from_q": [("retained_measure(&J, gated, tau_j, cprev, qi, mu);",
                                       "memcpy(mu, qi, (size_t)V * sizeof(double));")],
    # position and draw swapped in the Philox counter
    "counter_words_swapped": [("uint32_t ctr[4] = {(uint32_t)seq, pos, draw, (uint32_t)(seq >> 32)};",
                               "uint32_t ctr[4] = {(uint32_t)seq, draw, pos, (uint32_t)(seq >> 32)};")],
}


def _build(tmp_path, name, edits):
    with open(SOURCE) as f:
        src = f.read()
    for old, new in edits:
        assert src.count(old) == 1, (name, old)
        src = src.replace(old, new)
    d = tmp_path / name
    d.mkdir()
    c_file = d / "spec_verify_oracle.c"
    c_file.write_text(src)
    shutil.copy(os.path.join(ORACLE, "spec_verify_oracle.h"), d)
    lib = d / "liboracle_mutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared",
                    str(c_file), "-o", str(lib), "-lm", "-lpthread"], check=True)
    return str(lib)


def _pins(lib):
    from oracle import oracle as O
    env = dict(os.environ, **{O.LIBRARY_OVERRIDE_ENV: lib})
    return subprocess.run([sys.executable, "-m", "pytest", "-x", "-q", "-m", "not gpu", "-p", "no:cacheprovider",
                           os.path.join(HERE, "test_oracle.py"), os.path.join(HERE, "test_metrics.py")],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


@pytest.fixture(scope="module")
def results(tmp_path_factory):
    """Build every copy and run the pins against it, several at a time."""
    if shutil.which("gcc") is None:
        pytest.skip("gcc not found")
    base = tmp_path_factory.mktemp("mutants")
    names = ["unmutated"] + sorted(MUTATIONS)

    def one(name):
        return _pins(_build(base, name, MUTATIONS.get(name, [])))

    with ThreadPoolExecutor(max_workers=max(2, min(8, os.cpu_count() or 2))) as ex:
        futures = {name: ex.submit(one, name) for name in names}
        return {name: f.result() for name, f in futures.items()}


def test_unmutated_copy_passes_every_pin(results):
    r = results["unmutated"]
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]


@pytest.mark.parametrize("name", sorted(MUTATIONS))
def test_planted_mistake_fails_a_pin(results, name):
    r = results[name]
    # 1 = a test failed (not a collection error, a crash or a timeout)
    assert r.returncode == 1, f"{name}: pins returned {r.returncode}\n" + r.stdout[-3000:] + r.stderr[-2000:]
