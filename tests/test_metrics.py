"""Acceptance summary over the batch counters (metrics.py): the page's printed
summary line, the line format, and -- on oracle outputs -- that acceptance per
tested position is the quantity the closed form sum_x min(p, q) predicts,
while accepted / proposed is not."""
from __future__ import annotations

import math
import os

import numpy as np
import pytest

from oracle import oracle as O
from speculative_decoding_verification_online_gb300 import metrics

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _golden():
    vals = {}
    with open(os.path.join(GOLDEN, "acceptance_summary_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                key, value = line.split()
                vals[key] = float(value) if "." in value else int(value)
    return vals


def _counters(tested=0, accepted=0, null=0, rejected=0, bonus=0, boundary=0, invalid=0, degenerate=0):
    return [tested, accepted, null, rejected, bonus, boundary, invalid, degenerate]


def test_printed_summary_line_is_reproduced():
    g = _golden()
    k = g["proposed"] // g["rounds"]
    assert k * g["rounds"] == g["proposed"]
    s = metrics.acceptance_summary(_counters(tested=g["positions_tested"], accepted=g["accepted"]),
                                   rounds=g["rounds"], k=k)
    assert s["proposed"] == g["proposed"]
    for key in ("per_position_acceptance", "acceptance_rate", "mean_accepted_len"):
        assert round(s[key], 4) == g[key], key
    parsed = metrics.parse_summary_line(metrics.summary_line(s))
    assert parsed["rule"] == "stochastic"
    for key in ("rounds", "proposed", "positions_tested", "accepted"):
        assert parsed[key] == g[key]
    for key in ("per_position_acceptance", "acceptance_rate", "mean_accepted_len"):
        assert parsed[key] == g[key]


def test_invalid_sequences_leave_the_denominators_and_empty_counts_give_nan():
    s = metrics.acceptance_summary(_counters(tested=6, accepted=4, invalid=2), rounds=5, k=3)
    assert (s["rounds"], s["proposed"], s["invalid"]) == (3, 9, 2)
    assert s["mean_accepted_len"] == pytest.approx(4 / 3)
    e = metrics.acceptance_summary(_counters(), rounds=0, k=4)
    assert math.isnan(e["per_position_acceptance"]) and math.isnan(e["mean_accepted_len"])
    line = metrics.summary_line(e)
    assert "per_position_acceptance=nan" in line
    assert math.isnan(metrics.parse_summary_line(line)["acceptance_rate"])


@pytest.mark.parametrize("bad", [
    dict(counters=_counters(tested=10, accepted=11), rounds=5, k=4),   # accepted > tested
    dict(counters=_counters(tested=21, accepted=1), rounds=5, k=4),    # tested > proposed
    dict(counters=_counters(invalid=6), rounds=5, k=4),
    dict(counters=_counters()[:7], rounds=5, k=4),
    dict(counters=_counters(tested=-1), rounds=5, k=4),
    dict(counters=_counters(), rounds=5, k=0),
])
def test_inconsistent_counters_are_rejected(bad):
    with pytest.raises(ValueError):
        metrics.acceptance_summary(**bad)


def test_rule_ids():
    assert metrics.rule_id(0.0, False) == "greedy-argmax"
    assert metrics.rule_id(0.0, True) == "greedy-argmax"
    assert metrics.rule_id(0.7, False) == "stochastic"
    assert metrics.rule_id(1.0, True) == "stochastic-mu-null"


def _oracle_counters(ref, k):
    length = ref["accepted_len"]
    valid = length >= 0
    return _counters(tested=int(np.minimum(length[valid] + 1, k).sum()),
                     accepted=int(length[valid].sum()),
                     null=int((ref["flags"] == 3).sum()), rejected=int((ref["flags"] == 2).sum()),
                     bonus=int((length == k).sum()), invalid=int((~valid).sum()),
                     degenerate=int(np.asarray(ref["degenerate"]).sum()))


def test_per_tested_position_acceptance_meets_the_closed_form_and_the_rate_does_not():
    # the same target and draft rows at every position ("fixed logits"), drafts
    # drawn from q: each tested position accepts with probability sum min(p, q)
    # whatever happened before it, so accepted / tested estimates that closed
    # form; accepted / proposed counts untested positions and falls short
    rng = np.random.default_rng(5)
    B, k, V = 20000, 4, 6
    lt = rng.normal(0.0, 1.5, V)
    ld = lt + rng.normal(0.0, 1.0, V)
    p = np.exp(lt - lt.max()); p /= p.sum()
    q = np.exp(ld - ld.max()); q /= q.sum()
    Lt = np.broadcast_to(lt.astype(np.float32), (B, k + 1, V)).copy()
    Ld = np.broadcast_to(ld.astype(np.float32), (B, k, V)).copy()
    D = rng.choice(V, size=(B, k), p=q).astype(np.int32)
    ref = O.verify(Lt, Ld, D, 1.0, np.zeros(B, np.uint8), np.full(B, 0.5), seed=77, nthreads=4)
    s = metrics.acceptance_summary(_oracle_counters(ref, k), rounds=B, k=k)
    closed = float(np.minimum(p, q).sum())
    n = s["positions_tested"]
    sigma = math.sqrt(closed * (1 - closed) / n)
    assert abs(s["per_position_acceptance"] - closed) < 4 * sigma
    # expected tested positions per round: sum_{j<k} closed^j (a geometric chain)
    expect_rate = closed * sum(closed ** j for j in range(k)) / k
    assert s["acceptance_rate"] < closed - 10 * sigma
    assert abs(s["acceptance_rate"] - expect_rate) < 0.01
    assert s["mean_accepted_len"] == pytest.approx(ref["accepted_len"].mean())
    assert s["bonus"] + s["rejections"] == B
