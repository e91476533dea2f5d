"""Acceptance summary over the verifier's batch counters.

The mlxcel PR #992 page reports every speculative run with one greppable
summary line ("Observability: how to prove which rule ran") and corrects its
denominator ("Two metric corrections found by making it visible"): a chain
stops at its first rejection, so the draft positions behind the stop are never
tested, and the quantity that the closed form sum_x min(p, mu) predicts is the
acceptance per *tested* position; accepted / proposed understates it.

``spec_verify_run`` accumulates the counters on the GPU (``counters`` [8]
uint64, in the order of ``COUNTER_NAMES``; passing the same buffer to several
calls sums them).  This module only turns those counts into the summary's
ratios on the host; it does no verification arithmetic.

Definitions, for counters covering ``rounds`` sequence verifications (a
sequence in a call is one round) with ``k`` draft positions each:
  valid rounds             = rounds - invalid (an invalid sequence tests nothing)
  proposed                 = valid rounds * k
  positions_tested         = counters[tested] (accepted positions plus each stop
                             position before k)
  per_position_acceptance  = accepted / positions_tested
  acceptance_rate          = accepted / proposed
  mean_accepted_len        = accepted / valid rounds
A ratio whose denominator is 0 is NaN.
"""
from __future__ import annotations

import math
from typing import Dict, Sequence, Union

from .spec_verify import COUNTER_NAMES

Number = Union[int, float]


def _counts(counters) -> Sequence[int]:
    if hasattr(counters, "tolist"):  # torch tensor or numpy array
        counters = counters.tolist()
    vals = [int(x) for x in counters]
    if len(vals) != len(COUNTER_NAMES):
        raise ValueError(f"expected {len(COUNTER_NAMES)} counters, got {len(vals)}")
    if any(v < 0 for v in vals):
        raise ValueError("counters must be non-negative")
    return vals


def _ratio(a: int, b: int) -> float:
    return a / b if b else math.nan


def rule_id(temperature: float, gated: bool) -> str:
    """Stable identifier of the rule a call ran: greedy decoding at temperature
    0, modified rejection sampling otherwise (with the mu/NULL gate when gated)."""
    if temperature == 0:
        return "greedy-argmax"
    return "stochastic-mu-null" if gated else "stochastic"


def acceptance_summary(counters, rounds: int, k: int, rule: str = "stochastic") -> Dict[str, Number]:
    """The summary's fields from the counters of ``rounds`` sequence
    verifications with ``k`` draft positions each (definitions above)."""
    c = dict(zip(COUNTER_NAMES, _counts(counters)))
    if rounds < 0 or k < 1:
        raise ValueError("rounds must be >= 0 and k >= 1")
    if c["invalid"] > rounds:
        raise ValueError("more invalid sequences than rounds")
    valid = rounds - c["invalid"]
    proposed = valid * k
    if c["tested"] > proposed or c["accepted"] > c["tested"]:
        raise ValueError("counters inconsistent with rounds and k")
    return {
        "rule": rule,
        "rounds": valid,
        "proposed": proposed,
        "positions_tested": c["tested"],
        "accepted": c["accepted"],
        "per_position_acceptance": _ratio(c["accepted"], c["tested"]),
        "acceptance_rate": _ratio(c["accepted"], proposed),
        "mean_accepted_len": _ratio(c["accepted"], valid),
        "nulls": c["null"],
        "rejections": c["rejected"],
        "bonus": c["bonus"],
        "boundary_draws": c["boundary"],
        "invalid": c["invalid"],
        "degenerate": c["degenerate"],
    }


_LINE_KEYS = ("rule", "rounds", "proposed", "positions_tested", "accepted", "per_position_acceptance",
              "acceptance_rate", "mean_accepted_len", "nulls", "rejections", "bonus", "boundary_draws",
              "invalid", "degenerate")


def summary_line(summary: Dict[str, Number]) -> str:
    """One whitespace-separated ``key=value`` line (ratios to four decimals),
    led by ``[Speculative acceptance]``."""
    parts = []
    for key in _LINE_KEYS:
        v = summary[key]
        parts.append(f"{key}={v:.4f}" if isinstance(v, float) else f"{key}={v}")
    return "[Speculative acceptance] " + " ".join(parts)


def parse_summary_line(line: str) -> Dict[str, Union[str, int, float]]:
    """The fields of a line written by ``summary_line``."""
    prefix = "[Speculative acceptance] "
    if not line.startswith(prefix):
        raise ValueError("not an acceptance summary line")
    out: Dict[str, Union[str, int, float]] = {}
    for item in line[len(prefix):].split():
        key, _, value = item.partition("=")
        if key == "rule":
            out[key] = value
        elif "." in value or value == "nan":
            out[key] = float(value)
        else:
            out[key] = int(value)
    return out
