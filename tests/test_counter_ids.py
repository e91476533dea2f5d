"""The binding's counter indices are the header's SV_CNT_* enum, in the order
of COUNTER_NAMES (no GPU)."""
from __future__ import annotations

import pathlib
import re

import speculative_decoding_verification_online_gb300 as pkg


def test_counter_indices_match_the_header():
    h = (pathlib.Path(__file__).resolve().parents[1] / "include" / "spec_verify.h").read_text()
    enum = {m.group(1): int(m.group(2)) for m in re.finditer(r"\bSV_CNT_([A-Z]+)\s*=\s*(\d+)", h)}
    assert len(enum) == len(pkg.COUNTER_NAMES) == 8
    for name, idx in enum.items():
        assert getattr(pkg, f"SV_CNT_{name}") == idx, name
        assert pkg.COUNTER_NAMES[idx] == name.lower(), name
