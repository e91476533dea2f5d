"""GPU parity of the gate policy (per-step threshold schedules and the
cumulative prefix-product floor of the regolith audit's "schedule behavior"
section) against the oracle, on the fast candidate path and the dense
residual path, at temperature > 0 and 0, plus the policy's host errors."""
from __future__ import annotations

import os

import numpy as np
import pytest
import torch

import workloads
from tests.gpu_helpers import compare, oracle_for, peaked_workload as _peaked

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_online_gb300 as pkg
    from speculative_decoding_verification_online_gb300 import build as B
    B.build()
    pkg.load()
    return pkg


def _run(sv, ver, w, **kw):
    out = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=0.5,
                  gate_per_seq=w.gate, threshold_per_seq=w.tau, seed=w.philox_seed, **kw)
    torch.cuda.synchronize()
    return out


# (schedule, cumulative floor): which stop rows take the candidate fast path
# (every floor max(tau_j, min_cum) above ~0.2) or the dense re-read
POLICIES = {
    "schedule": ([0.3, 0.5, 0.7], 0.0),       # fast, last entry repeats for steps 3..5
    "cumulative": (None, 0.15),               # the sequences' own 0.5 plus a floor
    "cumulative_only": ([0.0], 0.25),         # fast through the floor alone
    "dense": ([0.1], 0.05),                   # floors below the fast path: dense residuals
    "mixed": ([0.6, 0.25, 0.0], 0.3),         # fast rows and a zero step floor
    "off": ([0.0], 0.0),                      # every token admitted: the plain rule
}


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("name", sorted(POLICIES))
def test_gate_policy_parity(sv, dtype, name):
    sched, cum = POLICIES[name]
    B, k, V = 64, 6, 20000
    gate = (np.arange(B) % 4 != 3).astype(np.uint8)  # every fourth sequence plain
    seed = 17 + 10 * sorted(POLICIES).index(name) + (dtype == "f32")
    w = _peaked(B, k, V, dtype, seed=seed, gate=gate)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_gate_policy(sched, cum)
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = _run(sv, ver, w, counters=cnt)
    ref = oracle_for(w, tau_sched=sched, min_cum=cum)
    st = compare(w, out, ref, what=f"policy {name} {dtype}", tau_sched=sched, min_cum=cum)
    flags = ref["flags"]
    # the workload really exercises the gate: NULL rows at more than one step
    if name != "off":
        steps_with_null = {int(j) for j in np.nonzero(flags == 3)[1]}
        assert len(steps_with_null) >= 2, steps_with_null
    c = cnt.cpu().numpy()
    if st["boundary"] == 0:
        assert c[1] == ref["accepted_len"].sum()
        assert c[2] == int((flags == 3).sum()) and c[3] == int((flags == 2).sum())
    if name == "off":
        # schedule 0 and floor 0 admit every token: the plain rule, bit for bit
        w_plain = _peaked(B, k, V, dtype, seed=seed, gate=0)
        ver.set_gate_policy(None, 0.0)
        plain = _run(sv, ver, w_plain)
        for key in ("accepted_len", "tokens", "accept_prob"):
            assert torch.equal(out[key], plain[key]), key
    ver.close()


@pytest.mark.parametrize("name", ["schedule", "cumulative_only", "mixed", "off"])
def test_gate_policy_greedy(sv, name):
    sched, cum = POLICIES[name]
    B, k, V = 48, 5, 4096
    w = _peaked(B, k, V, "bf16", seed=71, gate=(np.arange(B) % 2).astype(np.uint8), T=0.0)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_gate_policy(sched, cum)
    out = _run(sv, ver, w)
    ref = oracle_for(w, tau_sched=sched, min_cum=cum)
    compare(w, out, ref, what=f"greedy policy {name}", tau_sched=sched, min_cum=cum)
    ver.close()


def test_gate_policy_worked_examples_exactly(sv):
    # the retention numbers of the audit's "economics and confidence" section,
    # with draft probabilities that are exact in fp32 (1/n for n equal logits)
    rows = []
    with open(os.path.join(GOLDEN, "gate_schedule_example.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    V = 10
    for kind, qs, sched, cum, want in rows:
        q = [float(x) for x in qs.split(",")]
        k = len(q)
        Ld = torch.full((1, k, V), float("-inf"))
        for j, qj in enumerate(q):
            Ld[0, j, :int(round(1 / qj))] = 0.0
        Lt = torch.cat([Ld, Ld[:, :1]], dim=1)
        w = workloads.Workload(name="example", Lt=Lt.cuda(), Ld=Ld.cuda(),
                               D=torch.zeros(1, k, dtype=torch.int32, device="cuda"), T=1.0,
                               gate=torch.ones(1, dtype=torch.uint8, device="cuda"),
                               tau=torch.full((1,), 0.99, device="cuda"), philox_seed=3, B=1, k=k,
                               V=V, dtype="f32")
        ver = sv.SpecVerifier(1, k, V, device=0)
        sch = [float(x) for x in sched.split(",")]
        ver.set_gate_policy(sch, float(cum))
        got = int(_run(sv, ver, w)["accepted_len"][0])
        ref = int(oracle_for(w, tau_sched=sch, min_cum=float(cum))["accepted_len"][0])
        assert got == ref, (kind, qs, sched, cum)
        if want.startswith(">="):
            assert got >= int(want[2:])
        else:
            assert got == int(want), (kind, qs, sched, cum)
        ver.close()


def test_gate_policy_full_size_128k(sv):
    # the 128K-vocabulary batch under a schedule with a cumulative floor (fast
    # path) and under floors that force dense residual re-reads
    w = workloads.make("b64_v128256_zipf_gated", seed=1234, device="cuda")
    ver = sv.SpecVerifier(w.B, w.k, w.V, device=0)
    for sched, cum in (([0.25, 0.35], 0.21), ([0.05], 0.02)):
        ver.set_gate_policy(sched, cum)
        out = _run(sv, ver, w)
        ref = oracle_for(w, nthreads=16, tau_sched=sched, min_cum=cum)
        compare(w, out, ref, what=f"128k policy {sched} {cum}", tau_sched=sched, min_cum=cum)
    ver.close()


def test_gate_policy_host_errors_keep_the_previous_policy(sv):
    B, k, V = 16, 4, 3000
    w = _peaked(B, k, V, "f32", seed=5)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_gate_policy([0.4, 0.6], 0.1)
    for bad in (([], 0.0), ([0.5] * 33, 0.0), ([float("nan")], 0.0), ([-0.1], 0.0), ([1.5], 0.0),
                ([0.5], -0.2), ([0.5], 1.01), ([0.5], float("inf"))):
        with pytest.raises(sv.SpecVerifyError):
            ver.set_gate_policy(*bad)
    # a NULL schedule with a nonzero length is malformed too
    lib = sv.load()
    assert lib.spec_verify_set_gate_policy(ver.handle, None, 2, 0.0) == 1
    out = _run(sv, ver, w)
    ref = oracle_for(w, tau_sched=[0.4, 0.6], min_cum=0.1)
    compare(w, out, ref, what="policy kept", tau_sched=[0.4, 0.6], min_cum=0.1)
    # with a schedule the sequences' own thresholds are not used, so an
    # out-of-range one is no error
    w.tau.fill_(7.0)
    out = _run(sv, ver, w)
    assert bool((out["accepted_len"] >= 0).all())
    ver.close()


def test_gate_policy_host_buffer_entry_point(sv):
    B, k, V = 24, 5, 5000
    w = _peaked(B, k, V, "bf16", seed=9)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_gate_policy([0.3], 0.2)
    dev = _run(sv, ver, w)
    host = ver.run_host(w.Lt.cpu(), w.Ld.cpu(), w.D.cpu(), w.T, gate_mode=sv.SV_GATED_MU,
                        threshold=0.5, gate_per_seq=w.gate.cpu(), threshold_per_seq=w.tau.cpu(),
                        seed=w.philox_seed)
    for key in ("accepted_len", "tokens", "accept_prob"):
        assert torch.equal(dev[key].cpu(), host[key]), key
    ver.close()
