"""GPU parity of the closed-form acceptance diagnostics (mlxcel PR #992, "The
acceptance ceiling": sum min(p, mu), sum p q, q(argmax p) per draft position)
against the oracle, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from oracle import oracle as O
from tests.gpu_helpers import BOUNDARY, peaked_workload

pytestmark = pytest.mark.gpu

# fp32 probabilities (ex2.approx, an fp32 normaliser) summed in fp32 over up to
# 2^22 terms in 8-term pairwise groups per lane: 2e-5 relative plus 2e-6
# absolute covers the rounding with room; the argmax index is exact
RTOL, ATOL = 2e-5, 2e-6


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_online_gb300 as pkg
    from speculative_decoding_verification_online_gb300 import build as B
    B.build()
    pkg.load()
    return pkg


def _oracle(w, tau_sched=None, min_cum=0.0):
    return O.diagnostics(workloads.to_numpy_logits(w.Lt), workloads.to_numpy_logits(w.Ld),
                         w.D.cpu().numpy(), w.T, w.gate.cpu().numpy(),
                         w.tau.cpu().numpy().astype(np.float64), tau_sched=tau_sched,
                         min_cum=min_cum, nthreads=16)


def _diag(sv, ver, w):
    out = ver.diagnostics(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=0.5,
                          gate_per_seq=w.gate, threshold_per_seq=w.tau)
    torch.cuda.synchronize()
    return {key: v.cpu().numpy().astype(np.float64) for key, v in out.items()}


def _compare(got, ref, what):
    # a sequence with some q(x) within 1e-6 of its gate boundary may admit x on
    # one side and not the other: its min_sum is a boundary case
    keep = (ref["margin"] >= BOUNDARY)[:, None] & np.ones_like(ref["min_sum"], dtype=bool)
    for key in ("min_sum", "pq_sum", "argmax_q"):
        g, r = got[key], ref[key]
        assert np.array_equal(np.isnan(g), np.isnan(r)), (what, key)
        sel = ~np.isnan(r) & (keep if key == "min_sum" else True)
        np.testing.assert_allclose(g[sel], r[sel], rtol=RTOL, atol=ATOL, err_msg=f"{what} {key}")
    print(f"[diag] {what}: {int(keep.all(axis=1).sum())}/{keep.shape[0]} sequences off the gate boundary")


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [20000, 2048, 67, 1])
def test_diagnostics_parity(sv, dtype, V):
    B, k = 32, 4
    gate = (np.arange(B) % 2).astype(np.uint8)
    w = peaked_workload(B, k, V, dtype, seed=V + 5 * (dtype == "f32"), gate=gate, tau=0.3, T=0.9)
    ver = sv.SpecVerifier(B, k, V, device=0)
    got = _diag(sv, ver, w)
    _compare(got, _oracle(w), f"V={V} {dtype}")
    # the ceiling bounds sampler-match and is at most 1 (plain rows)
    plain = gate == 0
    assert np.all(got["min_sum"][plain] >= got["pq_sum"][plain] - 1e-6)
    assert np.all(got["min_sum"] <= 1.0 + 1e-5)
    ver.close()


@pytest.mark.parametrize("sched,cum", [([0.3, 0.5, 0.7], 0.0), ([0.0], 0.25), (None, 0.1)])
def test_diagnostics_parity_under_gate_policy(sv, sched, cum):
    B, k, V = 48, 6, 12000
    w = peaked_workload(B, k, V, "bf16", seed=int(cum * 100) + 3, gate=(np.arange(B) % 4 != 3))
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_gate_policy(sched, cum)
    _compare(_diag(sv, ver, w), _oracle(w, sched, cum), f"policy {sched} {cum}")
    ver.close()


@pytest.mark.parametrize("cum", [0.0, 0.5])
def test_diagnostics_greedy(sv, cum):
    B, k, V = 40, 5, 5000
    w = peaked_workload(B, k, V, "bf16", seed=13, gate=(np.arange(B) % 2), T=0.0)
    ver = sv.SpecVerifier(B, k, V, device=0)
    if cum:
        ver.set_gate_policy([0.0], cum)
    got = _diag(sv, ver, w)
    ref = _oracle(w, [0.0] if cum else None, cum)
    for key in ("min_sum", "pq_sum", "argmax_q"):
        np.testing.assert_array_equal(got[key], ref[key], err_msg=key)
    ver.close()


def test_diagnostics_full_size_128k(sv):
    w = workloads.make("b64_v128256_zipf_gated", seed=1234, device="cuda")
    ver = sv.SpecVerifier(w.B, w.k, w.V, device=0)
    _compare(_diag(sv, ver, w), _oracle(w), "128k gated")
    w = workloads.make("b64_v128256_zipf_gated", seed=1234, device="cuda", gate="plain")
    _compare(_diag(sv, ver, w), _oracle(w), "128k plain")
    ver.close()


def test_diagnostics_invalid_rows_and_host_errors(sv):
    B, k, V = 6, 3, 3000
    w = peaked_workload(B, k, V, "f32", seed=2, gate=1, tau=0.4)
    w.Lt[1, 2, 7] = float("nan")                # target row 2 of sequence 1
    w.Ld[2, 0, :] = float("-inf")               # draft row 0 of sequence 2
    w.D[3, 0] = V + 5                           # out-of-range drafted token
    w.tau[4] = 1.5                              # bad threshold (no schedule)
    ver = sv.SpecVerifier(B, k, V, device=0)
    got = _diag(sv, ver, w)
    _compare(got, _oracle(w), "invalid rows")
    assert np.isnan(got["min_sum"][1, 2]) and np.isfinite(got["min_sum"][1, :2]).all()
    assert np.isnan(got["pq_sum"][2, 0]) and np.isfinite(got["pq_sum"][2, 1:]).all()
    assert np.isfinite(got["min_sum"][3]).all()  # no cumulative floor: D is not read
    assert np.isnan(got["min_sum"][4]).all()
    ver.set_gate_policy([0.0], 0.1)              # now the product reads D[3, 0]
    got = _diag(sv, ver, w)
    _compare(got, _oracle(w, [0.0], 0.1), "invalid rows, cumulative floor")
    assert np.isfinite(got["min_sum"][3, 0]) and np.isnan(got["min_sum"][3, 1:]).all()
    lib = sv.load()
    rc = lib.spec_verify_diagnostics(None, None, 0, None, 0, None, 1, 1.0, 0, 0.5, None, None,
                                     None, None, None, None)
    assert rc == 1
    with pytest.raises(sv.SpecVerifyError):
        ver.diagnostics(w.Lt, w.Ld, w.D, -1.0)
    # no outputs asked for: nothing runs, success
    rc = lib.spec_verify_diagnostics(ver.handle, w.Lt.data_ptr(), 0, w.Ld.data_ptr(), 0,
                                     w.D.data_ptr(), B, 1.0, 0, 0.5, None, None, None, None, None,
                                     None)
    assert rc == 0
    ver.close()


def test_diagnostics_then_run_on_one_handle(sv):
    # the diagnostics' stream pass leaves no gate candidates behind: a run on
    # the same handle afterwards matches a fresh handle's
    from tests.gpu_helpers import compare, oracle_for
    B, k, V = 32, 4, 20000
    w = peaked_workload(B, k, V, "bf16", seed=77, gate=1, tau=0.5)
    ver = sv.SpecVerifier(B, k, V, device=0)
    _diag(sv, ver, w)
    out = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=0.5, gate_per_seq=w.gate,
                  threshold_per_seq=w.tau, seed=w.philox_seed)
    torch.cuda.synchronize()
    compare(w, out, oracle_for(w), what="run after diagnostics")
    ver.close()
