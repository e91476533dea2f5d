"""GPU parity of the sampler filters (mlxcel PR #992, "What changed": top-k,
top-p and min-p before the softmax of p and q; top_k = 1 greedy) against the
oracle, through the C ABI."""
from __future__ import annotations

import numpy as np
import pytest
import torch

import workloads
from oracle import oracle as O
from tests.gpu_helpers import compare, oracle_for, peaked_workload

pytestmark = pytest.mark.gpu

OFF = (0, 1.0, 0.0)
FILTERS = {
    "topk_target": ((50, 1.0, 0.0), OFF),
    "topp_both": ((0, 0.9, 0.0), (0, 0.9, 0.0)),
    "chain": ((40, 0.8, 0.05), (20, 0.95, 0.01)),
    "greedy_target": ((1, 1.0, 0.0), OFF),
    "minp_both": ((0, 1.0, 0.2), (0, 1.0, 0.2)),
    "topk_draft": (OFF, (3, 1.0, 0.0)),
}


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_online_gb300 as pkg
    from speculative_decoding_verification_online_gb300 import build as B
    B.build()
    pkg.load()
    return pkg


def _run(sv, ver, w, **kw):
    out = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=0.5, gate_per_seq=w.gate,
                  threshold_per_seq=w.tau, seed=w.philox_seed, **kw)
    torch.cuda.synchronize()
    return out


def _filtered_drafts(w, fd):
    """Drafted tokens drawn from the filtered q (a drafter that samples with its own filters)."""
    if fd == OFF:
        return w
    Ld = workloads.to_numpy_logits(w.Ld)
    rng = np.random.default_rng(w.philox_seed)
    D = np.zeros((w.B, w.k), dtype=np.int32)
    for b in range(w.B):
        for j in range(w.k):
            q, _ = O.filtered_row(Ld[b, j], w.T, *fd)
            D[b, j] = rng.choice(w.V, p=q / q.sum())
    w.D = torch.as_tensor(D, device=w.D.device)
    return w


@pytest.mark.parametrize("dtype,V", [("bf16", 20000), ("f32", 4099)])
@pytest.mark.parametrize("name", sorted(FILTERS))
def test_filter_parity(sv, dtype, V, name):
    ft, fd = FILTERS[name]
    B, k = 40, 4
    gate = (np.arange(B) % 2).astype(np.uint8)
    seed = 300 + 7 * sorted(FILTERS).index(name) + (dtype == "f32")
    w = _filtered_drafts(peaked_workload(B, k, V, dtype, seed=seed, gate=gate, tau=0.3, T=0.9), fd)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(ft, fd)
    out = _run(sv, ver, w, row_stats=True)
    ref = oracle_for(w, filters=(ft, fd))
    st = compare(w, out, ref, what=f"filters {name} {dtype} V={V}", filters=(ft, fd))
    ok = ref["margin"] >= 1e-6
    rs = out["row_stats"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rs[ok][..., 1], ref["row_stats"][ok][..., 1], rtol=1e-5, atol=1e-5)
    assert st["compared"] >= B // 2
    ver.close()


def test_filtered_target_support_is_never_violated_on_the_gpu(sv):
    # a top_k = 2 target against an unfiltered drafter: every emitted token is
    # in the target row's two-token support (zero tolerance)
    B, k, V = 256, 4, 3000
    w = peaked_workload(B, k, V, "bf16", seed=41, gate=0, T=1.0)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters((2, 1.0, 0.0), OFF)
    out = _run(sv, ver, w)
    top2 = torch.topk(w.Lt.float(), 2, dim=2).indices.cpu().numpy()
    al = out["accepted_len"].cpu().numpy()
    tok = out["tokens"].cpu().numpy()
    for b in range(B):
        for j in range(al[b] + 1):
            assert tok[b, j] in top2[b, j], (b, j)
    ver.close()


def test_top_k_one_on_both_sides_is_the_greedy_call(sv):
    B, k, V = 32, 4, 5000
    w = peaked_workload(B, k, V, "bf16", seed=9, gate=(np.arange(B) % 2), T=0.8)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters((1, 1.0, 0.0), (1, 1.0, 0.0))
    f = _run(sv, ver, w)
    ver.set_filters(OFF, OFF)
    g = ver.run(w.Lt, w.Ld, w.D, 0.0, gate_mode=sv.SV_GATED_MU, threshold=0.5, gate_per_seq=w.gate,
                threshold_per_seq=w.tau, seed=w.philox_seed)
    torch.cuda.synchronize()
    for key in ("accepted_len", "tokens", "flags"):
        assert torch.equal(f[key], g[key]), key
    ver.close()


def test_filters_off_again_match_a_fresh_handle(sv):
    B, k, V = 24, 3, 6000
    w = peaked_workload(B, k, V, "f32", seed=13, gate=1, tau=0.4)
    a = sv.SpecVerifier(B, k, V, device=0)
    a.set_filters((10, 0.9, 0.1), (5, 1.0, 0.0))
    _run(sv, a, w)
    a.set_filters(OFF, OFF)
    x = _run(sv, a, w)
    b = sv.SpecVerifier(B, k, V, device=0)
    y = _run(sv, b, w)
    for key in ("accepted_len", "tokens", "accept_prob", "flags"):
        assert torch.equal(x[key], y[key]), key
    for bad in (((-1, 1.0, 0.0), OFF), ((0, 0.0, 0.0), OFF), ((0, 1.5, 0.0), OFF), (OFF, (0, 1.0, -0.1)),
                (OFF, (0, 1.0, 1.5)), ((0, float("nan"), 0.0), OFF)):
        with pytest.raises(sv.SpecVerifyError):
            a.set_filters(*bad)
    a.close()
    b.close()


def test_filter_full_size_128k(sv):
    w = workloads.make("b64_v128256_zipf_gated", seed=1234, device="cuda")
    ver = sv.SpecVerifier(w.B, w.k, w.V, device=0)
    # top-p inside top-k (the usual serving setting): over a whole Zipf row
    # top-p alone sits within 1e-6 of some tail token's boundary in every row
    for filt in (((50, 0.9, 0.0), (40, 0.95, 0.0)), ((0, 1.0, 0.01), (64, 1.0, 0.0))):
        ver.set_filters(*filt)
        out = _run(sv, ver, w)
        st = compare(w, out, oracle_for(w, nthreads=16, filters=filt), what=f"128k filtered {filt}",
                     filters=filt)
        assert st["compared"] >= w.B // 2
    ver.close()


def test_filtered_diagnostics(sv):
    B, k, V = 24, 4, 8000
    w = peaked_workload(B, k, V, "bf16", seed=17, gate=(np.arange(B) % 2), tau=0.3)
    filt = ((30, 0.9, 0.0), (0, 1.0, 0.05))
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(*filt)
    out = ver.diagnostics(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=0.5,
                          gate_per_seq=w.gate, threshold_per_seq=w.tau)
    torch.cuda.synchronize()
    ref = O.diagnostics(workloads.to_numpy_logits(w.Lt), workloads.to_numpy_logits(w.Ld), w.D.cpu().numpy(),
                        w.T, w.gate.cpu().numpy(), w.tau.cpu().numpy().astype(np.float64), filters=filt,
                        nthreads=16)
    keep = ref["margin"] >= 1e-6
    for key in ("min_sum", "pq_sum", "argmax_q"):
        np.testing.assert_allclose(out[key].cpu().numpy()[keep], ref[key][keep], rtol=2e-5, atol=2e-6,
                                   err_msg=key)
    assert keep.sum() >= B // 2
    ver.close()


@pytest.mark.parametrize("dtype,filt", [
    ("f32", ((25, 0.9, 0.0), (0, 1.0, 0.05))),   # the statistics path, both rows masked as they load
    ("bf16", ((1, 1.0, 0.0), (12, 0.9, 0.0))),   # a top_k = 1 target: one kept index
    ("f32", ((0, 0.8, 0.0), (1, 1.0, 0.0))),     # a top_k = 1 draft: q one-hot
])
def test_filtered_diagnostics_paths(sv, dtype, filt):
    # the diagnostics read each row as its sampler filter leaves it, the
    # threshold (or the one kept index) applied as logits load
    B, k, V = 20, 3, 6000
    w = peaked_workload(B, k, V, dtype, seed=23 + (dtype == "f32"), gate=(np.arange(B) % 2), tau=0.3)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(*filt)
    out = ver.diagnostics(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=0.5,
                          gate_per_seq=w.gate, threshold_per_seq=w.tau)
    torch.cuda.synchronize()
    ref = O.diagnostics(workloads.to_numpy_logits(w.Lt), workloads.to_numpy_logits(w.Ld), w.D.cpu().numpy(),
                        w.T, w.gate.cpu().numpy(), w.tau.cpu().numpy().astype(np.float64), filters=filt,
                        nthreads=16)
    keep = ref["margin"] >= 1e-6
    for key in ("min_sum", "pq_sum", "argmax_q"):
        np.testing.assert_allclose(out[key].cpu().numpy()[keep], ref[key][keep], rtol=2e-5, atol=2e-6,
                                   err_msg=key)
    assert keep.sum() >= B // 2
    ver.close()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_filters_with_a_gate_policy(sv, dtype):
    # the features compose: filtered p and q, a per-step schedule and a
    # cumulative floor on the filtered q, gated and plain sequences mixed
    B, k, V = 48, 5, 9000
    filt = ((20, 0.9, 0.0), (0, 0.95, 0.02))
    sched, cum = [0.3, 0.5], 0.1
    w = _filtered_drafts(peaked_workload(B, k, V, dtype, seed=61 + (dtype == "f32"),
                                         gate=(np.arange(B) % 3 != 2), tau=0.4), filt[1])
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(*filt)
    ver.set_gate_policy(sched, cum)
    out = _run(sv, ver, w)
    ref = oracle_for(w, tau_sched=sched, min_cum=cum, filters=filt)
    st = compare(w, out, ref, what=f"filters + policy {dtype}", tau_sched=sched, min_cum=cum,
                     filters=filt)
    assert st["compared"] >= B // 2
    assert int((ref["flags"] == 3).sum()) > 0  # the gate still bites on the filtered q
    ver.close()


# Rows whose top-k set the gathering pass collects (2 <= top_k <= the number
# of 2048-entry chunks).  Both sides gathered: no statistics pass runs; one
# side: the statistics pass runs and the other side selects from it.
GATHERED = {
    "both_topk": ((8, 1.0, 0.0), (12, 1.0, 0.0)),
    "both_topk_topp_minp": ((16, 0.9, 0.02), (5, 0.85, 0.0)),
    "target_only": ((8, 1.0, 0.0), (0, 0.9, 0.0)),
}


@pytest.mark.parametrize("dtype,V", [("bf16", 40000), ("f32", 30001)])
@pytest.mark.parametrize("name", sorted(GATHERED))
def test_gathered_filter_parity(sv, dtype, V, name):
    filt = GATHERED[name]
    B, k = 32, 3
    gate = (np.arange(B) % 2).astype(np.uint8)
    seed = 500 + 5 * sorted(GATHERED).index(name) + (dtype == "f32")
    w = _filtered_drafts(peaked_workload(B, k, V, dtype, seed=seed, gate=gate, tau=0.3, T=0.9), filt[1])
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(*filt)
    out = _run(sv, ver, w, row_stats=True)
    ref = oracle_for(w, filters=filt)
    st = compare(w, out, ref, what=f"gathered {name} {dtype} V={V}", filters=filt)
    ok = ref["margin"] >= 1e-6
    rs = out["row_stats"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rs[ok][..., 1], ref["row_stats"][ok][..., 1], rtol=1e-5, atol=1e-5)
    assert st["compared"] >= B // 2
    ver.close()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gathered_lists_that_overflow_fall_back(sv, dtype):
    # integer logits: a chunk holds hundreds of logits tied at the top value,
    # more than its 32 gathering slots, so every row is selected by the
    # fallback (which, with no statistics pass, reads the row itself); the
    # kept sets (every tie of the k-th largest) stay exact
    B, k, V = 16, 2, 16384
    g = torch.Generator(device="cuda")
    g.manual_seed(71 + (dtype == "f32"))
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    Lt = torch.randint(-3, 4, (B, k + 1, V), generator=g, device="cuda").float()
    Ld = (Lt[:, :k] + torch.randint(-1, 2, (B, k, V), generator=g, device="cuda").float())
    u = torch.rand(B, k, V, generator=g, device="cuda").clamp_(1e-30, 1 - 1e-7)
    D = torch.argmax(Ld - torch.log(-torch.log(u)), dim=2).to(torch.int32)
    w = workloads.Workload(name="ties", Lt=Lt.to(dt), Ld=Ld.to(dt), D=D, T=1.0,
                           gate=torch.zeros(B, dtype=torch.uint8, device="cuda"),
                           tau=torch.full((B,), 0.5, device="cuda"), philox_seed=9, B=B, k=k, V=V,
                           dtype=dtype)
    filt = ((4, 1.0, 0.0), (4, 0.9, 0.0))
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(*filt)
    out = _run(sv, ver, w)
    ref = oracle_for(w, filters=filt)
    st = compare(w, out, ref, what=f"gathered overflow {dtype}", filters=filt)
    assert st["compared"] + st["boundary"] == B
    ver.close()


# bf16 rows take the histogram selection (one read of each row, a counter per
# bf16 value of magnitude in [2^-15, 2^9)); these rows exercise its side
# paths: logits >= 2^9, logits below -2^9 that still weigh under top-p, tiny
# values |x| < 2^-15 (listed with their masses, or too many to list), a
# threshold among the tiny values, masked vocabulary (-inf), and ties at zero
# with both signs.  V = 4100 rows are not 16-byte multiples (the scalar loop).
EDGE_KINDS = {
    "above_2^9": (1.0, 4096, ((100, 0.9, 0.0), (0, 0.8, 0.05))),
    "below_-2^9_hot": (100.0, 4100, ((100, 0.9, 0.0), (0, 0.8, 0.0))),
    "below_-2^9_topk": (100.0, 4096, ((100, 1.0, 0.0), (7, 1.0, 0.0))),
    "tiny_overflow": (1.0, 4096, ((0, 0.9, 0.0), (50, 1.0, 0.0))),
    "tiny_listed": (1.0, 4100, ((0, 0.9, 0.0), (100, 0.95, 0.02))),
    "tiny_threshold": (1.0, 4096, ((0, 0.05, 0.0), (0, 0.05, 0.0))),
    "masked_vocab": (1.0, 4096, ((600, 0.9, 0.0), (20, 1.0, 0.1))),
    # values -2..2, about 820 of each: top_k = 2000 and top_p = 0.9 both end at zero
    "signed_zero_ties": (1.0, 4100, ((2000, 1.0, 0.0), (0, 0.9, 0.0))),
}


def _edge_workload(kind, B, k, V, T, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    R = B * (2 * k + 1)
    x = torch.randn(R, V, generator=g, device="cuda")
    if kind == "above_2^9":
        x[:, : V // 16] += 600.0
    elif kind.startswith("below_-2^9"):
        x = x * 150.0 - 300.0  # max near 300; about 8 % below -512, weighing 2^-12 of the max at T = 100
    elif kind == "tiny_overflow":
        x = x * 1e-5
    elif kind == "tiny_listed":
        x[:, :20] = (torch.rand(R, 20, generator=g, device="cuda") - 0.5) * 4e-5
    elif kind == "tiny_threshold":
        # mass from the top: two tokens at 2 (14.8), forty tiny ones (40.0),
        # the rest at -1 (735.8): top-p 0.05 ends among the tiny values
        x.fill_(-1.0)
        x[:, 0:2] = 2.0
        x[:, 2:42] = 1e-6 * torch.arange(1, 41, device="cuda", dtype=torch.float32)
        x[:, 2042:] = float("-inf")
        x = x[:, torch.randperm(V, generator=g, device="cuda")]
    elif kind == "masked_vocab":
        x[torch.rand(R, V, generator=g, device="cuda") < 0.9] = float("-inf")
    elif kind == "signed_zero_ties":
        x = torch.randint(-2, 3, (R, V), generator=g, device="cuda").float()
        neg = torch.rand(R, V, generator=g, device="cuda") < 0.5
        x = torch.where((x == 0) & neg, torch.full_like(x, -0.0), x)
    Lt = x[: B * (k + 1)].reshape(B, k + 1, V).to(torch.bfloat16)
    Ld = x[B * (k + 1):].reshape(B, k, V).to(torch.bfloat16)
    u = torch.rand(B, k, V, generator=g, device="cuda").clamp_(1e-30, 1 - 1e-7)
    D = torch.argmax(Ld.float() / T - torch.log(-torch.log(u)), dim=2).to(torch.int32)
    gate = torch.as_tensor((np.arange(B) % 2).astype(np.uint8), device="cuda")
    return workloads.Workload(name=kind, Lt=Lt, Ld=Ld, D=D, T=T, gate=gate,
                              tau=torch.full((B,), 0.3, device="cuda"), philox_seed=seed + 1, B=B, k=k, V=V,
                              dtype="bf16")


@pytest.mark.parametrize("kind", sorted(EDGE_KINDS))
def test_histogram_selection_edge_rows(sv, kind):
    T, V, filt = EDGE_KINDS[kind]
    B, k = 12, 2
    w = _edge_workload(kind, B, k, V, T, seed=700 + sorted(EDGE_KINDS).index(kind))
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(*filt)
    out = _run(sv, ver, w, row_stats=True)
    ref = oracle_for(w, filters=filt)
    st = compare(w, out, ref, what=f"histogram edge rows {kind}", filters=filt)
    # the filtered rows' statistics pin every row's kept set
    ok = ref["margin"] >= 1e-6
    rs = out["row_stats"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rs[ok][..., 0], ref["row_stats"][ok][..., 0], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(rs[ok][..., 1], ref["row_stats"][ok][..., 1], rtol=1e-5, atol=1e-5)
    assert ok.sum() >= B // 2
    assert st["compared"] >= B // 2
    ver.close()


# Top-k rows count their first 8192 logits in full and, past them, only the
# vectors holding a logit at or above the k-th largest of those (queued per
# warp).  These rows (V = 20000, the vector path) put what that must not miss
# past the first 8192: a NaN or +inf (an invalid row), logits >= 2^9 (the
# radix fallback), the row's largest logits (a low cut: most vectors queued),
# and a first 8192 of signed zeros, so that the cut is zero and top-k ends in
# zeros of both signs.
CUT_KINDS = {
    "late_nan": ((50, 0.9, 0.0), (40, 0.95, 0.0)),
    "late_posinf": ((50, 0.9, 0.0), (40, 1.0, 0.0)),
    "late_above_2^9": ((50, 0.9, 0.0), (30, 0.8, 0.0)),
    "largest_late": ((200, 0.9, 0.0), (64, 0.95, 0.0)),
    "zero_cut": ((6000, 0.9, 0.0), (3000, 1.0, 0.0)),
}


def _cut_workload(kind, B, k, V, seed):
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    R = B * (2 * k + 1)
    x = torch.randn(R, V, generator=g, device="cuda")
    late = 8192 + torch.randint(0, V - 8192, (R,), generator=g, device="cuda")
    rows = torch.arange(R, device="cuda")
    some = rows % 5 == 1  # a fifth of the rows, leaving sequences 1, 4, 6, 9, 11 whole
    if kind == "late_nan":
        x[rows[some], late[some]] = float("nan")
    elif kind == "late_posinf":
        x[rows[some], late[some]] = float("inf")
    elif kind == "late_above_2^9":
        x[rows[some], late[some]] = 700.0
    elif kind == "largest_late":
        x[:, :8192] -= 3.0
        x[:, 8192:] += 3.0
    elif kind == "zero_cut":
        x = torch.randint(-2, 3, (R, V), generator=g, device="cuda").float()
        x[:, :8192] = 0.0
        neg = torch.rand(R, V, generator=g, device="cuda") < 0.5
        x = torch.where((x == 0) & neg, torch.full_like(x, -0.0), x)
    Lt = x[: B * (k + 1)].reshape(B, k + 1, V).to(torch.bfloat16)
    Ld = x[B * (k + 1):].reshape(B, k, V).to(torch.bfloat16)
    u = torch.rand(B, k, V, generator=g, device="cuda").clamp_(1e-30, 1 - 1e-7)
    xd = torch.nan_to_num(Ld.float(), nan=0.0, posinf=0.0)
    D = torch.argmax(xd - torch.log(-torch.log(u)), dim=2).to(torch.int32)
    gate = torch.as_tensor((np.arange(B) % 2).astype(np.uint8), device="cuda")
    return workloads.Workload(name=kind, Lt=Lt, Ld=Ld, D=D, T=1.0, gate=gate,
                              tau=torch.full((B,), 0.3, device="cuda"), philox_seed=seed + 1, B=B, k=k, V=V,
                              dtype="bf16")


@pytest.mark.parametrize("kind", sorted(CUT_KINDS))
def test_histogram_selection_cut_rows(sv, kind):
    filt = CUT_KINDS[kind]
    B, k, V = 12, 2, 20000
    w = _cut_workload(kind, B, k, V, seed=900 + sorted(CUT_KINDS).index(kind))
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(*filt)
    out = _run(sv, ver, w, row_stats=True)
    ref = oracle_for(w, filters=filt)
    st = compare(w, out, ref, what=f"histogram cut rows {kind}", filters=filt)
    invalid = ref["accepted_len"] < 0
    if kind in ("late_nan", "late_posinf"):
        # sequences with a NaN or +inf in one of their rows are invalid on both sides
        assert invalid.any()
        assert np.array_equal(out["accepted_len"].cpu().numpy() < 0, invalid)
    else:
        assert not invalid.any()
    # the filtered rows' statistics pin every valid row's kept set
    ok = (ref["margin"] >= 1e-6) & ~invalid
    rs = out["row_stats"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rs[ok][..., 0], ref["row_stats"][ok][..., 0], rtol=1e-5, atol=1e-5)
    np.testing.assert_allclose(rs[ok][..., 1], ref["row_stats"][ok][..., 1], rtol=1e-5, atol=1e-5)
    assert st["compared"] >= 2 and ok.sum() >= 2
    ver.close()


def _same_rows_workload(B, k, V, dtype, x, gate, tau, seed):
    """Draft rows equal to the target rows (p = q at every position) and each
    drafted token the smallest draft logit, outside any filtered set: every
    position is rejected (p(D) = 0) or NULL (q(D) = 0 < tau)."""
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    Lt = x.to(dt)
    Ld = x[:, :k].contiguous().to(dt)
    D = torch.argmin(Ld.float(), dim=2).to(torch.int32)
    return workloads.Workload(name="same_rows", Lt=Lt, Ld=Ld, D=D, T=1.0,
                              gate=torch.as_tensor(np.broadcast_to(np.asarray(gate, dtype=np.uint8), (B,)).copy(),
                                                   device="cuda"),
                              tau=torch.full((B,), tau, device="cuda"), philox_seed=seed, B=B, k=k, V=V, dtype=dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("filt", [((5, 1.0, 0.0), (5, 1.0, 0.0)), ((0, 0.5, 0.0), (0, 0.5, 0.0))])
def test_degenerate_residuals_fall_back_to_p(sv, dtype, filt):
    # p = q on the kept sets and D outside them: a plain stop row's residual
    # (p - q)+ is exactly empty, so the token is drawn from p (the reading of
    # the oracle); the GPU must find it empty too, not sample rounding noise
    B, k, V = 16, 2, 4096
    g = torch.Generator(device="cuda")
    g.manual_seed(5)
    x = torch.randn(B, k + 1, V, generator=g, device="cuda") * 2
    w = _same_rows_workload(B, k, V, dtype, x, np.arange(B) % 2, 0.3, seed=11)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(*filt)
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = _run(sv, ver, w, counters=cnt)
    ref = oracle_for(w, filters=filt)
    compare(w, out, ref, what=f"degenerate {dtype} {filt}", filters=filt)
    assert int(cnt[sv.SV_CNT_DEGENERATE]) == int(ref["degenerate"].sum()) >= B // 2
    ver.close()


def test_degenerate_gated_residual_on_the_candidate_path(sv):
    # two tied top tokens kept by top_k = 2 on both sides, q = 0.5 >= tau:
    # both admitted, so mu = q = p and the residual of a NULL stop row is
    # empty; the gated fast path computes it from chunk statistics minus the
    # admitted overlap, which leaves only rounding -- still empty, drawn from p
    B, k, V = 16, 2, 6000
    g = torch.Generator(device="cuda")
    g.manual_seed(6)
    x = torch.randn(B, k + 1, V, generator=g, device="cuda") - 10.0
    top = torch.stack([torch.randperm(V, generator=g, device="cuda")[:2] for _ in range(B * (k + 1))])
    x.view(-1, V).scatter_(1, top, 5.0)
    w = _same_rows_workload(B, k, V, "bf16", x, 1, 0.3, seed=13)
    ver = sv.SpecVerifier(B, k, V, device=0)
    filt = ((2, 1.0, 0.0), (2, 1.0, 0.0))
    ver.set_filters(*filt)
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=0.3, seed=w.philox_seed,
                  counters=cnt)
    torch.cuda.synchronize()
    ref = oracle_for(w, filters=filt)
    compare(w, out, ref, what="degenerate gated", filters=filt)
    assert int(cnt[sv.SV_CNT_DEGENERATE]) == int(ref["degenerate"].sum()) == B
    assert (out["tokens"][:, 0] >= 0).all()
    ver.close()


@pytest.mark.parametrize("V", [1, 8, 67, 2047])
def test_histogram_selection_small_vocabularies(sv, V):
    # one logit, one 16-byte vector, the scalar read (rows not 16-byte
    # multiples), and top_k at or above V (no top-k)
    filt = ((3, 0.9, 0.0), (0, 0.8, 0.1))
    B, k = 16, 3
    w = peaked_workload(B, k, V, "bf16", seed=900 + V, gate=(np.arange(B) % 2), tau=0.3, T=0.9)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_filters(*filt)
    out = _run(sv, ver, w, row_stats=True)
    ref = oracle_for(w, filters=filt)
    st = compare(w, out, ref, what=f"histogram small V={V}", filters=filt)
    ok = ref["margin"] >= 1e-6
    rs = out["row_stats"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rs[ok][..., 1], ref["row_stats"][ok][..., 1], rtol=1e-5, atol=1e-5)
    assert st["compared"] >= B // 2
    ver.close()
