"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle on
the same seeded inputs.  See tests/gpu_helpers.py for the comparison rules."""
from __future__ import annotations

import numpy as np
import pytest
import torch
from scipy.stats import chi2

import workloads
from tests.gpu_helpers import compare, oracle_for, peaked_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_online_gb300 as pkg
    from speculative_decoding_verification_online_gb300 import build as B
    B.build()
    pkg.load()
    return pkg


def _verifier(sv, w, max_B=None):
    return sv.SpecVerifier(max_B or w.B, w.k, w.V, device=0)


def _run(sv, ver, w, **kw):
    out = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=0.5,
                  gate_per_seq=w.gate, threshold_per_seq=w.tau, seed=w.philox_seed, **kw)
    torch.cuda.synchronize()
    return out


def _custom(B, k, V, dtype, T, gate, tau, seed, device="cuda", scale=3.0, noise=1.0):
    """A small custom workload (normal logits) with its own shape."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    t = torch.randn(B, k + 1, V, generator=g, device=device) * scale
    d = t[:, :k] + torch.randn(B, k, V, generator=g, device=device) * noise
    Lt, Ld = t.to(dt), d.to(dt)
    u = torch.rand(B, k, V, generator=g, device=device).clamp_(1e-30, 1 - 1e-7)
    D = torch.argmax(Ld.float() / T - torch.log(-torch.log(u)), dim=2).to(torch.int32)
    gate_t = torch.as_tensor(np.broadcast_to(np.asarray(gate, dtype=np.uint8), (B,)).copy(),
                             device=device)
    tau_t = torch.full((B,), float(tau), dtype=torch.float32, device=device)
    return workloads.Workload(name="custom", Lt=Lt, Ld=Ld, D=D, T=T, gate=gate_t, tau=tau_t,
                              philox_seed=seed + 2, B=B, k=k, V=V, dtype=dtype)


# ------------------------------------------------------------- small shapes

@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [20000, 8192, 67, 1])
def test_parity_small_shapes_ragged_tails(sv, dtype, V):
    B, k = 40, 4
    gate = (np.arange(B) % 2).astype(np.uint8)
    w = _custom(B, k, V, dtype, 0.7, gate, 0.3, seed=V + (dtype == "f32"))
    ver = _verifier(sv, w)
    out = _run(sv, ver, w, row_stats=True)
    ref = oracle_for(w)
    compare(w, out, ref, what=f"V={V} {dtype}")
    rs = out["row_stats"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rs[..., 0], ref["row_stats"][..., 0], rtol=1e-6, atol=1e-6)
    np.testing.assert_allclose(rs[..., 1], ref["row_stats"][..., 1], rtol=1e-5, atol=1e-5)
    ver.close()


@pytest.mark.parametrize("tau", [0.5, 0.3, 0.21, 0.1, 1.0])
def test_parity_gate_thresholds_fast_and_dense_paths(sv, tau):
    # tau > ~0.2 takes the candidate fast path, 0.1 the dense residual path
    B, k, V = 48, 3, 12000
    w = _custom(B, k, V, "bf16", 1.0, 1, tau, seed=int(tau * 100), scale=2.5, noise=0.7)
    ver = _verifier(sv, w)
    out = _run(sv, ver, w)
    ref = oracle_for(w)
    compare(w, out, ref, what=f"tau={tau}")
    ver.close()


def _run_scalar_gate(sv, ver, w, tau):
    # uniform gate settings as scalars: with tau on the candidate fast path the
    # finishing kernel without the dense pass runs
    out = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=tau, seed=w.philox_seed)
    torch.cuda.synchronize()
    return out


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_parity_scalar_fast_gate(sv, dtype):
    B, k, V = 40, 4, 30000
    w = peaked_workload(B, k, V, dtype, seed=81 + (dtype == "f32"), gate=1, tau=0.5)
    ver = _verifier(sv, w)
    out = _run_scalar_gate(sv, ver, w, 0.5)
    ref = oracle_for(w)
    compare(w, out, ref, what=f"scalar fast gate {dtype}")
    assert int((ref["flags"] == 3).sum()) > 0 and int((ref["flags"] == 1).sum()) > 0
    ver.close()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_candidate_overflow_on_the_fast_path_takes_the_chunk_pass(sv, dtype):
    # Every chunk of a draft row holds four equal spikes (in-chunk probability
    # ~1/4 each, above slack * 0.21), so a row yields 4 * 80 = 320 gate
    # candidates -- more than a sequence's candidate list holds.  The row's
    # admitted set is then unknown, and the stop row (position 0: q(D) is
    # ~1/320 < tau, a NULL) needs the dense residual, which the fast-path
    # kernel computes one chunk per pass.
    B, k, nch = 12, 2, 80
    V = nch * 2048
    g = torch.Generator(device="cuda")
    g.manual_seed(97 + (dtype == "f32"))
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    Lt = (torch.randn(B, k + 1, V, generator=g, device="cuda") * 2.0).to(dt)
    Ld = torch.full((B, k, V), -30.0, device="cuda")
    off = torch.randint(0, 2048 - 4, (B, k, nch), generator=g, device="cuda")
    idx = (torch.arange(nch, device="cuda") * 2048).view(1, 1, nch) + off
    for s_ in range(4):
        Ld.scatter_(2, idx + s_, 4.0)
    Ld = Ld.to(dt)
    u = torch.rand(B, k, V, generator=g, device="cuda").clamp_(1e-30, 1 - 1e-7)
    D = torch.argmax(Ld.float() - torch.log(-torch.log(u)), dim=2).to(torch.int32)
    w = workloads.Workload(name="spikes", Lt=Lt, Ld=Ld, D=D, T=1.0,
                           gate=torch.ones(B, dtype=torch.uint8, device="cuda"),
                           tau=torch.full((B,), 0.21, device="cuda"), philox_seed=5, B=B, k=k, V=V,
                           dtype=dtype)
    ver = _verifier(sv, w)
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=0.21, seed=w.philox_seed,
                  counters=cnt)
    torch.cuda.synchronize()
    ref = oracle_for(w)
    compare(w, out, ref, what=f"candidate overflow {dtype}")
    # every sequence stops at position 0 with a NULL and emits a residual token
    assert (ref["flags"][:, 0] == 3).all()
    assert (out["accepted_len"] == 0).all()
    assert int(cnt[2]) == B  # NULL stops
    ver.close()


def test_parity_mixed_dtypes(sv):
    B, k, V = 24, 2, 9000
    w = _custom(B, k, V, "bf16", 0.8, (np.arange(B) % 2), 0.4, seed=5)
    w.Ld = w.Ld.float().contiguous()
    ver = _verifier(sv, w)
    compare(w, _run(sv, ver, w), oracle_for(w), what="bf16 target, f32 draft")
    w2 = _custom(B, k, V, "f32", 0.8, 0, 0.4, seed=6)
    w2.Ld = w2.Ld.to(torch.bfloat16).contiguous()
    compare(w2, _run(sv, ver, w2), oracle_for(w2), what="f32 target, bf16 draft")
    ver.close()


def test_parity_k1_and_max_k(sv):
    for k in (1, 32):
        w = _custom(16, k, 700, "f32", 1.3, (np.arange(16) % 2), 0.35, seed=k, scale=1.0, noise=0.3)
        ver = _verifier(sv, w)
        compare(w, _run(sv, ver, w), oracle_for(w), what=f"k={k}")
        ver.close()


@pytest.mark.parametrize("V,dtype", [(4104, "bf16"), (4099, "bf16"), (2050, "f32"), (2047, "f32"), (7, "bf16")])
def test_parity_partial_last_chunks_and_unaligned_rows(sv, V, dtype):
    # the last chunk of a row: its whole 16-byte slots arrive by cp.async and
    # the rest (a partial slot, the -inf padding) by plain loads; odd V also
    # makes the rows unaligned, so every slot takes the plain path
    B, k = 24, 3
    w = _custom(B, k, V, dtype, 1.0, (np.arange(B) % 2), 0.3, seed=V + 11, scale=2.0, noise=0.5)
    ver = _verifier(sv, w)
    out = _run(sv, ver, w, row_stats=True)
    ref = oracle_for(w)
    compare(w, out, ref, what=f"partial V={V} {dtype}")
    rs = out["row_stats"].cpu().numpy().astype(np.float64)
    np.testing.assert_allclose(rs[..., 1], ref["row_stats"][..., 1], rtol=1e-5, atol=1e-5)
    ver.close()


# ------------------------------------------------------ tiny config, 1e5 trials

@pytest.mark.parametrize("gated", [0, 1])
def test_tiny_config_1e5_trials_bit_exact_and_chi_square(sv, gated):
    # tiny config: V=8, k=3, fp32, target N(0, 2^2), draft = target + N(0, 1), T = 1,
    # 1e5 trials that share the logits and draw their own drafts and uniforms
    base = workloads.make("tiny_v8_f32", seed=3, device="cuda")
    n = 100000
    g = torch.Generator(device="cuda")
    g.manual_seed(17)
    Lt = base.Lt.expand(n, -1, -1).contiguous()
    Ld = base.Ld.expand(n, -1, -1).contiguous()
    q = torch.softmax(Ld[0].double() / base.T, dim=-1)
    D = torch.stack([torch.multinomial(q[j].float(), n, replacement=True, generator=g)
                     for j in range(3)], dim=1).to(torch.int32)
    w = workloads.Workload(name="tiny", Lt=Lt, Ld=Ld, D=D, T=base.T,
                           gate=torch.full((n,), gated, dtype=torch.uint8, device="cuda"),
                           tau=torch.full((n,), 0.5, device="cuda"), philox_seed=99, B=n, k=3,
                           V=8, dtype="f32")
    ver = _verifier(sv, w)
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = _run(sv, ver, w, counters=cnt)
    ref = oracle_for(w)
    st = compare(w, out, ref, what=f"tiny gated={gated}")
    # V = 8: every boundary kind is rare; all of them together stay under 1e-5 of draws
    assert st["boundary"] <= 1e-5 * st["draws"] + 3
    # emitted tokens at position 0 follow p_0 (Pearson, alpha = 1e-4, dof 7)
    p0 = torch.softmax(Lt[0, 0].double() / base.T, dim=-1).cpu().numpy()
    tok0 = out["tokens"][:, 0].cpu().numpy()
    counts = np.bincount(tok0, minlength=8)
    stat = ((counts - n * p0) ** 2 / (n * p0)).sum()
    assert stat < chi2.ppf(1 - 1e-4, 7)
    # the same statistic against q (the drafter's law) must reject: the test has power
    q0 = q[0].cpu().numpy()
    assert ((counts - n * q0) ** 2 / (n * q0)).sum() > chi2.ppf(1 - 1e-4, 7)
    # counters agree with the outputs
    c = cnt.cpu().numpy()
    al = out["accepted_len"].cpu().numpy()
    assert c[1] == al.sum() and c[4] == (al == 3).sum() and c[6] == 0
    assert c[0] == np.minimum(al + 1, 3).sum()
    assert c[2] + c[3] == (al < 3).sum()
    ver.close()


# ------------------------------------------------------------- full configs

FULL = [
    ("b16_v32000_bf16", None, None),
    ("b64_v128256_zipf_gated", None, None),
    ("b256_v151936_f32_mixed", None, 48),
    ("b1024_v262144_zipf_stress", None, 40),
]


@pytest.mark.parametrize("name,B,sample", FULL)
def test_full_size_configs(sv, name, B, sample):
    w = workloads.make(name, seed=1234, device="cuda", B=B)
    ver = _verifier(sv, w)
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = _run(sv, ver, w, counters=cnt)
    if sample is None:
        ref = oracle_for(w, nthreads=16)
        idx = None
    else:
        rng = np.random.default_rng(7)
        idx = np.sort(rng.choice(w.B, size=sample, replace=False))
        ref = oracle_for(w, idx=idx)
    compare(w, out, ref, idx=idx, what=name)
    # whole-batch invariants at full size
    al = out["accepted_len"].cpu().numpy()
    tok = out["tokens"].cpu().numpy()
    assert np.all((al >= 0) & (al <= w.k))
    assert np.all((tok[np.arange(w.B), al] >= 0) & (tok[np.arange(w.B), al] < w.V))
    pad = np.arange(w.k + 1)[None, :] > al[:, None]
    assert np.all(tok[pad] == -1)
    c = cnt.cpu().numpy()
    assert c[1] == al.sum() and c[6] == 0
    ver.close()
    del w
    torch.cuda.empty_cache()


# The call the benchmark times: uniform gate settings given as the scalar
# arguments, so the host knows every row is on the candidate fast path and the
# finishing kernel without the dense pass runs -- at full size, every sequence
# of the 128K-vocabulary batch, and sampled sequences of the 262144-token one.
SCALAR_FULL = [
    ("b64_v128256_zipf_gated", None),
    ("b1024_v262144_zipf_stress", 48),
]


@pytest.mark.parametrize("name,sample", SCALAR_FULL)
def test_full_size_benchmarked_call_scalar_gate(sv, name, sample):
    w = workloads.make(name, seed=1234, device="cuda")
    cfg = workloads.CONFIGS[name]
    assert cfg["gate"] == "gated"
    ver = _verifier(sv, w)
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=float(cfg["tau"]),
                  seed=w.philox_seed, counters=cnt)
    torch.cuda.synchronize()
    if sample is None:
        ref = oracle_for(w, nthreads=16)
        idx = None
    else:
        rng = np.random.default_rng(11)
        idx = np.sort(rng.choice(w.B, size=sample, replace=False))
        ref = oracle_for(w, idx=idx)
    st = compare(w, out, ref, idx=idx, what=f"{name} scalar gate (benchmarked call)")
    assert st["compared"] >= (w.B if idx is None else len(idx)) // 2
    al = out["accepted_len"].cpu().numpy()
    c = cnt.cpu().numpy()
    assert np.all((al >= 0) & (al <= w.k)) and c[1] == al.sum() and c[6] == 0
    # the same call repeated gives the same outputs (the workspace is restored)
    again = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=float(cfg["tau"]),
                    seed=w.philox_seed)
    torch.cuda.synchronize()
    for key in ("accepted_len", "tokens", "accept_prob", "flags"):
        assert torch.equal(out[key], again[key]), key
    ver.close()
    del w
    torch.cuda.empty_cache()


# -------------------------------------------------------------- edge cases

def test_invalid_inputs_fail_closed_without_trapping(sv):
    B, k, V = 6, 3, 300
    w = _custom(B, k, V, "f32", 1.0, 0, 0.5, seed=2)
    w.Lt[1, 2, 5] = float("nan")
    w.Ld[2, 0, :] = float("-inf")
    w.D[3, 1] = V
    w.D[4, 0] = -1
    w.Lt[5, 0, 7] = float("inf")
    ver = _verifier(sv, w)
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = _run(sv, ver, w, counters=cnt)
    al = out["accepted_len"].cpu().numpy()
    assert al[0] >= 0 and np.all(al[1:] == -1)
    assert torch.all(out["tokens"][1:] == -1)
    assert torch.all(out["flags"][1:] == sv.SV_FLAG_INVALID)
    assert cnt[6].item() == 5
    # the context still works: a clean call afterwards
    w2 = _custom(B, k, V, "f32", 1.0, 0, 0.5, seed=3)
    compare(w2, _run(sv, ver, w2), oracle_for(w2), what="after invalid")
    ver.close()


def test_zero_target_mass_never_accepted_or_emitted(sv):
    n, V = 2000, 16
    Lt = torch.zeros(n, 2, V, device="cuda")
    Lt[:, :, 0] = float("-inf")
    Ld = torch.zeros(n, 1, V, device="cuda")
    Ld[:, 0, 0] = 5.0
    Ld[: n // 2, 0, 0] = float("-inf")  # q(D) = 0 too: u * 0 <= 0 must not accept
    D = torch.zeros(n, 1, dtype=torch.int32, device="cuda")
    for gated in (0, 1):
        w = workloads.Workload(name="support", Lt=Lt, Ld=Ld, D=D, T=1.0,
                               gate=torch.full((n,), gated, dtype=torch.uint8, device="cuda"),
                               tau=torch.full((n,), 0.3, device="cuda"), philox_seed=4, B=n, k=1,
                               V=V, dtype="f32")
        ver = _verifier(sv, w)
        out = _run(sv, ver, w)
        assert torch.all(out["accepted_len"] == 0)
        assert torch.all(out["tokens"][:, 0] != 0)
        assert torch.all(out["accept_prob"] == 0)
        compare(w, out, oracle_for(w), what=f"support gated={gated}")
        ver.close()


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_gate_equality_all_null_and_all_accepted(sv, dtype):
    # every draft and target row holds two equal logits (tokens 5 and 2100, in
    # different chunks of a ragged 4104-token row) and -inf elsewhere, so
    # q(D) = p(D) = 1/2 exactly in fp32: at tau = 1/2 the gate admits D
    # (equality passes), alpha = 1 and every sequence takes the bonus; at the
    # next float above 1/2 every position-0 draft is an explicit NULL row and
    # the residual (mu = 0 everywhere) samples p
    B, k, V, hot = 64, 2, 4104, (5, 2100)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    Lt = torch.full((B, k + 1, V), float("-inf"), device="cuda")
    Lt[:, :, list(hot)] = 0.0
    Ld = Lt[:, :k].clone()
    D = torch.tensor(hot, dtype=torch.int32, device="cuda")[torch.arange(B * k, device="cuda") % 2]
    D = D.view(B, k).contiguous()
    above = float(np.nextafter(np.float32(0.5), np.float32(1.0)))
    for tau, want_len, want_flag in ((0.5, k, 1), (above, 0, 3)):
        w = workloads.Workload(name="equality", Lt=Lt.to(dt), Ld=Ld.to(dt), D=D, T=1.0,
                               gate=torch.ones(B, dtype=torch.uint8, device="cuda"),
                               tau=torch.full((B,), tau, device="cuda"), philox_seed=17, B=B, k=k,
                               V=V, dtype=dtype)
        ver = _verifier(sv, w)
        for scalar in (False, True):
            if scalar:  # the same setting given as the scalar arguments
                out = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=sv.SV_GATED_MU, threshold=tau,
                              seed=w.philox_seed)
                torch.cuda.synchronize()
            else:
                out = _run(sv, ver, w)
            assert torch.all(out["accepted_len"] == want_len), (tau, scalar)
            assert torch.all(out["flags"][:, 0] == want_flag), (tau, scalar)
            emitted = out["tokens"][:, want_len]
            assert torch.all((emitted == hot[0]) | (emitted == hot[1])), (tau, scalar)
            if want_len == k:
                assert torch.all(out["accept_prob"] == 1.0)
                assert torch.equal(out["tokens"][:, :k], D)
            else:
                assert torch.all(out["accept_prob"][:, 0] == 0.0)
                assert torch.all(out["tokens"][:, 1:] == -1)
        ref = oracle_for(w)
        assert np.all(ref["accepted_len"] == want_len)
        assert np.array_equal(out["tokens"].cpu().numpy(), ref["tokens"])
        ver.close()


def test_plain_draft_with_zero_proposal_mass_is_accepted(sv):
    # plain mode, q(D) = 0 (the drafted token's logit is -inf) and p(D) > 0:
    # u0 * 0 <= p(D) always holds, so the draft is accepted with alpha = 1
    B, k, V = 256, 1, 3000
    w = _custom(B, k, V, "f32", 1.0, 0, 0.5, seed=23)
    Ld = w.Ld.clone()
    Ld.view(B * k, V)[torch.arange(B * k, device="cuda"), w.D.view(-1).long()] = float("-inf")
    w = workloads.Workload(name="zero_q", Lt=w.Lt, Ld=Ld, D=w.D, T=1.0, gate=w.gate, tau=w.tau,
                           philox_seed=w.philox_seed, B=B, k=k, V=V, dtype="f32")
    ver = _verifier(sv, w)
    out = _run(sv, ver, w)
    assert torch.all(out["flags"][:, 0] == 1)
    assert torch.all(out["accept_prob"][:, 0] == 1.0)
    assert torch.all(out["accepted_len"] == k)
    compare(w, out, oracle_for(w), what="zero proposal mass")
    ver.close()


def test_explicit_uniforms_probe_decisions(sv):
    # u0 at 0 accepts everything with p > 0; u0 just below 1 rejects every ratio < 1
    B, k, V = 32, 4, 5000
    w = _custom(B, k, V, "bf16", 1.0, (np.arange(B) % 2), 0.3, seed=8)
    ver = _verifier(sv, w)
    for u0v, u1v in ((0.0, 0.0), (1.0 - 2.0 ** -24, 1.0 - 2.0 ** -24), (0.5, 0.25)):
        u0 = torch.full((B, k), u0v, device="cuda")
        u1 = torch.full((B,), u1v, device="cuda")
        out = _run(sv, ver, w, u_accept=u0, u_residual=u1)
        u0n, u1n = u0.double().cpu().numpy(), u1.double().cpu().numpy()
        ref = oracle_for(w, u0=u0n, u1=u1n)
        compare(w, out, ref, what=f"u0={u0v} u1={u1v}", u0=u0n, u1=u1n)
    ver.close()


def test_sequence_offset_splits_match_the_whole_batch(sv):
    B, k, V = 32, 3, 4000
    w = _custom(B, k, V, "bf16", 0.9, (np.arange(B) % 2), 0.45, seed=12)
    ver = _verifier(sv, w)
    full = _run(sv, ver, w)
    halves = []
    for lo in (0, 16):
        sl = slice(lo, lo + 16)
        out = ver.run(w.Lt[sl].contiguous(), w.Ld[sl].contiguous(), w.D[sl].contiguous(), w.T,
                      gate_mode=sv.SV_GATED_MU, threshold=0.5,
                      gate_per_seq=w.gate[sl].contiguous(), threshold_per_seq=w.tau[sl].contiguous(),
                      seed=w.philox_seed, seq_offset=lo)
        halves.append(out)
    torch.cuda.synchronize()
    for key in ("accepted_len", "tokens", "accept_prob", "flags"):
        assert torch.equal(torch.cat([h[key] for h in halves]), full[key]), key
    ver.close()


def test_repeated_calls_are_deterministic_and_reset_state(sv):
    w = workloads.make("b16_v32000_bf16", seed=21, device="cuda")
    ver = _verifier(sv, w, max_B=64)
    a = _run(sv, ver, w)
    b = _run(sv, ver, w)
    for key in a:
        assert torch.equal(a[key], b[key]), key
    # a smaller batch on the same handle, then the full one again
    small = ver.run(w.Lt[:3].contiguous(), w.Ld[:3].contiguous(), w.D[:3].contiguous(), w.T,
                    seed=w.philox_seed)
    c = _run(sv, ver, w)
    torch.cuda.synchronize()
    for key in a:
        assert torch.equal(a[key], c[key]), key
        assert torch.equal(a[key][:3], small[key]), key
    ver.close()


def test_host_side_argument_errors(sv):
    w = _custom(4, 2, 100, "f32", 1.0, 0, 0.5, seed=1)
    ver = _verifier(sv, w)
    with pytest.raises(sv.SpecVerifyError):
        ver.run(w.Lt, w.Ld, w.D, -1.0)
    with pytest.raises(sv.SpecVerifyError):
        ver.run(w.Lt, w.Ld, w.D, float("nan"))
    with pytest.raises(sv.SpecVerifyError):
        ver.run(w.Lt, w.Ld, w.D, float("inf"))
    with pytest.raises(sv.SpecVerifyError):
        ver.run(w.Lt, w.Ld, w.D, 1.0, gate_mode=sv.SV_GATED_MU, threshold=0.0)
    with pytest.raises(sv.SpecVerifyError):
        ver.run(w.Lt, w.Ld, w.D, 1.0, gate_mode=sv.SV_GATED_MU, threshold=1.5)
    big = _custom(5, 2, 100, "f32", 1.0, 0, 0.5, seed=1)
    with pytest.raises(sv.SpecVerifyError):
        ver.run(big.Lt, big.Ld, big.D, 1.0)
    # per-sequence threshold outside (0, 1]: that sequence alone is invalid
    tau = torch.tensor([0.5, 0.0, 0.5, 2.0], device="cuda")
    out = ver.run(w.Lt, w.Ld, w.D, 1.0, gate_mode=sv.SV_GATED_MU, threshold=0.5,
                  threshold_per_seq=tau)
    torch.cuda.synchronize()
    al = out["accepted_len"].cpu().numpy()
    assert al[1] == -1 and al[3] == -1 and al[0] >= 0 and al[2] >= 0
    ver.close()


def test_host_buffer_entry_point_matches_device_path(sv):
    w = workloads.make("b16_v32000_bf16", seed=31, device="cuda")
    ver = _verifier(sv, w)
    dev = ver.run(w.Lt, w.Ld, w.D, w.T, seed=w.philox_seed)
    torch.cuda.synchronize()
    host = ver.run_host(w.Lt.cpu().pin_memory(), w.Ld.cpu().pin_memory(), w.D.cpu().pin_memory(),
                        w.T, seed=w.philox_seed)
    for key in ("accepted_len", "tokens", "accept_prob", "flags"):
        assert torch.equal(dev[key].cpu(), host[key]), key
    ver.close()


@pytest.mark.parametrize("mode", ["gated_scalar", "greedy", "plain"])
def test_host_buffer_entry_point_reads_pinned_logits_in_place(sv, mode):
    # pinned logits are read in place by the fast-path and greedy calls, and
    # staged by a call with dense residuals; every way matches the device path
    w = peaked_workload(24, 4, 20000, "bf16", seed=57, gate=1, tau=0.5, T=0.0 if mode == "greedy" else 1.0)
    ver = _verifier(sv, w)
    gm = sv.SV_PLAIN if mode == "plain" else sv.SV_GATED_MU
    dev = ver.run(w.Lt, w.Ld, w.D, w.T, gate_mode=gm, threshold=0.5, seed=w.philox_seed)
    torch.cuda.synchronize()
    host = ver.run_host(w.Lt.cpu().pin_memory(), w.Ld.cpu().pin_memory(), w.D.cpu().pin_memory(),
                        w.T, gate_mode=gm, threshold=0.5, seed=w.philox_seed)
    for key in ("accepted_len", "tokens", "accept_prob", "flags"):
        assert torch.equal(dev[key].cpu(), host[key]), key
    ver.close()


# ------------------------------------------------------ temperature 0 (greedy)

def _greedy_custom(B, k, V, dtype, seed, gate):
    """Integer-valued logits (exact ties across and inside chunks) with drafted
    tokens that often equal a row's argmax."""
    g = torch.Generator(device="cuda")
    g.manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    t = torch.randint(-6, 7, (B, k + 1, V), generator=g, device="cuda").float()
    d = t[:, :k] + torch.randint(-1, 2, (B, k, V), generator=g, device="cuda").float()
    ta, da = torch.argmax(t[:, :k], dim=2), torch.argmax(d, dim=2)
    r = torch.rand(B, k, generator=g, device="cuda")
    rnd = torch.randint(0, V, (B, k), generator=g, device="cuda")
    D = torch.where(r < 0.7, ta, torch.where(r < 0.85, da, rnd)).to(torch.int32)
    gate_t = torch.as_tensor(np.broadcast_to(np.asarray(gate, dtype=np.uint8), (B,)).copy(), device="cuda")
    tau_t = torch.full((B,), 0.5, dtype=torch.float32, device="cuda")
    return workloads.Workload(name="greedy", Lt=t.to(dt), Ld=d.to(dt), D=D, T=0.0, gate=gate_t, tau=tau_t,
                              philox_seed=seed + 2, B=B, k=k, V=V, dtype=dtype)


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
@pytest.mark.parametrize("V", [20000, 4096, 67, 1])
def test_greedy_parity(sv, dtype, V):
    B, k = 48, 5
    gate = (np.arange(B) % 2).astype(np.uint8)
    w = _greedy_custom(B, k, V, dtype, seed=V + 3 * (dtype == "f32"), gate=gate)
    ver = _verifier(sv, w)
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    rs = ver.run(w.Lt, w.Ld, w.D, 0.0, gate_mode=sv.SV_GATED_MU, threshold=0.5, gate_per_seq=w.gate,
                 threshold_per_seq=w.tau, seed=w.philox_seed, counters=cnt, row_stats=True)
    torch.cuda.synchronize()
    ref = oracle_for(w)
    compare(w, rs, ref, what=f"greedy {dtype} V={V}")
    # alpha is exactly 0 or 1, row statistics are (max L, max L)
    a = rs["accept_prob"].cpu().numpy()
    assert np.all((a == 0.0) | (a == 1.0))
    np.testing.assert_array_equal(rs["row_stats"].cpu().numpy().astype(np.float64), ref["row_stats"])
    c = cnt.cpu().numpy()
    assert c[1] == ref["accepted_len"].sum() and c[5] == 0 and c[7] == ref["degenerate"].sum()
    ver.close()


def test_greedy_full_size_128k(sv):
    w = workloads.make("b64_v128256_zipf_gated", seed=1234, device="cuda")
    w.T = 0.0
    for gate in (None, "plain"):
        if gate is not None:
            w = workloads.make("b64_v128256_zipf_gated", seed=1234, device="cuda", gate=gate)
            w.T = 0.0
        ver = _verifier(sv, w)
        out = ver.run(w.Lt, w.Ld, w.D, 0.0, gate_mode=sv.SV_GATED_MU, threshold=0.5,
                      gate_per_seq=w.gate, threshold_per_seq=w.tau, seed=w.philox_seed)
        torch.cuda.synchronize()
        compare(w, out, oracle_for(w, nthreads=16), what=f"greedy 128k {gate}")
        ver.close()
