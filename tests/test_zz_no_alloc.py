"""The allocation-free entry point (spec_verify_run_noalloc) against the
handle-based spec_verify_run on the same inputs: the same kernels run on a
static workspace buffer, so every output must match bit for bit.  Two calls in
a row per case check that a call leaves the buffer ready for the next one (the
gate candidate slots are emptied again).  Kept in a file of its own, collected
last, so it also runs after every other GPU test in the same process."""
from __future__ import annotations

import ctypes

import numpy as np
import pytest
import torch

import workloads
from speculative_decoding_verification_online_gb300 import spec_verify as svm

SV_OK, SV_EINVAL, SV_EUNSUPPORTED = 0, 1, 4


def _raw(B, k, V, ptrs=None):
    """The raw call with size arguments only (and optional output pointers)."""
    p = ptrs or {}
    return svm.spec_verify_run_noalloc(None, svm.SV_BF16, None, svm.SV_BF16, None, B, k, V, 1.0,
                                       svm.SV_PLAIN, 0.5, None, None, 0, p.get("al"), p.get("tok"),
                                       p.get("ap"), p.get("fl"), None, None)


def test_noalloc_checks_sizes_before_touching_the_device():
    svm.load()
    assert _raw(4, 0, 100) == SV_EINVAL
    assert _raw(4, 3, 0) == SV_EINVAL
    assert _raw(-1, 3, 100) == SV_EINVAL
    assert _raw(4, 33, 100) == SV_EUNSUPPORTED
    # B=256, k=8, V=151936 needs 614,400 candidate slots > 2^19
    assert _raw(256, 8, 151936) == SV_EUNSUPPORTED
    # B * k beyond the row-flag region
    assert _raw(20000, 1, 1) == SV_EUNSUPPORTED
    assert _raw(0, 5, 128256) == SV_OK  # empty batch: nothing to do


gpu = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_online_gb300 as pkg
    from speculative_decoding_verification_online_gb300 import build as B
    B.build()
    pkg.load()
    return pkg


def _pair(sv, w, ver, counters):
    kw = dict(gate_mode=sv.SV_GATED_MU, threshold=0.5, gate_per_seq=w.gate,
              threshold_per_seq=w.tau, seed=w.philox_seed)
    c_ref = torch.zeros(8, dtype=torch.int64, device="cuda") if counters else None
    c_na = torch.zeros(8, dtype=torch.int64, device="cuda") if counters else None
    ref = ver.run(w.Lt, w.Ld, w.D, w.T, counters=c_ref, **kw)
    got = sv.run_noalloc(w.Lt, w.Ld, w.D, w.T, counters=c_na, **kw)
    torch.cuda.synchronize()
    for name in ("accepted_len", "tokens", "accept_prob", "flags"):
        assert torch.equal(ref[name], got[name]), name
    if counters:
        assert torch.equal(c_ref, c_na)
    return ref


@gpu
@pytest.mark.parametrize("name,B,gate", [
    ("b16_v32000_bf16", None, None),          # plain: dense residual re-read
    ("b64_v128256_zipf_gated", 16, None),     # gated: candidate slots used and emptied
    ("b64_v128256_zipf_gated", 16, "plain"),
    ("tiny_v8_f32", None, "gated"),
])
def test_noalloc_matches_the_handle_path_on_two_calls_in_a_row(sv, name, B, gate):
    w1 = workloads.make(name, seed=101, device="cuda", B=B, gate=gate)
    w2 = workloads.make(name, seed=202, device="cuda", B=B, gate=gate)
    ver = sv.SpecVerifier(w1.B, w1.k, w1.V, device=0)
    try:
        a = _pair(sv, w1, ver, counters=True)
        b = _pair(sv, w2, ver, counters=False)
        # the two calls saw different inputs (a stale buffer could not pass both)
        assert not torch.equal(a["accept_prob"], b["accept_prob"])
    finally:
        ver.close()


@gpu
def test_noalloc_mixed_dtypes_and_shapes_back_to_back(sv):
    # shapes change from call to call: the fixed buffer layout keeps the
    # candidate slots valid for any of them
    shapes = [(8, 3, 5000, "f32", "bf16"), (3, 7, 40000, "bf16", "f32"), (8, 3, 5000, "f32", "bf16")]
    for i, (B, k, V, dt_t, dt_d) in enumerate(shapes):
        g = torch.Generator(device="cuda")
        g.manual_seed(900 + i)
        t = torch.randn(B, k + 1, V, generator=g, device="cuda") * 3.0
        t[:, :, 7] += 9.0  # a dominant token, so that gated rows keep candidates
        d = t[:, :k] + torch.randn(B, k, V, generator=g, device="cuda") * 0.5
        Lt = t.to(torch.float32 if dt_t == "f32" else torch.bfloat16)
        Ld = d.to(torch.float32 if dt_d == "f32" else torch.bfloat16)
        D = torch.argmax(Ld.float(), dim=2).to(torch.int32)
        gate = torch.ones(B, dtype=torch.uint8, device="cuda")
        tau = torch.full((B,), 0.4, dtype=torch.float32, device="cuda")
        w = workloads.Workload(name="custom", Lt=Lt, Ld=Ld, D=D, T=1.0, gate=gate, tau=tau,
                               philox_seed=33 + i, B=B, k=k, V=V, dtype=dt_t)
        ver = sv.SpecVerifier(B, k, V, device=0)
        try:
            _pair(sv, w, ver, counters=True)
        finally:
            ver.close()


@gpu
def test_noalloc_oversize_launches_nothing(sv):
    B, k = 256, 8
    al = torch.full((B,), 12345, dtype=torch.int32, device="cuda")
    tok = torch.full((B, k + 1), 12345, dtype=torch.int32, device="cuda")
    ap = torch.full((B, k), 7.0, dtype=torch.float32, device="cuda")
    fl = torch.full((B, k), 9, dtype=torch.int8, device="cuda")
    rc = _raw(B, k, 151936, dict(al=al.data_ptr(), tok=tok.data_ptr(), ap=ap.data_ptr(),
                                 fl=fl.data_ptr()))
    torch.cuda.synchronize()
    assert rc == SV_EUNSUPPORTED
    assert bool((al == 12345).all()) and bool((tok == 12345).all())
    assert bool((ap == 7.0).all()) and bool((fl == 9).all())
