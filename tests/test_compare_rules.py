"""The parity comparison's rules, checked on the CPU with results made by the
oracle itself: a result that differs from the oracle only inside a boundary
band, in a way a lower-precision computation could, is accepted; a wrong token
or a flipped decision away from every boundary is not.  (The GPU parity tests
apply the same rules to the CUDA path.)"""
import numpy as np
import pytest
import torch

import workloads
from oracle import oracle as O
from tests.gpu_helpers import compare


def _case(seed=3, B=12, k=3, V=50, gate=1, tau=0.3):
    g = torch.Generator().manual_seed(seed)
    Lt = torch.randn(B, k + 1, V, generator=g) * 2.0
    Ld = Lt[:, :k] + torch.randn(B, k, V, generator=g)
    D = torch.argmax(Ld, dim=2).to(torch.int32)
    D[::3, 0] = torch.randint(0, V, (len(range(0, B, 3)),), generator=g).to(torch.int32)
    return workloads.Workload(name="rules", Lt=Lt, Ld=Ld, D=D, T=1.0,
                              gate=torch.full((B,), gate, dtype=torch.uint8),
                              tau=torch.full((B,), tau), philox_seed=9, B=B, k=k, V=V, dtype="f32")


def _ref(w, u0=None, u1=None):
    return O.verify(w.Lt.numpy(), w.Ld.numpy(), w.D.numpy(), w.T, w.gate.numpy(),
                    w.tau.numpy().astype(np.float64), seed=w.philox_seed, u0=u0, u1=u1)


def _got(ref):
    return {"accepted_len": torch.as_tensor(ref["accepted_len"].copy()),
            "tokens": torch.as_tensor(ref["tokens"].copy()),
            "accept_prob": torch.as_tensor(ref["alpha"].astype(np.float32)),
            "flags": torch.as_tensor(ref["flags"].copy())}


def test_identical_results_pass():
    w = _case()
    ref = _ref(w)
    st = compare(w, _got(ref), ref, what="identical")
    assert st["boundary_mismatch"] == 0 and st["compared"] + st["boundary"] == w.B


def test_a_wrong_token_away_from_every_boundary_fails():
    w = _case()
    ref = _ref(w)
    b = int(np.nonzero(ref["margin"] >= 1e-6)[0][0])
    got = _got(ref)
    j = int(ref["accepted_len"][b])
    got["tokens"][b, j] = (got["tokens"][b, j] + 1) % w.V
    with pytest.raises(AssertionError, match="non-boundary"):
        compare(w, got, ref, what="planted")


def _edge_u1(w, b, j, v):
    """u1 exactly at the upper end of token v's interval of the stop row j."""
    Lt, Ld, D = w.Lt[b].numpy(), w.Ld[b].numpy(), w.D[b].numpy()
    _, _, hi, _ = O.pick_interval(Lt, Ld, D, w.T, int(w.gate[b]), float(w.tau[b]), j, v)
    return hi


def test_a_neighbouring_pick_at_an_interval_edge_is_accepted_and_a_distant_one_is_not():
    w = _case(gate=0)
    # explicit uniforms: every draft accepted (u0 = 0) so every sequence takes
    # the bonus row k; u1 at the upper edge of the oracle's own pick, so a
    # lower-precision pick may land on the next token with weight
    B, k = w.B, w.k
    u0 = np.zeros((B, k))
    ref0 = _ref(w, u0=u0, u1=np.full(B, 0.5))
    u1 = np.array([_edge_u1(w, b, k, int(ref0["tokens"][b, k])) for b in range(B)])
    ref = _ref(w, u0=u0, u1=u1)
    assert np.all(ref["margin_pick"] < 1e-6)
    got = _got(ref)
    # the oracle now picks the token whose interval starts at u1; the result
    # under test keeps the token whose interval ends there
    got["tokens"][:, k] = torch.as_tensor(ref0["tokens"][:, k])
    st = compare(w, got, ref, what="edge picks", u0=u0, u1=u1)
    assert st["mismatch_pick"] == st["boundary_mismatch"] > 0
    got["tokens"][0, k] = (int(ref["tokens"][0, k]) + 7) % w.V
    with pytest.raises(AssertionError, match="does not explain"):
        compare(w, got, ref, what="distant pick", u0=u0, u1=u1)


def test_a_flipped_decision_needs_its_draw_at_the_boundary():
    w = _case(gate=0)
    B, k = w.B, w.k
    ref1 = _ref(w, u0=np.zeros((B, k)), u1=np.full(B, 0.3))
    a0 = ref1["alpha"][:, 0]
    b = int(np.nonzero((a0 > 0) & (a0 < 1))[0][0])
    # u0 at position 0 exactly alpha_0: the oracle accepts (equality passes);
    # a lower-precision test may reject there and emit a residual token
    u0 = np.zeros((B, k))
    u0[b, 0] = a0[b]
    u1 = np.full(B, 0.3)
    ref = _ref(w, u0=u0, u1=u1)
    assert ref["accepted_len"][b] == k and ref["margin"][b] < 1e-6
    # the rejected branch, as the oracle computes it (u0 a little above alpha)
    u0r = u0.copy()
    u0r[b, 0] = a0[b] + 1e-9
    rej = _ref(w, u0=u0r, u1=u1)
    assert rej["accepted_len"][b] == 0
    got = _got(ref)
    got["accepted_len"][b] = 0
    got["tokens"][b] = torch.as_tensor(rej["tokens"][b])
    got["flags"][b] = torch.as_tensor(rej["flags"][b])
    st = compare(w, got, ref, what="flip at the boundary", u0=u0, u1=u1)
    assert st["mismatch_decision"] == 1
    # the same flip with u0 far from alpha is not a boundary case
    u0f = u0.copy()
    u0f[b, 0] = 0.0
    reff = _ref(w, u0=u0f, u1=u1)
    reff["margin"][b] = 0.0  # even if the sequence counted as a boundary one
    with pytest.raises(AssertionError, match="does not explain"):
        compare(w, got, reff, what="flip away from the boundary", u0=u0f, u1=u1)
