"""The synthetic input recipe (workloads/synthetic.py) on small CPU samples:
shapes and types of every named workload, the Zipf and normal target rows, the
draft rows as scale * target + noise, drafted tokens distributed as
softmax(Ld / T), the gate recipes, and seeding."""
from __future__ import annotations

import numpy as np
import pytest
import torch
from scipy.stats import chi2

import workloads

SMALL_B = {"tiny_v8_f32": 1, "b16_v32000_bf16": 4, "b64_v128256_zipf_gated": 2,
           "b256_v151936_f32_mixed": 2, "b1024_v262144_zipf_stress": 1}


@pytest.mark.parametrize("name", sorted(workloads.CONFIGS))
def test_shapes_types_and_seeding(name):
    cfg = workloads.CONFIGS[name]
    B, k, V = SMALL_B[name], cfg["k"], cfg["V"]
    w = workloads.make(name, seed=3, B=B)
    dt = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
    assert w.Lt.shape == (B, k + 1, V) and w.Lt.dtype == dt
    assert w.Ld.shape == (B, k, V) and w.Ld.dtype == dt
    assert w.D.shape == (B, k) and w.D.dtype == torch.int32
    assert bool(((w.D >= 0) & (w.D < V)).all())
    assert (w.T, w.philox_seed) == (float(cfg["T"]), 5)
    assert w.logits_bytes() == B * (2 * k + 1) * V * (2 if cfg["dtype"] == "bf16" else 4)
    again = workloads.make(name, seed=3, B=B)
    assert torch.equal(again.Lt, w.Lt) and torch.equal(again.Ld, w.Ld) and torch.equal(again.D, w.D)
    other = workloads.make(name, seed=4, B=B)
    assert not torch.equal(other.Lt, w.Lt)


def test_zipf_rows_follow_minus_s_log_rank():
    # no noise: every row is a permutation of -1.0 ln(rank), rank = 1..V, up
    # to the bf16 rounding of the stored values (half an ulp: 2^-9 relative)
    w = workloads.make("b1024_v262144_zipf_stress", seed=1, B=1)
    want = -np.log(np.arange(1, w.V + 1, dtype=np.float64))
    for row in w.Lt[0].float().numpy().astype(np.float64):
        got = -np.sort(-row)
        assert np.all(np.abs(got - want) <= 2.0 ** -8 * np.abs(want) + 1e-6)
    # rows differ: the permutation is drawn per row
    assert not torch.equal(w.Lt[0, 0], w.Lt[0, 1])
    # with noise N(0, 0.3^2) the sorted logits still fall with slope about
    # -1.1 against ln(rank)
    w = workloads.make("b64_v128256_zipf_gated", seed=2, B=1)
    srt = -np.sort(-w.Lt[0, 0].float().numpy().astype(np.float64))
    x = np.log(np.arange(1, w.V + 1, dtype=np.float64))
    slope = np.polyfit(x[100:], srt[100:], 1)[0]
    assert -1.25 < slope < -0.95


@pytest.mark.parametrize("name,scale,noise", [("b16_v32000_bf16", 1.0, 0.5),
                                              ("b1024_v262144_zipf_stress", 0.7, 1.0)])
def test_draft_rows_are_scaled_target_plus_noise(name, scale, noise):
    w = workloads.make(name, seed=6, B=1)
    k = w.k
    resid = (w.Ld.float() - scale * w.Lt[:, :k].float()).numpy().ravel()
    assert abs(resid.mean()) < 0.01
    # bf16 storage adds rounding of a few 2^-8 relative; the noise dominates
    assert abs(resid.std() - noise) < 0.05 * noise


def test_normal_target_rows_have_the_stated_spread():
    w = workloads.make("b16_v32000_bf16", seed=8, B=2)
    x = w.Lt.float().numpy().ravel()
    assert abs(x.mean()) < 0.02 and abs(x.std() - 3.0) < 0.02


def test_drafted_tokens_are_distributed_as_q():
    # every drafted token is a draw from its row's softmax(Ld / T): over many
    # rows, the counts of each token match the summed probabilities
    w = workloads.make("tiny_v8_f32", seed=11, B=20000)
    q = torch.softmax(w.Ld.double() / w.T, dim=2).reshape(-1, w.V).numpy()
    d = w.D.reshape(-1).numpy()
    expect = q.sum(axis=0)
    seen = np.bincount(d, minlength=w.V)
    stat = ((seen - expect) ** 2 / expect).sum()
    assert stat < chi2.ppf(1 - 1e-4, w.V - 1), (seen, expect)
    # and each token's own probability is what the draws favour: the mean
    # q(D) exceeds the mean q of a uniformly chosen token
    assert q[np.arange(len(d)), d].mean() > q.mean() * 1.2


def test_gate_recipes():
    w = workloads.make("b256_v151936_f32_mixed", seed=1, B=6)
    assert w.gate.tolist() == [0, 0, 0, 1, 1, 1]
    assert torch.all(w.tau == 0.3)
    assert workloads.make("b64_v128256_zipf_gated", seed=1, B=2).gate.tolist() == [1, 1]
    assert workloads.make("b16_v32000_bf16", seed=1, B=2).gate.tolist() == [0, 0]
    assert workloads.make("b16_v32000_bf16", seed=1, B=2, gate="gated").gate.tolist() == [1, 1]
    with pytest.raises(ValueError):
        workloads.make("b16_v32000_bf16", seed=1, B=2, gate="other")


def test_peaked_rows_raise_one_token_by_eight_in_half_the_rows():
    # the peaked recipe draws the same normal rows as the plain one, then adds
    # +8 to one random token of each row with probability 1/2
    from workloads import synthetic as S
    n, V = 4000, 64
    g1, g2 = torch.Generator(), torch.Generator()
    g1.manual_seed(5)
    g2.manual_seed(5)
    peaked = S._target_rows(("peaked", 4.0, 8.0, 0.5), n, V, g1, torch.device("cpu"))
    plain = S._target_rows(("normal", 4.0), n, V, g2, torch.device("cpu"))
    diff = (peaked - plain).numpy()
    changed = np.count_nonzero(diff, axis=1)
    assert set(np.unique(changed)) <= {0, 1}
    assert np.allclose(diff[changed == 1].max(axis=1), 8.0, atol=1e-5)
    frac = (changed == 1).mean()
    assert abs(frac - 0.5) < 4 * np.sqrt(0.25 / n)
