"""Synthetic verification workloads, seeded and reproducible.

Each workload is a batch of B sequences with k draft positions over a
vocabulary of V tokens: target logits [B, k+1, V], draft logits [B, k, V],
drafted tokens [B, k] (drawn from the draft distribution softmax(Ld / T) by
the Gumbel-max trick, i.e. "draft tokens sampled from q"), a temperature, and
a per-sequence gate mode and threshold.

Value recipes (one per named workload):
  tiny_v8_f32              B=1,    k=3, V=8,      f32,  target N(0, 2^2), draft = target + N(0, 1),
                           T=1.0, plain or gated (threshold 0.5)
  b16_v32000_bf16          B=16,   k=4, V=32000,  bf16, target N(0, 3^2), draft = target + N(0, 0.5^2),
                           T=0.7, plain
  b64_v128256_zipf_gated   B=64,   k=5, V=128256, bf16, target -1.1 ln(rank) + N(0, 0.3^2), ranks a
                           random permutation per row, draft = target + N(0, 1), T=1.0, gated 0.5
  b256_v151936_f32_mixed   B=256,  k=8, V=151936, f32,  target N(0, 4^2) plus +8 on one random token
                           in half the rows (Bernoulli per row), draft = target + N(0, 0.8^2),
                           T=0.8, sequences b < B/2 plain, b >= B/2 gated (threshold 0.3)
  b1024_v262144_zipf_stress B=1024, k=4, V=262144, bf16, target -1.0 ln(rank) (no noise), draft =
                           0.7 target + N(0, 1), T=1.0, gated 0.5

The target logits come from a generator seeded with ``seed``, drafted tokens
from ``seed + 1``; the verifier's Philox seed is ``seed + 2``.  Rows are made
in blocks so that device memory stays bounded at the largest sizes.
"""
from __future__ import annotations

import dataclasses

import numpy as np
import torch

CONFIGS = {
    "tiny_v8_f32": dict(B=1, k=3, V=8, dtype="f32", T=1.0, target=("normal", 2.0),
                        draft=(1.0, 1.0), gate="plain", tau=0.5),
    "b16_v32000_bf16": dict(B=16, k=4, V=32000, dtype="bf16", T=0.7, target=("normal", 3.0),
                            draft=(1.0, 0.5), gate="plain", tau=0.5),
    "b64_v128256_zipf_gated": dict(B=64, k=5, V=128256, dtype="bf16", T=1.0,
                                   target=("zipf", 1.1, 0.3), draft=(1.0, 1.0), gate="gated",
                                   tau=0.5),
    "b256_v151936_f32_mixed": dict(B=256, k=8, V=151936, dtype="f32", T=0.8,
                                   target=("peaked", 4.0, 8.0, 0.5), draft=(1.0, 0.8),
                                   gate="half", tau=0.3),
    "b1024_v262144_zipf_stress": dict(B=1024, k=4, V=262144, dtype="bf16", T=1.0,
                                      target=("zipf", 1.0, 0.0), draft=(0.7, 1.0), gate="gated",
                                      tau=0.5),
}


@dataclasses.dataclass
class Workload:
    name: str
    Lt: torch.Tensor          # [B, k+1, V] target logits
    Ld: torch.Tensor          # [B, k, V]   draft logits
    D: torch.Tensor           # [B, k]      int32 drafted tokens
    T: float
    gate: torch.Tensor        # [B] uint8, 0 plain, 1 gated
    tau: torch.Tensor         # [B] float32 thresholds
    philox_seed: int
    B: int
    k: int
    V: int
    dtype: str

    def logits_bytes(self) -> int:
        return self.Lt.numel() * self.Lt.element_size() + self.Ld.numel() * self.Ld.element_size()


def _target_rows(kind, n, V, gen, device):
    if kind[0] == "normal":
        return torch.randn(n, V, generator=gen, device=device) * kind[1]
    if kind[0] == "peaked":
        x = torch.randn(n, V, generator=gen, device=device) * kind[1]
        hit = torch.rand(n, generator=gen, device=device) < kind[3]
        tok = torch.randint(0, V, (n,), generator=gen, device=device)
        rows = torch.arange(n, device=device)
        x[rows[hit], tok[hit]] += kind[2]
        return x
    if kind[0] == "zipf":
        # argsort of iid uniforms is a uniformly random permutation: the rank of each token
        rank = torch.argsort(torch.rand(n, V, generator=gen, device=device), dim=1).float() + 1.0
        x = -kind[1] * torch.log(rank)
        if kind[2] > 0:
            x += torch.randn(n, V, generator=gen, device=device) * kind[2]
        return x
    raise ValueError(kind)


def make(name: str, seed: int = 0, device="cpu", B: int | None = None, gate: str | None = None,
         block_rows: int = 64) -> Workload:
    """Build workload ``name`` (a key of CONFIGS) on ``device``.

    ``B`` overrides the batch size (smaller samples or shards); ``gate``
    overrides the gate recipe ("plain", "gated" or "half").
    """
    cfg = CONFIGS[name]
    B = cfg["B"] if B is None else B
    k, V, T = cfg["k"], cfg["V"], float(cfg["T"])
    dt = torch.bfloat16 if cfg["dtype"] == "bf16" else torch.float32
    device = torch.device(device)
    gen = torch.Generator(device=device)
    gen.manual_seed(seed)
    gen_d = torch.Generator(device=device)
    gen_d.manual_seed(seed + 1)
    scale, noise = cfg["draft"]

    Lt = torch.empty(B, k + 1, V, dtype=dt, device=device)
    Ld = torch.empty(B, k, V, dtype=dt, device=device)
    D = torch.empty(B, k, dtype=torch.int32, device=device)
    seq_block = max(1, block_rows // (k + 1))
    for b0 in range(0, B, seq_block):
        nb = min(seq_block, B - b0)
        t = _target_rows(cfg["target"], nb * (k + 1), V, gen, device).view(nb, k + 1, V)
        d = t[:, :k] * scale + torch.randn(nb, k, V, generator=gen, device=device) * noise
        Lt[b0:b0 + nb] = t.to(dt)
        Ld[b0:b0 + nb] = d.to(dt)
        # drafted tokens ~ softmax(Ld / T) of the logits as stored, by Gumbel-max
        u = torch.rand(nb, k, V, generator=gen_d, device=device).clamp_(1e-30, 1.0 - 1e-7)
        g = -torch.log(-torch.log(u))
        D[b0:b0 + nb] = torch.argmax(Ld[b0:b0 + nb].float() / T + g, dim=2).to(torch.int32)
        del t, d, u, g

    mode = cfg["gate"] if gate is None else gate
    if mode == "plain":
        g8 = torch.zeros(B, dtype=torch.uint8)
    elif mode == "gated":
        g8 = torch.ones(B, dtype=torch.uint8)
    elif mode == "half":
        g8 = (torch.arange(B) >= B // 2).to(torch.uint8)
    else:
        raise ValueError(mode)
    tau = torch.full((B,), float(cfg["tau"]), dtype=torch.float32)
    return Workload(name=name, Lt=Lt, Ld=Ld, D=D, T=T, gate=g8.to(device), tau=tau.to(device),
                    philox_seed=seed + 2, B=B, k=k, V=V, dtype=cfg["dtype"])


def to_numpy_logits(x: torch.Tensor) -> np.ndarray:
    """float32 -> numpy float32; bfloat16 -> numpy uint16 bit patterns."""
    x = x.detach().cpu().contiguous()
    if x.dtype == torch.bfloat16:
        return x.view(torch.int16).numpy().view(np.uint16)
    if x.dtype == torch.float32:
        return x.numpy()
    raise TypeError(x.dtype)
