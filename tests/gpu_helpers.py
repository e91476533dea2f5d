"""Shared helpers of the GPU parity tests: run the CUDA path and the oracle on
the same seeded inputs and compare them the way the tolerances demand.

Comparison rules:
  * accepted lengths, emitted tokens and flags are compared bit for bit on
    every sequence whose oracle margin (the distance of every used uniform, or
    gated q, to its decision boundary) is at least 1e-6; a mismatch there fails;
  * sequences below that margin are boundary draws: they are counted, and so
    are the mismatches among them.  Draws of the accept test and the gate must
    number under 1e-5 of those draws (plus a small allowance for small
    samples); the residual / bonus pick over V tokens has V interval edges,
    so at large V many picks sit within 1e-6 of an edge whatever the
    arithmetic -- those are reported, and mismatches among them bounded;
  * acceptance probabilities agree within 1e-5 relative (fp32 against fp64),
    except on positions whose gated q(D) lies within 1e-6 of the threshold
    (there the NULL decision itself is a boundary case).
"""
from __future__ import annotations

import numpy as np
import torch

import workloads
from oracle import oracle as O

BOUNDARY = 1e-6
ALPHA_RTOL = 1e-5
ALPHA_ATOL = 1e-30


def oracle_for(w: workloads.Workload, idx=None, nthreads=8, u0=None, u1=None, tau_sched=None,
               min_cum=0.0, filters=None):
    """Oracle outputs for workload w (all sequences, or the listed ones), with
    an optional gate policy (per-step schedule, cumulative floor) and sampler
    filters ((top_k, top_p, min_p) of the target rows, of the draft rows)."""
    gate = w.gate.cpu().numpy()
    tau = w.tau.cpu().numpy().astype(np.float64)
    pol = dict(tau_sched=tau_sched, min_cum=min_cum, filters=filters)
    if idx is None:
        return O.verify(workloads.to_numpy_logits(w.Lt), workloads.to_numpy_logits(w.Ld),
                        w.D.cpu().numpy(), w.T, gate, tau, seed=w.philox_seed,
                        u0=u0, u1=u1, nthreads=nthreads, **pol)
    parts = []
    for b in idx:
        parts.append(O.verify(workloads.to_numpy_logits(w.Lt[b:b + 1]),
                              workloads.to_numpy_logits(w.Ld[b:b + 1]), w.D[b:b + 1].cpu().numpy(),
                              w.T, gate[b:b + 1], tau[b:b + 1], seed=w.philox_seed,
                              seq_offset=int(b), nthreads=1, **pol))
    return {key: np.concatenate([p[key] for p in parts]) for key in parts[0]}


def gated_q_of_drafts(w: workloads.Workload, ref, idx=None):
    """q_j(D_j) in fp64 from the oracle's row statistics (for excluding gate-boundary alphas);
    at temperature 0, 1 where D_j is the first largest draft logit and 0 elsewhere."""
    sel = slice(None) if idx is None else torch.as_tensor(idx)
    Ld = w.Ld[sel].float().cpu().double()
    D = w.D[sel].cpu().long()
    k = w.k
    if w.T == 0:
        # greedy decoding: q is one-hot at the first largest draft logit
        return (D.numpy() == np.argmax(Ld.numpy(), axis=2)).astype(np.float64)
    x = torch.gather(Ld, 2, D.unsqueeze(-1)).squeeze(-1) / w.T
    lse = torch.as_tensor(ref["row_stats"][:, k + 1:, 1])
    return torch.exp(x - lse).numpy()


def gate_near_boundary(w: workloads.Workload, ref, idx=None, tau_sched=None, min_cum=0.0):
    """[B, k] mask of gated positions whose gate decision lies within 1e-6 of a
    boundary: |q(D) - tau_j| (tau_j > 0) or, with a cumulative floor,
    |prod_{i<j} q_i(D_i) * q_j(D_j) - min_cum| (q in fp64 from the oracle)."""
    sel = slice(None) if idx is None else np.asarray(idx)
    gate = w.gate.cpu().numpy()[sel].astype(bool)
    qd = gated_q_of_drafts(w, ref, idx)
    k = w.k
    if tau_sched is None:
        tau = np.broadcast_to(w.tau.cpu().numpy()[sel].astype(np.float64)[:, None], qd.shape)
    else:
        tau = np.broadcast_to(np.array([tau_sched[min(j, len(tau_sched) - 1)] for j in range(k)]),
                              qd.shape)
    near = (tau > 0) & (np.abs(qd - tau) < BOUNDARY)
    if min_cum > 0:
        incl = np.cumprod(qd, axis=1)
        near |= np.abs(incl - min_cum) < BOUNDARY
    return gate[:, None] & near


def compare(w: workloads.Workload, got: dict, ref: dict, idx=None, what="", tau_sched=None,
            min_cum=0.0):
    """Assert parity; returns a dict of counts (compared, boundary, boundary_decision,
    boundary_pick, boundary_mismatch, draws).  tau_sched / min_cum: the gate
    policy both sides ran with."""
    sel = slice(None) if idx is None else np.asarray(idx)
    g_len = got["accepted_len"].cpu().numpy()[sel]
    g_tok = got["tokens"].cpu().numpy()[sel]
    g_alpha = got["accept_prob"].cpu().numpy()[sel].astype(np.float64)
    g_flags = got["flags"].cpu().numpy()[sel] if "flags" in got else None
    margin = ref["margin"]
    ok = margin >= BOUNDARY
    mism = (g_len != ref["accepted_len"]) | np.any(g_tok != ref["tokens"], axis=1)
    if g_flags is not None:
        mism |= np.any(g_flags != ref["flags"], axis=1)
    bad = np.nonzero(ok & mism)[0]
    assert bad.size == 0, (
        f"{what}: {bad.size} non-boundary mismatches, first b={bad[:5]}: "
        f"gpu len {g_len[bad[:3]]} tok {g_tok[bad[:3]]} | oracle len {ref['accepted_len'][bad[:3]]} "
        f"tok {ref['tokens'][bad[:3]]} margin {margin[bad[:3]]}")
    gate = w.gate.cpu().numpy()[sel].astype(bool)
    keep = np.ones_like(g_alpha, dtype=bool)
    if gate.any():
        keep &= ~gate_near_boundary(w, ref, idx, tau_sched, min_cum)
    np.testing.assert_allclose(g_alpha[keep], ref["alpha"][keep], rtol=ALPHA_RTOL, atol=ALPHA_ATOL,
                               err_msg=what)
    valid = ref["accepted_len"] >= 0
    tested = np.where(valid, np.minimum(ref["accepted_len"] + 1, w.k), 0)
    pick_bnd = ref["margin_pick"] < BOUNDARY
    # a top-p or min-p boundary within 1e-6 of some token of a row: on
    # near-flat rows single-token mass steps are ~1e-5, so such rows are
    # common; they are counted apart like pick boundaries
    filt_bnd = ref.get("margin_filter", np.full(len(margin), np.inf)) < BOUNDARY
    dec_bnd = ~ok & ~pick_bnd & ~filt_bnd
    stats = dict(compared=int(ok.sum()), boundary=int((~ok).sum()),
                 boundary_decision=int(dec_bnd.sum()), boundary_pick=int(pick_bnd.sum()),
                 boundary_filter=int(filt_bnd.sum()),
                 boundary_mismatch=int((~ok & mism).sum()),
                 draws=int((tested + valid).sum()))
    print(f"[parity] {what}: {stats}")
    assert stats["boundary_decision"] <= 1e-5 * stats["draws"] + 2, (what, stats)
    assert stats["boundary_mismatch"] <= 0.1 * max(stats["boundary"], 1) + 1, (what, stats)
    return stats


def peaked_workload(B, k, V, dtype, seed, gate=1, tau=0.5, T=1.0, device="cuda"):
    """Rows with one boosted token whose boost varies from row to row, so the
    drafted tokens' q spans (0, 1) and gates pass and fail at every step."""
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    dt = torch.bfloat16 if dtype == "bf16" else torch.float32
    t = torch.randn(B, k + 1, V, generator=g, device=device)
    peak = torch.randint(0, V, (B, k + 1), generator=g, device=device)
    boost = 6.0 + 9.0 * torch.rand(B, k + 1, generator=g, device=device)
    t.scatter_add_(2, peak.unsqueeze(-1), boost.unsqueeze(-1))
    d = t[:, :k] + torch.randn(B, k, V, generator=g, device=device) * 0.5
    Lt, Ld = t.to(dt), d.to(dt)
    u = torch.rand(B, k, V, generator=g, device=device).clamp_(1e-30, 1 - 1e-7)
    # drafted tokens ~ softmax(Ld / T) (Gumbel-max; at T = 0 the draw uses T = 1)
    Tg = T if T > 0 else 1.0
    D = torch.argmax(Ld.float() / Tg - torch.log(-torch.log(u)), dim=2).to(torch.int32)
    gate_t = torch.as_tensor(np.broadcast_to(np.asarray(gate, dtype=np.uint8), (B,)).copy(),
                             device=device)
    tau_t = torch.full((B,), float(tau), dtype=torch.float32, device=device)
    return workloads.Workload(name="peaked", Lt=Lt, Ld=Ld, D=D, T=T, gate=gate_t, tau=tau_t,
                              philox_seed=seed + 2, B=B, k=k, V=V, dtype=dtype)
