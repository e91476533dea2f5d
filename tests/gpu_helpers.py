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
    arithmetic -- those are counted and reported apart;
  * every mismatch inside a band must be a result that is still correct to
    within the band: a flipped decision only where that decision's draw lies
    within 1e-6 of its boundary, and an emitted token only where it is a
    valid pick of the oracle's own stop-row distribution, u1 within 1e-6 of
    its interval (see _judge_boundary_mismatch);
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


def _judge_boundary_mismatch(w, i, b, g_len, g_tok, g_flags, ref, gate_near, u0, u1,
                             tau_sched, min_cum, filters):
    """Why a GPU result inside a boundary band differs from the oracle's, or
    None when nothing explains it.  Sequence b (row i of the compared arrays):
      * a flipped decision (a different stop position, or REJECT against NULL
        at the same one) is explained only by that position's draw lying within
        1e-6 of its boundary: |u0 - p/mu| where p/mu < 1, or a gate decision
        within 1e-6 of its threshold;
      * the token the GPU emits at its own stop position j must be a valid
        pick of the oracle's stop-row distribution at j (the residual, or p for
        the bonus row): weight > 0 and u1 within 1e-6 of the token's interval
        [C(v-1)/Z, C(v)/Z) in fp64 -- unless a token of that row sits within
        1e-6 of the gate (then the retained measure itself is a boundary case)
        or a sampler filter decision of the sequence does (the kept set is)."""
    gl, ol = int(g_len[i]), int(ref["accepted_len"][i])
    if gl < 0 or ol < 0:
        return None  # validity never depends on a draw
    D = w.D[b].cpu().numpy()
    if not np.array_equal(g_tok[i, :gl], D[:gl]):
        return None
    seed = w.philox_seed
    kind = "pick"
    # every decision the GPU took on its way to its stop position j: accepted
    # before j, not accepted at j (when j < k).  The oracle decides position
    # i by alpha_i = min(1, p/mu) (0 for NULL or p = 0): accept iff alpha_i > 0
    # and u0 <= alpha_i.  A disagreement is a boundary case only if u0 lies
    # within 1e-6 of alpha_i < 1, or the gate decision lies within 1e-6.
    for j in range(min(gl + 1, w.k)):
        a = float(ref["alpha"][i, j])
        uj = float(u0[b, j]) if u0 is not None else O.uniform(seed, b, j, 0)
        if (a > 0.0 and uj <= a) != (j < gl):
            if not (gate_near[i, j] or (0.0 < a < 1.0 and abs(uj - a) < BOUNDARY)):
                return None
            kind = "decision"
    # REJECT against NULL at the same stop position: the gate decision flipped
    if g_flags is not None and gl == ol and gl < w.k and g_flags[i, gl] != ref["flags"][i, gl]:
        if not gate_near[i, gl]:
            return None
        kind = "decision"
    filt_near = ref.get("margin_filter", np.full(len(g_len), np.inf))[i] < BOUNDARY
    gate_b = int(w.gate[b].item())
    tau_b = float(w.tau[b].item())
    Lt = workloads.to_numpy_logits(w.Lt[b:b + 1])[0]
    Ld = workloads.to_numpy_logits(w.Ld[b:b + 1])[0]
    v = int(g_tok[i, gl])
    if not 0 <= v < w.V:
        return None
    wt, lo, hi, gm = O.pick_interval(Lt, Ld, D, w.T, gate_b, tau_b, gl, v, tau_sched=tau_sched,
                                     min_cum=min_cum, filters=filters)
    uj = float(u1[b]) if u1 is not None else O.uniform(seed, b, gl, 1)
    if wt > 0.0 and (w.T == 0.0 or lo - BOUNDARY <= uj < hi + BOUNDARY):
        return kind
    if gm < BOUNDARY:
        return "gate_row"
    if filt_near:
        return "filter"
    return None


def compare(w: workloads.Workload, got: dict, ref: dict, idx=None, what="", tau_sched=None,
            min_cum=0.0, filters=None, u0=None, u1=None):
    """Assert parity; returns a dict of counts.  tau_sched / min_cum: the gate
    policy both sides ran with; filters: their sampler filters; u0 [B, k] /
    u1 [B]: explicit uniforms both sides were given (else the Philox draws,
    keyed on the sequence's index in w).

    Every sequence outside the boundary bands must match bit for bit.  Every
    mismatch inside them must be explained (see _judge_boundary_mismatch).
    Counts: compared, boundary (sequences with a draw within 1e-6 of a
    boundary), boundary_decision / boundary_pick / boundary_filter (by the
    kind of the closest draw), boundary_mismatch and its kinds, draws (accept
    draws of the tested positions plus one pick per valid sequence)."""
    sel = slice(None) if idx is None else np.asarray(idx)
    gidx = np.arange(w.B)[sel]
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
    near = gate_near_boundary(w, ref, idx, tau_sched, min_cum) if gate.any() else \
        np.zeros_like(g_alpha, dtype=bool)
    keep = ~near
    np.testing.assert_allclose(g_alpha[keep], ref["alpha"][keep], rtol=ALPHA_RTOL, atol=ALPHA_ATOL,
                               err_msg=what)
    kinds = {"decision": 0, "pick": 0, "gate_row": 0, "filter": 0}
    unexplained = []
    for i in np.nonzero(~ok & mism)[0]:
        kind = _judge_boundary_mismatch(w, i, int(gidx[i]), g_len, g_tok, g_flags, ref, near, u0, u1,
                                        tau_sched, min_cum, filters)
        if kind is None:
            unexplained.append(int(gidx[i]))
        else:
            kinds[kind] += 1
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
                 mismatch_decision=kinds["decision"], mismatch_pick=kinds["pick"],
                 mismatch_gate_row=kinds["gate_row"], mismatch_filter=kinds["filter"],
                 draws=int((tested + valid).sum()))
    print(f"[parity] {what}: {stats}")
    assert not unexplained, (f"{what}: boundary-band mismatches the oracle does not explain, "
                             f"sequences {unexplained[:8]}", stats)
    assert stats["boundary_decision"] <= 1e-5 * stats["draws"] + 2, (what, stats)
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
