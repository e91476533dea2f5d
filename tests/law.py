"""Exact output law of a verification rule at tiny sizes, by enumeration.

For one sequence (target rows p_0..p_k, draft rows q_0..q_{k-1}) every draft
outcome D in [V]^k is enumerated with weight prod_j q_j(D_j), every stop
position s with the cells of the uniforms that lead there, and the oracle is
asked for its decision at one point inside each cell.  The law of the oracle's
outputs is the cell-volume-weighted sum of those decisions.

Cells: the accept uniform u0_j is split at the oracle's own alpha_j (accept
below, reject above); the residual uniform u1 is split at the cumulative sums
of every candidate emission distribution of every row (p_s, (p_s - mu_s)+,
(p_s - q_s)+, the renormalised-mu residual) plus a uniform grid.  A rule whose
picks are inverse CDFs of any of those distributions is therefore constant on
each cell, and its law comes out exactly (up to float rounding).

The distributions used for the cells come from scipy's softmax, not from the
oracle.  The law itself is never compared with this module's own arithmetic:
tests compare it with what the pages fix (the emitted marginal is p, the pass
rate is sum_x min(p, mu), the worked example's printed numbers).
"""
from __future__ import annotations

import itertools

import numpy as np
from scipy.special import softmax

from oracle import oracle as O


def distributions(Lt: np.ndarray, Ld: np.ndarray, T: float, filters=None):
    """Row distributions: scipy's softmax, or -- with sampler filters -- the
    oracle's filtered rows (pinned on their own by the filter examples)."""
    if filters is None:
        P = softmax(Lt.astype(np.float64) / T, axis=-1)
        Q = softmax(Ld.astype(np.float64) / T, axis=-1)
        return P, Q
    P = np.stack([O.filtered_row(r, T, *filters[0])[0] for r in Lt])
    Q = np.stack([O.filtered_row(r, T, *filters[1])[0] for r in Ld])
    return P, Q


def _step_tau(tau, tau_sched, s):
    if tau_sched is None:
        return tau
    return tau_sched[min(s, len(tau_sched) - 1)]


def _u1_edges(P, Q, gated, tau, grid, tau_sched=None, min_cum=0.0):
    """Cell edges of u1: the cumulative sums of every distribution a stop row
    could sample.  With a cumulative floor the admitted set of step s depends
    on the drafted prefix, so every prefix's product contributes its own."""
    k, V = Q.shape
    edges = set(np.linspace(0.0, 1.0, grid + 1).tolist())
    for s in range(k + 1):
        cands = [P[s]]
        if s < k:
            ts = _step_tau(tau, tau_sched, s)
            prods = {1.0}
            if min_cum > 0.0:
                prods = {float(np.prod(Q[np.arange(s), list(pre)])) if s else 1.0
                         for pre in itertools.product(range(V), repeat=s)}
            for c in sorted(prods):
                keep = Q[s] >= ts
                mus = [Q[s] * keep]
                if min_cum > 0.0:
                    mus.append(Q[s] * (keep & (c * Q[s] >= min_cum)))
                for mu in (mus if gated else [Q[s]]):
                    cands.append(np.maximum(P[s] - mu, 0.0))
                    if gated and mu.sum() > 0:
                        cands.append(np.maximum(P[s] - mu / mu.sum(), 0.0))
            cands.append(np.maximum(P[s] - Q[s], 0.0))
        for w in cands:
            Z = w.sum()
            if Z > 0:
                edges.update((np.cumsum(w) / Z).tolist())
    e = np.array(sorted(x for x in edges if 0.0 <= x <= 1.0))
    keep = np.concatenate([[True], np.diff(e) > 1e-13])
    e = e[keep]
    e[0], e[-1] = 0.0, 1.0
    return e


def exact_law(Lt, Ld, T, gated, tau, rule=O.RULE_MU, grid=32, tau_sched=None, min_cum=0.0, filters=None):
    """Law of (accepted_len, tokens) for one sequence, as a dict -> probability.

    Lt [k+1, V], Ld [k, V] float32 (one sequence); tau_sched / min_cum: the
    gate policy passed through to the oracle.
    """
    pol = dict(tau_sched=tau_sched, min_cum=min_cum, filters=filters)
    Lt = np.asarray(Lt, dtype=np.float32)
    Ld = np.asarray(Ld, dtype=np.float32)
    k1, V = Lt.shape
    k = k1 - 1
    P, Q = distributions(Lt, Ld, T, filters)
    drafts = np.array(list(itertools.product(range(V), repeat=k)), dtype=np.int32)
    nD = drafts.shape[0]
    wD = np.prod(Q[np.arange(k)[None, :], drafts], axis=1)

    # the oracle's acceptance probability of every position for every draft outcome
    base = O.verify(np.broadcast_to(Lt, (nD, k1, V)), np.broadcast_to(Ld, (nD, k, V)), drafts, T,
                    gated, tau, u0=np.full((nD, k), 0.5), u1=np.full(nD, 0.5), rule=rule, **pol)
    alpha = base["alpha"]

    edges = _u1_edges(P, Q, gated, tau, grid, tau_sched, min_cum)
    lo, hi = edges[:-1], edges[1:]
    mids = 0.5 * (lo + hi)
    vols = hi - lo

    probes_d, probes_u0, probes_u1, probes_w = [], [], [], []
    for d in range(nD):
        if wD[d] == 0.0:
            continue
        for s in range(k + 1):
            w = wD[d] * np.prod(alpha[d, :s])
            if s < k:
                w *= 1.0 - alpha[d, s]
            if w == 0.0:
                continue
            u0 = np.full(k, 0.5)
            u0[:s] = 0.5 * alpha[d, :s]
            if s < k:
                u0[s] = 0.5 * (alpha[d, s] + 1.0)
            probes_d.append(np.full(len(mids), d))
            probes_u0.append(np.broadcast_to(u0, (len(mids), k)))
            probes_u1.append(mids)
            probes_w.append(w * vols)
    pd = np.concatenate(probes_d)
    pu0 = np.concatenate(probes_u0)
    pu1 = np.concatenate(probes_u1)
    pw = np.concatenate(probes_w)
    n = pd.shape[0]
    out = O.verify(np.broadcast_to(Lt, (n, k1, V)), np.broadcast_to(Ld, (n, k, V)), drafts[pd], T,
                   gated, tau, u0=pu0, u1=pu1, rule=rule, nthreads=4, **pol)
    law: dict = {}
    for acc, toks, w in zip(out["accepted_len"], out["tokens"], pw):
        key = (int(acc), tuple(int(t) for t in toks))
        law[key] = law.get(key, 0.0) + float(w)
    return law


def position_marginals(law, k, V):
    """reach[j] = P(position j reached), emit[j, x] = P(reached and token x at j),
    passed[j] = P(position j reached and accepted)."""
    reach = np.zeros(k + 1)
    emit = np.zeros((k + 1, V))
    passed = np.zeros(k)
    for (acc, toks), pr in law.items():
        if acc < 0:
            continue
        for j in range(acc + 1):
            reach[j] += pr
            emit[j, toks[j]] += pr
        for j in range(acc):
            passed[j] += pr
    return reach, emit, passed
