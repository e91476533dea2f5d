"""Python binding of the plain CPU oracle (``spec_verify_oracle.c``).

TEST INFRASTRUCTURE, NOT PART OF THE PRODUCT PATH.  Only the test suite, the
smoke check and the CPU-baseline leg of the benchmark import this module.  It
shares no code with the CUDA library and never imports it.

The arithmetic lives in C (fp64); this file only builds the shared object with
gcc, marshals numpy arrays and names the rules.  Logits are numpy ``float32``
arrays, or ``uint16`` arrays holding bf16 bit patterns.
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
SOURCE = os.path.join(HERE, "spec_verify_oracle.c")
LIBRARY = os.path.join(HERE, "liboracle.so")

F32, BF16 = 0, 1
RULE_MU = 0
RULE_ORIGINAL_GATE = 1
RULE_SAMPLER_MATCH = 2
RULE_ARGMAX = 3
RULE_RESAMPLE_P = 4
RULE_RENORM_MU = 5
RULE_RESIDUAL_Q = 6
RULE_MU_STEP_ONLY = 7

FLAG_UNREACHED, FLAG_ACCEPT, FLAG_REJECT, FLAG_NULL, FLAG_INVALID = 0, 1, 2, 3, 4

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (no fast-math, no FMA contraction, so x86
    and aarch64 hosts evaluate the same expressions)."""
    with _lock:
        fresh = os.path.exists(LIBRARY) and os.path.getmtime(LIBRARY) >= max(
            os.path.getmtime(SOURCE), os.path.getmtime(os.path.join(HERE, "spec_verify_oracle.h")))
        if force or not fresh:
            tmp = LIBRARY + f".tmp{os.getpid()}"
            subprocess.run(["gcc", "-O2", "-std=c11", "-Wall", "-Wextra", "-ffp-contract=off",
                            "-fno-fast-math", "-fPIC", "-shared", SOURCE, "-o", tmp, "-lm",
                            "-lpthread"], check=True)
            os.replace(tmp, LIBRARY)
    return LIBRARY


# A test that checks whether the pins catch a planted mistake points this
# variable at an oracle library built from a mutated copy of the source;
# nothing else sets it.
LIBRARY_OVERRIDE_ENV = "SPEC_VERIFY_ORACLE_LIBRARY"


def lib() -> ctypes.CDLL:
    global _lib
    if _lib is None:
        override = os.environ.get(LIBRARY_OVERRIDE_ENV)
        if not override:
            build()
        L = ctypes.CDLL(override or LIBRARY)
        P = ctypes.c_void_p
        L.oracle_philox4x32_10.argtypes = [P, P, P]
        L.oracle_philox4x32_10.restype = None
        L.oracle_uniform.argtypes = [ctypes.c_uint64, ctypes.c_uint64, ctypes.c_uint32, ctypes.c_uint32]
        L.oracle_uniform.restype = ctypes.c_double
        L.oracle_softmax_row.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_double, P, P, P]
        L.oracle_softmax_row.restype = ctypes.c_int
        L.oracle_inverse_cdf.argtypes = [P, ctypes.c_int64, ctypes.c_double, P]
        L.oracle_inverse_cdf.restype = ctypes.c_int64
        L.oracle_verify.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int, ctypes.c_int,
                                    ctypes.c_int64, ctypes.c_double, P, P, ctypes.c_uint64,
                                    ctypes.c_uint64, P, P, ctypes.c_int, P, P, P, P, P, P, P, P,
                                    ctypes.c_int]
        L.oracle_verify.restype = ctypes.c_int
        L.oracle_verify_policy.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int,
                                           ctypes.c_int, ctypes.c_int64, ctypes.c_double, P, P, P,
                                           ctypes.c_int, ctypes.c_double, ctypes.c_uint64,
                                           ctypes.c_uint64, P, P, ctypes.c_int, P, P, P, P, P, P, P,
                                           P, ctypes.c_int]
        L.oracle_verify_policy.restype = ctypes.c_int
        L.oracle_diagnostics.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int,
                                         ctypes.c_int, ctypes.c_int64, ctypes.c_double, P, P, P,
                                         ctypes.c_int, ctypes.c_double, P, P, P, P, P, P, P,
                                         ctypes.c_int]
        L.oracle_diagnostics.restype = ctypes.c_int
        L.oracle_filtered_row.argtypes = [P, ctypes.c_int, ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                          ctypes.c_double, ctypes.c_double, P, P, P]
        L.oracle_filtered_row.restype = ctypes.c_int
        L.oracle_verify_filtered.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int,
                                             ctypes.c_int, ctypes.c_int64, ctypes.c_double, P, P, P,
                                             ctypes.c_int, ctypes.c_double, P, P, P, ctypes.c_uint64,
                                             ctypes.c_uint64, P, P, ctypes.c_int, P, P, P, P, P, P,
                                             P, P, P, ctypes.c_int]
        L.oracle_verify_filtered.restype = ctypes.c_int
        L.oracle_pick_interval.argtypes = [P, ctypes.c_int, P, ctypes.c_int, P, ctypes.c_int,
                                           ctypes.c_int64, ctypes.c_double, ctypes.c_int,
                                           ctypes.c_double, P, ctypes.c_int, ctypes.c_double, P, P, P,
                                           ctypes.c_int, ctypes.c_int64, P, P, P, P]
        L.oracle_pick_interval.restype = ctypes.c_int
        _lib = L
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _dtype_code(a: np.ndarray) -> int:
    if a.dtype == np.float32:
        return F32
    if a.dtype == np.uint16:
        return BF16
    raise TypeError(f"logits must be float32 or uint16 (bf16 bits), got {a.dtype}")


def philox4x32_10(ctr, key) -> np.ndarray:
    c = np.ascontiguousarray(ctr, dtype=np.uint32)
    k = np.ascontiguousarray(key, dtype=np.uint32)
    out = np.zeros(4, dtype=np.uint32)
    lib().oracle_philox4x32_10(_ptr(c), _ptr(k), _ptr(out))
    return out


def uniform(seed: int, seq: int, pos: int, draw: int) -> float:
    return lib().oracle_uniform(seed, seq, pos, draw)


def softmax_row(logits: np.ndarray, T: float):
    """Returns (p, row_max, row_lse, valid)."""
    x = np.ascontiguousarray(logits)
    p = np.zeros(x.shape[-1], dtype=np.float64)
    mx = np.zeros(1, dtype=np.float64)
    lse = np.zeros(1, dtype=np.float64)
    bad = lib().oracle_softmax_row(_ptr(x), _dtype_code(x), x.shape[-1], float(T), _ptr(p),
                                   _ptr(mx), _ptr(lse))
    return p, float(mx[0]), float(lse[0]), bad == 0


def inverse_cdf(r: np.ndarray, u: float):
    """Returns (index, margin)."""
    w = np.ascontiguousarray(r, dtype=np.float64)
    m = np.zeros(1, dtype=np.float64)
    v = lib().oracle_inverse_cdf(_ptr(w), w.shape[0], float(u), _ptr(m))
    return int(v), float(m[0])


def filtered_row(logits: np.ndarray, T: float, top_k: int = 0, top_p: float = 1.0,
                 min_p: float = 0.0):
    """The filtered distribution of one row (temperature softmax, then top-k,
    top-p, min-p): returns (p, margin)."""
    p, _, _, ok = softmax_row(logits, T)
    if not ok:
        raise ValueError("invalid row")
    x = np.ascontiguousarray(logits)
    m = np.zeros(1, dtype=np.float64)
    rc = lib().oracle_filtered_row(_ptr(x), _dtype_code(x), x.shape[-1], float(T), int(top_k),
                                   float(top_p), float(min_p), _ptr(p), _ptr(m), None)
    if rc != 0:
        raise MemoryError("oracle_filtered_row")
    return p, float(m[0])


def verify(Lt: np.ndarray, Ld: np.ndarray, D: np.ndarray, T: float, gate, tau, seed: int = 0,
           seq_offset: int = 0, u0=None, u1=None, rule: int = RULE_MU, nthreads: int = 1,
           tau_sched=None, min_cum: float = 0.0, filters=None):
    """Run the oracle on a batch.

    Lt [B, k+1, V], Ld [B, k, V] (float32, or uint16 bf16 bits), D [B, k] int32.
    ``gate`` and ``tau`` are per-sequence arrays (or scalars broadcast to B).
    ``u0`` [B, k] / ``u1`` [B] give explicit uniforms instead of Philox draws.
    ``tau_sched`` (a sequence of per-step thresholds, the last repeating) and
    ``min_cum`` (the cumulative floor, 0 = off) are the gate policy of gated
    sequences (``oracle_verify_policy``).  ``filters`` = ((top_k, top_p,
    min_p) of the target rows, (top_k, top_p, min_p) of the draft rows) turns
    on the sampler filters (``oracle_verify_filtered``).
    Returns a dict of numpy arrays: accepted_len, tokens, alpha, flags,
    row_stats [B, 2k+1, 2] (max, lse of L/T), margin (all used draws),
    margin_pick (the residual / bonus pick alone), margin_filter (the sampler
    filters' decisions alone), degenerate.
    """
    Lt = np.ascontiguousarray(Lt)
    Ld = np.ascontiguousarray(Ld)
    B, k1, V = Lt.shape
    k = k1 - 1
    if Ld.shape != (B, k, V):
        raise ValueError(f"draft logits shape {Ld.shape} != {(B, k, V)}")
    D = np.ascontiguousarray(D, dtype=np.int32).reshape(B, k)
    gate = np.ascontiguousarray(np.broadcast_to(np.asarray(gate, dtype=np.uint8), (B,)))
    tau = np.ascontiguousarray(np.broadcast_to(np.asarray(tau, dtype=np.float64), (B,)))
    if u0 is not None:
        u0 = np.ascontiguousarray(u0, dtype=np.float64).reshape(B, k)
    if u1 is not None:
        u1 = np.ascontiguousarray(u1, dtype=np.float64).reshape(B)
    out = dict(
        accepted_len=np.zeros(B, dtype=np.int32),
        tokens=np.zeros((B, k + 1), dtype=np.int32),
        alpha=np.zeros((B, k), dtype=np.float64),
        flags=np.zeros((B, k), dtype=np.int8),
        row_stats=np.zeros((B, 2 * k + 1, 2), dtype=np.float64),
        margin=np.zeros(B, dtype=np.float64),
        margin_pick=np.zeros(B, dtype=np.float64),
        margin_filter=np.full(B, np.inf, dtype=np.float64),
        degenerate=np.zeros(B, dtype=np.int32),
    )
    sched = None if tau_sched is None else np.ascontiguousarray(tau_sched, dtype=np.float64).ravel()
    n_sched = 0 if sched is None else int(sched.shape[0])
    fk, fp, fm = _filter_arrays(filters)
    rc = lib().oracle_verify_filtered(_ptr(Lt), _dtype_code(Lt), _ptr(Ld), _dtype_code(Ld), _ptr(D),
                                      B, k, V, float(T), _ptr(gate), _ptr(tau), _ptr(sched), n_sched,
                                      float(min_cum), _ptr(fk), _ptr(fp), _ptr(fm), int(seed),
                                      int(seq_offset), _ptr(u0), _ptr(u1), int(rule),
                                      _ptr(out["accepted_len"]), _ptr(out["tokens"]),
                                      _ptr(out["alpha"]), _ptr(out["flags"]), _ptr(out["row_stats"]),
                                      _ptr(out["margin"]), _ptr(out["margin_pick"]),
                                      _ptr(out["margin_filter"]), _ptr(out["degenerate"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_verify rejected its arguments")
    return out


def pick_interval(Lt: np.ndarray, Ld: np.ndarray, D: np.ndarray, T: float, gated: int, tau: float,
                  j: int, v: int, tau_sched=None, min_cum: float = 0.0, filters=None):
    """Where token v lies in the distribution the stop row of ONE sequence
    samples from when its chain stops at position j (``oracle_pick_interval``).

    Lt [k+1, V], Ld [k, V] (float32, or uint16 bf16 bits), D [k].  Returns
    (weight, lo, hi, gate_margin): r(v) / Z and the interval [C(v-1) / Z,
    C(v) / Z) of the stop row's weights r, and the closest q_j(x) of a gated
    stop row to a gate boundary (inf otherwise)."""
    Lt = np.ascontiguousarray(Lt)
    Ld = np.ascontiguousarray(Ld)
    k1, V = Lt.shape
    k = k1 - 1
    if Ld.shape != (k, V):
        raise ValueError(f"draft logits shape {Ld.shape} != {(k, V)}")
    D = np.ascontiguousarray(D, dtype=np.int32).reshape(k)
    sched = None if tau_sched is None else np.ascontiguousarray(tau_sched, dtype=np.float64).ravel()
    n_sched = 0 if sched is None else int(sched.shape[0])
    fk, fp, fm = _filter_arrays(filters)
    out = np.zeros(4, dtype=np.float64)
    P = ctypes.c_void_p
    ptrs = [P(out.ctypes.data + 8 * i) for i in range(4)]
    rc = lib().oracle_pick_interval(_ptr(Lt), _dtype_code(Lt), _ptr(Ld), _dtype_code(Ld), _ptr(D), k, V,
                                    float(T), int(gated), float(tau), _ptr(sched), n_sched,
                                    float(min_cum), _ptr(fk), _ptr(fp), _ptr(fm), int(j), int(v),
                                    *ptrs)
    if rc != 0:
        raise ValueError("oracle_pick_interval rejected its arguments (or the row is invalid)")
    return float(out[0]), float(out[1]), float(out[2]), float(out[3])


def _filter_arrays(filters):
    if filters is None:
        return None, None, None
    return (np.array([int(filters[0][0]), int(filters[1][0])], dtype=np.int32),
            np.array([float(filters[0][1]), float(filters[1][1])], dtype=np.float64),
            np.array([float(filters[0][2]), float(filters[1][2])], dtype=np.float64))


def diagnostics(Lt: np.ndarray, Ld: np.ndarray, D: np.ndarray, T: float, gate, tau, tau_sched=None,
                min_cum: float = 0.0, nthreads: int = 1, filters=None):
    """Closed-form acceptance of every draft position (``oracle_diagnostics``).

    Returns a dict of numpy arrays: min_sum [B, k] (sum min(p, mu)), pq_sum
    [B, k] (sum p q), argmax_q [B, k] (q at the first largest p), margin [B]
    (gated sequences: the closest q(x) to a gate boundary).
    """
    Lt = np.ascontiguousarray(Lt)
    Ld = np.ascontiguousarray(Ld)
    B, k1, V = Lt.shape
    k = k1 - 1
    if Ld.shape != (B, k, V):
        raise ValueError(f"draft logits shape {Ld.shape} != {(B, k, V)}")
    D = np.ascontiguousarray(D, dtype=np.int32).reshape(B, k)
    gate = np.ascontiguousarray(np.broadcast_to(np.asarray(gate, dtype=np.uint8), (B,)))
    tau = np.ascontiguousarray(np.broadcast_to(np.asarray(tau, dtype=np.float64), (B,)))
    sched = None if tau_sched is None else np.ascontiguousarray(tau_sched, dtype=np.float64).ravel()
    n_sched = 0 if sched is None else int(sched.shape[0])
    out = dict(min_sum=np.zeros((B, k)), pq_sum=np.zeros((B, k)), argmax_q=np.zeros((B, k)),
               margin=np.zeros(B))
    fk, fp, fm = _filter_arrays(filters)
    rc = lib().oracle_diagnostics(_ptr(Lt), _dtype_code(Lt), _ptr(Ld), _dtype_code(Ld), _ptr(D), B, k,
                                  V, float(T), _ptr(gate), _ptr(tau), _ptr(sched), n_sched,
                                  float(min_cum), _ptr(fk), _ptr(fp), _ptr(fm),
                                  _ptr(out["min_sum"]), _ptr(out["pq_sum"]),
                                  _ptr(out["argmax_q"]), _ptr(out["margin"]), int(nthreads))
    if rc != 0:
        raise ValueError("oracle_diagnostics rejected its arguments")
    return out
