"""ctypes binding of the CUDA verifier library (``libspec_verify.so``).

Argument marshalling only: every step of the verification runs in the CUDA
kernels behind the C ABI of ``include/spec_verify.h``.  Functions keep the C
names; ``SpecVerifier`` bundles a handle with torch-tensor marshalling
(``data_ptr()`` and the current CUDA stream).  There is no CPU fallback: if
the shared library is missing, loading raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIBRARY = os.path.join(HERE, "libspec_verify.so")

SV_OK, SV_EINVAL, SV_ENOMEM, SV_ECUDA, SV_EUNSUPPORTED = 0, 1, 2, 3, 4
SV_F32, SV_BF16 = 0, 1
SV_PLAIN, SV_GATED_MU = 0, 1
SV_FLAG_UNREACHED, SV_FLAG_ACCEPT, SV_FLAG_REJECT, SV_FLAG_NULL, SV_FLAG_INVALID = 0, 1, 2, 3, 4
(SV_CNT_TESTED, SV_CNT_ACCEPTED, SV_CNT_NULL, SV_CNT_REJECTED, SV_CNT_BONUS, SV_CNT_BOUNDARY, SV_CNT_INVALID,
 SV_CNT_DEGENERATE) = range(8)
COUNTER_NAMES = ("tested", "accepted", "null", "rejected", "bonus", "boundary", "invalid",
                 "degenerate")
SV_MAX_K = 32
SV_MAX_V = 1 << 22

_lib = None


class SpecVerifyError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {spec_verify_status_string(status)} (status {status})")


def load() -> ctypes.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(LIBRARY):
        raise RuntimeError(f"CUDA library {LIBRARY} is not built; run __graft_entry__.build()")
    L = ctypes.CDLL(LIBRARY)
    P, I, F, U64 = ctypes.c_void_p, ctypes.c_int, ctypes.c_float, ctypes.c_uint64
    L.spec_verify_init.argtypes = [ctypes.POINTER(P), I, I, I, I]
    L.spec_verify_init.restype = I
    run_common = [P, P, I, P, I, P, I, F, I, F, P, P, U64]
    L.spec_verify_run.argtypes = run_common + [P, P, P, P, P, P]
    L.spec_verify_run.restype = I
    L.spec_verify_run_ex.argtypes = run_common + [U64, P, P, P, P, P, P, P, P, P]
    L.spec_verify_run_ex.restype = I
    L.spec_verify_run_host.argtypes = run_common + [P, P, P, P, P, P]
    L.spec_verify_run_host.restype = I
    L.spec_verify_free.argtypes = [P]
    L.spec_verify_free.restype = I
    L.spec_verify_status_string.argtypes = [I]
    L.spec_verify_status_string.restype = ctypes.c_char_p
    L.spec_verify_launches_per_run.argtypes = []
    L.spec_verify_launches_per_run.restype = I
    L.spec_verify_mark_next.argtypes = [P, P, P]
    L.spec_verify_mark_next.restype = I
    L.spec_verify_run_noalloc.argtypes = [P, I, P, I, P, I, I, I, F, I, F, P, P, U64, P, P, P, P, P, P]
    L.spec_verify_run_noalloc.restype = I
    L.spec_verify_set_gate_policy.argtypes = [P, P, I, F]
    L.spec_verify_set_gate_policy.restype = I
    L.spec_verify_diagnostics.argtypes = [P, P, I, P, I, P, I, F, I, F, P, P, P, P, P, P]
    L.spec_verify_diagnostics.restype = I
    L.spec_verify_set_filters.argtypes = [P, I, F, F, I, F, F]
    L.spec_verify_set_filters.restype = I
    L.spec_verify_launches_per_filtered_run.argtypes = []
    L.spec_verify_launches_per_filtered_run.restype = I
    _lib = L
    return L


# ------------------------------------------------------------- C names

def spec_verify_status_string(status: int) -> str:
    return load().spec_verify_status_string(int(status)).decode()


def spec_verify_init(max_B: int, k: int, V: int, device: int = 0) -> int:
    h = ctypes.c_void_p()
    rc = load().spec_verify_init(ctypes.byref(h), int(max_B), int(k), int(V), int(device))
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_init")
    return h.value


def spec_verify_run(h, Lt, tdt, Ld, ddt, D, B, temperature, gate_mode, threshold, gate_per_seq,
                    threshold_per_seq, seed, accepted_len, tokens, accept_prob, flags, counters,
                    stream) -> int:
    """Raw call with integer pointers; returns the status code."""
    return load().spec_verify_run(h, Lt, tdt, Ld, ddt, D, B, temperature, gate_mode, threshold,
                                  gate_per_seq, threshold_per_seq, seed, accepted_len, tokens,
                                  accept_prob, flags, counters, stream)


def spec_verify_run_ex(h, Lt, tdt, Ld, ddt, D, B, temperature, gate_mode, threshold, gate_per_seq,
                       threshold_per_seq, seed, seq_offset, u_accept, u_residual, accepted_len,
                       tokens, accept_prob, flags, counters, row_stats, stream) -> int:
    return load().spec_verify_run_ex(h, Lt, tdt, Ld, ddt, D, B, temperature, gate_mode, threshold,
                                     gate_per_seq, threshold_per_seq, seed, seq_offset, u_accept,
                                     u_residual, accepted_len, tokens, accept_prob, flags, counters,
                                     row_stats, stream)


def spec_verify_run_host(h, Lt, tdt, Ld, ddt, D, B, temperature, gate_mode, threshold,
                         gate_per_seq, threshold_per_seq, seed, accepted_len, tokens, accept_prob,
                         flags, counters, stream) -> int:
    return load().spec_verify_run_host(h, Lt, tdt, Ld, ddt, D, B, temperature, gate_mode,
                                       threshold, gate_per_seq, threshold_per_seq, seed,
                                       accepted_len, tokens, accept_prob, flags, counters, stream)


def spec_verify_free(h) -> int:
    return load().spec_verify_free(h)


def spec_verify_set_gate_policy(h, schedule, n_schedule, min_cum) -> int:
    """Raw call: schedule is a ctypes float array (or None), min_cum a float."""
    return load().spec_verify_set_gate_policy(h, schedule, n_schedule, min_cum)


def spec_verify_diagnostics(h, Lt, tdt, Ld, ddt, D, B, temperature, gate_mode, threshold,
                            gate_per_seq, threshold_per_seq, min_sum, pq_sum, argmax_q, stream) -> int:
    """Raw call of the acceptance diagnostics; returns the status."""
    return load().spec_verify_diagnostics(h, Lt, tdt, Ld, ddt, D, B, temperature, gate_mode,
                                          threshold, gate_per_seq, threshold_per_seq, min_sum,
                                          pq_sum, argmax_q, stream)


def spec_verify_set_filters(h, top_k_t, top_p_t, min_p_t, top_k_d, top_p_d, min_p_d) -> int:
    """Raw call: sampler filters of the target and draft rows."""
    return load().spec_verify_set_filters(h, top_k_t, top_p_t, min_p_t, top_k_d, top_p_d, min_p_d)


def spec_verify_launches_per_filtered_run() -> int:
    return load().spec_verify_launches_per_filtered_run()


def spec_verify_launches_per_run() -> int:
    return load().spec_verify_launches_per_run()


def spec_verify_mark_next(h, ev_before, ev_after) -> int:
    """Record two CUDA events (raw cudaEvent_t handles) around the next call's stream pass."""
    return load().spec_verify_mark_next(h, ev_before, ev_after)


def spec_verify_run_noalloc(Lt, tdt, Ld, ddt, D, B, k, V, temperature, gate_mode, threshold,
                            gate_per_seq, threshold_per_seq, seed, accepted_len, tokens, accept_prob,
                            flags, counters, stream) -> int:
    """Raw call of the allocation-free entry point (current device); returns the status."""
    return load().spec_verify_run_noalloc(Lt, tdt, Ld, ddt, D, B, k, V, temperature, gate_mode,
                                          threshold, gate_per_seq, threshold_per_seq, seed,
                                          accepted_len, tokens, accept_prob, flags, counters,
                                          stream)


# ------------------------------------------------------ torch marshalling

def _dt(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return SV_BF16
    if t.dtype == torch.float32:
        return SV_F32
    raise TypeError(f"logits must be bfloat16 or float32, got {t.dtype}")


def _ptr(t):
    return None if t is None else t.data_ptr()


def _check(t: torch.Tensor, name: str, shape, dtype=None, device=None):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name}: shape {tuple(t.shape)} != {tuple(shape)}")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: dtype {t.dtype} != {dtype}")
    if device is not None and t.device != device:
        raise ValueError(f"{name}: on {t.device}, expected {device}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


class SpecVerifier:
    """A verifier handle for batches up to ``max_B`` with ``k`` drafts over ``V`` tokens."""

    def __init__(self, max_B: int, k: int, V: int, device: int = 0):
        self.max_B, self.k, self.V = int(max_B), int(k), int(V)
        self.device = torch.device("cuda", device)
        self.handle = spec_verify_init(max_B, k, V, device)

    def close(self):
        if self.handle:
            spec_verify_free(self.handle)
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass

    def mark_next(self, ev_before: torch.cuda.Event, ev_after: torch.cuda.Event):
        """Time the next call's stream pass with two torch CUDA events (enable_timing=True,
        already recorded once so that torch has created them)."""
        if not ev_before.cuda_event or not ev_after.cuda_event:
            raise ValueError("record both events once before passing them (torch creates them lazily)")
        rc = spec_verify_mark_next(self.handle, ev_before.cuda_event, ev_after.cuda_event)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_mark_next")

    def set_filters(self, target=(0, 1.0, 0.0), draft=(0, 1.0, 0.0)):
        """Sampler filters (top_k, top_p, min_p) of the target rows and of the
        draft rows for later calls; (0, 1.0, 0.0) is off."""
        rc = spec_verify_set_filters(self.handle, int(target[0]), float(target[1]), float(target[2]),
                                     int(draft[0]), float(draft[1]), float(draft[2]))
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_set_filters")

    def set_gate_policy(self, schedule=None, min_cum: float = 0.0):
        """Per-step thresholds (a sequence of floats in [0, 1], the last one
        repeating; None for none) and the cumulative floor (0 = off) of the
        gated sequences of later calls.  Raises on a malformed policy, which
        then leaves the previous one in place."""
        arr, n = None, 0
        if schedule is not None:
            vals = [float(x) for x in schedule]
            n = len(vals)
            arr = (ctypes.c_float * max(n, 1))(*vals)
        rc = spec_verify_set_gate_policy(self.handle, arr, n, float(min_cum))
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_set_gate_policy")

    def outputs(self, B: int):
        dev = self.device
        return dict(
            accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
            tokens=torch.empty(B, self.k + 1, dtype=torch.int32, device=dev),
            accept_prob=torch.empty(B, self.k, dtype=torch.float32, device=dev),
            flags=torch.empty(B, self.k, dtype=torch.int8, device=dev),
        )

    def run(self, Lt, Ld, D, temperature, gate_mode=SV_PLAIN, threshold=0.5, gate_per_seq=None,
            threshold_per_seq=None, seed=0, seq_offset=0, u_accept=None, u_residual=None,
            counters=None, row_stats=False, out=None, stream=None):
        """Verify device tensors; returns a dict of device output tensors."""
        B = Lt.shape[0]
        k, V, dev = self.k, self.V, self.device
        _check(Lt, "target_logits", (B, k + 1, V), device=dev)
        _check(Ld, "draft_logits", (B, k, V), device=dev)
        _check(D, "draft_tokens", (B, k), torch.int32, dev)
        if gate_per_seq is not None:
            _check(gate_per_seq, "gate_mode_per_seq", (B,), torch.uint8, dev)
        if threshold_per_seq is not None:
            _check(threshold_per_seq, "threshold_per_seq", (B,), torch.float32, dev)
        if u_accept is not None:
            _check(u_accept, "u_accept", (B, k), torch.float32, dev)
        if u_residual is not None:
            _check(u_residual, "u_residual", (B,), torch.float32, dev)
        if counters is not None:
            _check(counters, "counters", (8,), torch.int64, dev)
        o = self.outputs(B) if out is None else out
        rs = torch.empty(B, 2 * k + 1, 2, dtype=torch.float32, device=dev) if row_stats else None
        st = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream
        rc = spec_verify_run_ex(self.handle, Lt.data_ptr(), _dt(Lt), Ld.data_ptr(), _dt(Ld),
                                D.data_ptr(), B, float(temperature), int(gate_mode),
                                float(threshold), _ptr(gate_per_seq), _ptr(threshold_per_seq),
                                int(seed), int(seq_offset), _ptr(u_accept), _ptr(u_residual),
                                o["accepted_len"].data_ptr(), o["tokens"].data_ptr(),
                                o["accept_prob"].data_ptr(), _ptr(o.get("flags")),
                                _ptr(counters), _ptr(rs), st)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_run_ex")
        if rs is not None:
            o["row_stats"] = rs
        return o

    def diagnostics(self, Lt, Ld, D, temperature, gate_mode=SV_PLAIN, threshold=0.5,
                    gate_per_seq=None, threshold_per_seq=None, out=None, stream=None):
        """Closed-form acceptance of every draft position: a dict of [B, k]
        float device tensors min_sum (sum min(p, mu)), pq_sum (sum p q) and
        argmax_q (q at the first largest p); NaN where the rows are invalid."""
        B = Lt.shape[0]
        k, V, dev = self.k, self.V, self.device
        _check(Lt, "target_logits", (B, k + 1, V), device=dev)
        _check(Ld, "draft_logits", (B, k, V), device=dev)
        _check(D, "draft_tokens", (B, k), torch.int32, dev)
        if gate_per_seq is not None:
            _check(gate_per_seq, "gate_mode_per_seq", (B,), torch.uint8, dev)
        if threshold_per_seq is not None:
            _check(threshold_per_seq, "threshold_per_seq", (B,), torch.float32, dev)
        if out is None:
            out = {key: torch.empty(B, k, dtype=torch.float32, device=dev)
                   for key in ("min_sum", "pq_sum", "argmax_q")}
        st = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream
        rc = spec_verify_diagnostics(self.handle, Lt.data_ptr(), _dt(Lt), Ld.data_ptr(), _dt(Ld),
                                     D.data_ptr(), B, float(temperature), int(gate_mode),
                                     float(threshold), _ptr(gate_per_seq), _ptr(threshold_per_seq),
                                     _ptr(out.get("min_sum")), _ptr(out.get("pq_sum")),
                                     _ptr(out.get("argmax_q")), st)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_diagnostics")
        return out

    def run_host(self, Lt, Ld, D, temperature, gate_mode=SV_PLAIN, threshold=0.5,
                 gate_per_seq=None, threshold_per_seq=None, seed=0, out=None, counters=None,
                 stream=None):
        """Verify host (ideally pinned) tensors through the host-buffer entry point."""
        B = Lt.shape[0]
        k, V, cpu = self.k, self.V, torch.device("cpu")
        _check(Lt, "target_logits", (B, k + 1, V), device=cpu)
        _check(Ld, "draft_logits", (B, k, V), device=cpu)
        _check(D, "draft_tokens", (B, k), torch.int32, cpu)
        if out is None:
            out = dict(accepted_len=torch.empty(B, dtype=torch.int32),
                       tokens=torch.empty(B, k + 1, dtype=torch.int32),
                       accept_prob=torch.empty(B, k, dtype=torch.float32),
                       flags=torch.empty(B, k, dtype=torch.int8))
        st = torch.cuda.current_stream(self.device).cuda_stream if stream is None else stream
        rc = spec_verify_run_host(self.handle, Lt.data_ptr(), _dt(Lt), Ld.data_ptr(), _dt(Ld),
                                  D.data_ptr(), B, float(temperature), int(gate_mode),
                                  float(threshold), _ptr(gate_per_seq), _ptr(threshold_per_seq),
                                  int(seed), out["accepted_len"].data_ptr(),
                                  out["tokens"].data_ptr(), out["accept_prob"].data_ptr(),
                                  _ptr(out.get("flags")), _ptr(counters), st)
        if rc != SV_OK:
            raise SpecVerifyError(rc, "spec_verify_run_host")
        return out


def run_noalloc(Lt, Ld, D, temperature, gate_mode=SV_PLAIN, threshold=0.5, gate_per_seq=None,
                threshold_per_seq=None, seed=0, out=None, counters=None, stream=None):
    """Verify device tensors through the allocation-free entry point on their device.

    The outputs are the caller's tensors (``out``, or new ones made here by
    torch); the library itself allocates nothing.  Calls on one device must
    not overlap."""
    B, k1, V = Lt.shape
    k = k1 - 1
    dev = Lt.device
    _check(Lt, "target_logits", (B, k + 1, V), device=dev)
    _check(Ld, "draft_logits", (B, k, V), device=dev)
    _check(D, "draft_tokens", (B, k), torch.int32, dev)
    if out is None:
        out = dict(accepted_len=torch.empty(B, dtype=torch.int32, device=dev),
                   tokens=torch.empty(B, k + 1, dtype=torch.int32, device=dev),
                   accept_prob=torch.empty(B, k, dtype=torch.float32, device=dev),
                   flags=torch.empty(B, k, dtype=torch.int8, device=dev))
    with torch.cuda.device(dev):
        st = torch.cuda.current_stream(dev).cuda_stream if stream is None else stream
        rc = spec_verify_run_noalloc(Lt.data_ptr(), _dt(Lt), Ld.data_ptr(), _dt(Ld), D.data_ptr(), B,
                                     k, V, float(temperature), int(gate_mode), float(threshold),
                                     _ptr(gate_per_seq), _ptr(threshold_per_seq), int(seed),
                                     out["accepted_len"].data_ptr(), out["tokens"].data_ptr(),
                                     out["accept_prob"].data_ptr(), _ptr(out.get("flags")),
                                     _ptr(counters), st)
    if rc != SV_OK:
        raise SpecVerifyError(rc, "spec_verify_run_noalloc")
    return out
