"""Benchmark of batched speculative-decoding verification on GB300.

One step = one spec_verify_run call (the whole hot path: row statistics,
gate/accept decisions, residual or bonus sampling) over one batch of the
synthetic workload, inputs resident in HBM.  Prints one JSON line.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--temperature T] [--gate plain|gated|half]
                  [--gate-schedule T0,T1,...] [--min-cum F] [--diagnostics]
                  [--target-filter K,P,M] [--draft-filter K,P,M]

--temperature and --gate override the workload's temperature (0 = greedy
decoding) and gate recipe; the logits and drafted tokens stay the same.
--gate-schedule / --min-cum set the gate policy of the gated sequences
(per-step thresholds, the last repeating; the cumulative prefix-product floor).
--target-filter / --draft-filter set the sampler filters (top_k, top_p, min_p)
of the target and draft rows.
--diagnostics times spec_verify_diagnostics (the closed-form acceptance of
every draft position: a stream pass plus a second read of each (p_j, q_j)
pair) instead of the verification call; it has no host-buffer entry point, so
that line carries no e2e figure.

--impl reference times the fp64 CPU oracle on the host cores (the baseline
arm); under torchrun only rank 0 runs it.  Multi-GPU runs shard sequences
across ranks (weak scaling, Philox keys stay global via seq_offset).
"""
from __future__ import annotations

import argparse
import glob
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import workloads  # noqa: E402

METRIC = "verified draft positions/sec and logits GB/s (fraction of GB300 HBM peak)"
DEFAULT_WORKLOAD = "b64_v128256_zipf_gated"
NOMINAL_HBM_GBS = 8000.0
L2_BYTES = 126 * 1024 * 1024
PROFILE = os.path.join(ROOT, "profiles", "stream_kernel_b64_v128256_zipf_gated.md")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=5000)
    ap.add_argument("--warmup", type=int, default=50)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=DEFAULT_WORKLOAD, choices=sorted(workloads.CONFIGS))
    ap.add_argument("--seed", type=int, default=1234)
    ap.add_argument("--temperature", type=float, default=None,
                    help="override the workload's temperature (0 = greedy decoding)")
    ap.add_argument("--gate", choices=["plain", "gated", "half"], default=None,
                    help="override the workload's gate recipe")
    ap.add_argument("--gate-schedule", default=None,
                    help="per-step gate thresholds, comma-separated (the last repeats)")
    ap.add_argument("--min-cum", type=float, default=0.0,
                    help="cumulative floor on the drafted prefix's product of draft probabilities")
    ap.add_argument("--target-filter", default=None, help="top_k,top_p,min_p of the target rows")
    ap.add_argument("--draft-filter", default=None, help="top_k,top_p,min_p of the draft rows")
    ap.add_argument("--diagnostics", action="store_true",
                    help="time the closed-form acceptance diagnostics instead of verification")
    ap.add_argument("--e2e-steps", type=int, default=20)
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--single-replays", type=int, default=60,
                    help="cold single-call replays (L2 flushed before each) for the latency median")
    ap.add_argument("--clock-window", type=float, default=1.0,
                    help="seconds of load (timed region plus untimed steps) seen by the clock sampler")
    return ap.parse_args()


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def make_workload(args, seed, device, B=None):
    """The named workload with the command line's temperature / gate overrides."""
    w = workloads.make(args.workload, seed=seed, device=device, B=B, gate=args.gate)
    if args.temperature is not None:
        w.T = float(args.temperature)
    return w


def overridden(args) -> bool:
    return (args.temperature is not None or args.gate is not None or args.gate_schedule is not None
            or args.min_cum > 0 or args.diagnostics or filters_of(args) is not None)


def filters_of(args):
    """((top_k, top_p, min_p) target, (...) draft), or None when both are off."""
    def parse_one(text):
        if text is None:
            return (0, 1.0, 0.0)
        k, p, m = text.split(",")
        return (int(k), float(p), float(m))
    ft, fd = parse_one(args.target_filter), parse_one(args.draft_filter)
    return None if ft == fd == (0, 1.0, 0.0) else (ft, fd)


def filter_launches(filt, V, dtypes):
    """Launches the sampler filters add in front of a verifying or diagnostics
    call.  When every filtered side holds bf16 logits and none is top_k = 1:
    the histogram selection (1).  Otherwise the statistics pass and the
    selection (2), plus the bound, gathering and list-selection passes when a
    side has 2 <= top_k <= the number of 2048-entry chunks (at most 512
    chunks)."""
    def on(f):
        return f[0] != 0 or f[1] < 1.0 or f[2] > 0.0
    if all(not on(f) or (dt == "bf16" and f[0] != 1) for f, dt in zip(filt, dtypes)):
        return 1
    nchunk = (V + 2047) // 2048
    gathers = any(2 <= f[0] <= nchunk and nchunk <= 512 for f in filt)
    return 2 + (3 if gathers else 0)


def gate_args(args, w, cfg, sv):
    """The gate arguments of a call: the scalars when every sequence shares one
    mode and threshold (what a caller with one configuration passes; the host
    then knows whether dense residuals can occur), else the per-sequence arrays."""
    recipe = args.gate or cfg["gate"]
    if recipe == "gated":
        return dict(gate_mode=sv.SV_GATED_MU, threshold=float(cfg["tau"]))
    if recipe == "plain":
        return dict(gate_mode=sv.SV_PLAIN, threshold=float(cfg["tau"]))
    return dict(gate_mode=sv.SV_GATED_MU, threshold=float(cfg["tau"]), gate_per_seq=w.gate,
                threshold_per_seq=w.tau)


def gate_policy(args):
    sched = None
    if args.gate_schedule is not None:
        sched = [float(x) for x in args.gate_schedule.split(",")]
    return sched, float(args.min_cum)


# the sources the verifying call's stream and finishing kernels are built
# from: their code, launch configuration and arguments (the filter and
# diagnostics kernels live in files of their own)
STREAM_SOURCES = ("csrc/verify_kernel.cuh", "csrc/philox.cuh", "csrc/launch.cuh", "csrc/handle.h",
                  "csrc/spec_verify.cu", "csrc/pair_bf16_bf16.cu")


def kernel_hash() -> str:
    """Hash of the files the stream kernel's profile depends on."""
    h = hashlib.sha256()
    pkg = os.path.join(ROOT, "speculative_decoding_verification_online_gb300")
    for f in sorted(STREAM_SOURCES):
        h.update(open(os.path.join(pkg, f), "rb").read())
    h.update(open(os.path.join(ROOT, "include", "spec_verify.h"), "rb").read())
    return h.hexdigest()[:16]


def profile_traffic(path=PROFILE, current_hash=None):
    """DRAM bytes per launch from the committed ncu summary, if it was taken on
    the current kernel sources (else None).  The summary lists
    `- kernel_hash: ...` and `- traffic_bytes_per_launch: ...` lines."""
    if not os.path.exists(path):
        return None
    vals = {}
    for line in open(path):
        item = line.strip().lstrip("-* ")
        if ":" in item and item.startswith(("kernel_hash", "traffic_bytes_per_launch")):
            key, val = item.split(":", 1)
            vals[key.strip(" `")] = val.strip(" `\n")
    if vals.get("kernel_hash") != (current_hash or kernel_hash()):
        return None
    try:
        return int(vals["traffic_bytes_per_launch"])
    except (KeyError, ValueError):
        return None


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        self.lines = [ln for ln in out.splitlines() if ln.strip()]

    def summary(self):
        rows = []
        for ln in self.lines:
            f = [x.strip() for x in ln.split(",")]
            if len(f) < 9:
                continue
            try:
                rows.append(dict(sm=float(f[1]), smax=float(f[2]), hw=f[5], hwt=f[6], swt=f[7],
                                 pcap=f[8]))
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        reasons = set()
        for r in rows:
            for key, name in (("hw", "hw_slowdown"), ("hwt", "hw_thermal_slowdown"),
                              ("swt", "sw_thermal_slowdown"), ("pcap", "sw_power_cap")):
                if r[key].lower() == "active":
                    reasons.add(name)
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["smax"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows)}


def cpu_oracle_rate(w, seconds: float, nthreads: int, sched=None, cum=0.0, filters=None):
    """Time the fp64 oracle on the workload's sequences for about `seconds`."""
    from oracle import oracle as O
    Lt = workloads.to_numpy_logits(w.Lt)
    Ld = workloads.to_numpy_logits(w.Ld)
    D = w.D.cpu().numpy()
    gate = w.gate.cpu().numpy()
    tau = w.tau.cpu().numpy().astype(np.float64)
    pol = dict(tau_sched=sched, min_cum=cum)
    O.verify(Lt[:1], Ld[:1], D[:1], w.T, gate[:1], tau[:1], seed=w.philox_seed,
             **dict(pol, filters=filters))  # build + warm
    reps, t0 = 0, time.perf_counter()
    while True:
        O.verify(Lt, Ld, D, w.T, gate, tau, seed=w.philox_seed, nthreads=nthreads, filters=filters, **pol)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return reps * w.B * w.k / el, reps, el


def cpu_diag_rate(w, seconds: float, nthreads: int, sched=None, cum=0.0, filters=None):
    """Time the fp64 oracle's diagnostics on the workload's sequences for about `seconds`."""
    from oracle import oracle as O
    Lt = workloads.to_numpy_logits(w.Lt)
    Ld = workloads.to_numpy_logits(w.Ld)
    D = w.D.cpu().numpy()
    gate = w.gate.cpu().numpy()
    tau = w.tau.cpu().numpy().astype(np.float64)
    pol = dict(tau_sched=sched, min_cum=cum)
    reps, t0 = 0, time.perf_counter()
    while True:
        O.diagnostics(Lt, Ld, D, w.T, gate, tau, nthreads=nthreads, filters=filters, **pol)
        reps += 1
        el = time.perf_counter() - t0
        if el >= seconds:
            break
    return reps * w.B * w.k / el, reps, el


def run_reference(args, ws, rank):
    """The baseline arm: the fp64 CPU oracle on host cores."""
    if rank != 0:
        return
    from oracle import oracle as O
    cfg = workloads.CONFIGS[args.workload]
    sample_B = max(1, min(cfg["B"], 8))
    w = make_workload(args, args.seed, "cpu", B=sample_B)
    Lt = workloads.to_numpy_logits(w.Lt)
    Ld = workloads.to_numpy_logits(w.Ld)
    D = w.D.cpu().numpy()
    gate = w.gate.cpu().numpy()
    tau = w.tau.cpu().numpy().astype(np.float64)
    cores = os.cpu_count() or 1
    sched, cum = gate_policy(args)
    pol = dict(tau_sched=sched, min_cum=cum)

    filt = filters_of(args)

    def one():
        if args.diagnostics:
            O.diagnostics(Lt, Ld, D, w.T, gate, tau, nthreads=cores, filters=filt, **pol)
        else:
            O.verify(Lt, Ld, D, w.T, gate, tau, seed=w.philox_seed, nthreads=cores, filters=filt, **pol)
    t0 = time.perf_counter()
    one()
    t_step = time.perf_counter() - t0
    # a deliberately slow program: bound the whole run to a few minutes
    budget = 150.0
    steps = args.steps
    warm = args.warmup
    if (steps + warm) * t_step > budget:
        warm = min(warm, 3)
        steps = max(1, int(budget / t_step) - warm)
    for _ in range(warm):
        one()
    t0 = time.perf_counter()
    for _ in range(steps):
        one()
    el = time.perf_counter() - t0
    value = steps * sample_B * w.k / el
    sample = (f"{sample_B} of {cfg['B']} sequences of {args.workload} per step; "
              f"{steps} of {args.steps} requested steps timed")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "positions/s",
        "n_gpus": ws, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": 1e3 * el / steps, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": args.workload, "B_sample": sample_B, "k": w.k, "V": w.V,
                   "logits_dtype": w.dtype, "T": w.T,
                   "gate": args.gate or workloads.CONFIGS[args.workload]["gate"],
                   "gate_schedule": sched, "min_cum": cum, "filters": filt,
                   "call": "oracle_diagnostics" if args.diagnostics else "oracle_verify"},
        "cpu_baseline": {"value": value, "unit": "positions/s", "cores": cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": value, "unit": "positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    args = parse()
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        dist.init_process_group("gloo" if args.impl == "reference" else "nccl")
    if args.impl == "reference":
        run_reference(args, ws, rank)
        if ws > 1:
            import torch.distributed as dist
            dist.destroy_process_group()
        return

    import speculative_decoding_verification_online_gb300 as sv
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    cfg = workloads.CONFIGS[args.workload]
    B = cfg["B"]
    # inputs larger than L2 for the big configs; rotate copies so each step reads
    # logits that the previous steps have evicted
    per_set = None
    sets = []
    nsets = 1
    for i in range(8):
        w = make_workload(args, args.seed + 1000 * rank + 7 * i, dev)
        sets.append(w)
        per_set = w.logits_bytes()
        nsets = len(sets)
        if nsets * per_set >= 3 * L2_BYTES and nsets >= 2:
            break
    w0 = sets[0]
    k, V = w0.k, w0.V
    ver = sv.SpecVerifier(B, k, V, device=local)
    sched, cum = gate_policy(args)
    if sched is not None or cum > 0:
        ver.set_gate_policy(sched, cum)
    filt = filters_of(args)
    if filt is not None:
        ver.set_filters(*filt)
    outs = [ver.outputs(B) for _ in range(nsets)]
    douts = [{key: torch.empty(B, k, dtype=torch.float32, device=dev)
              for key in ("min_sum", "pq_sum", "argmax_q")} for _ in range(nsets)]
    seq_offset = rank * B
    stream = torch.cuda.current_stream(dev)

    gargs = [gate_args(args, w, cfg, sv) for w in sets]

    def step(i):
        w = sets[i % nsets]
        if args.diagnostics:
            ver.diagnostics(w.Lt, w.Ld, w.D, w.T, out=douts[i % nsets], **gargs[i % nsets])
            return
        ver.run(w.Lt, w.Ld, w.D, w.T, seed=w.philox_seed, seq_offset=seq_offset,
                out=outs[i % nsets], **gargs[i % nsets])

    sampler = ClockSampler(local)
    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)

    # The K timed steps as CUDA graph replays: the same launches (programmatic
    # dependent launches become programmatic edges of the graph), without the
    # Python marshalling of each call in front of the device.  Graphs of at
    # most 500 steps, replayed once each untimed first (upload).
    graphs = []
    first = 0
    while first < args.steps:
        n = min(500, args.steps - first)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(first, first + n):
                step(i)
        graphs.append(g)
        first += n
    for g in graphs:
        g.replay()
    torch.cuda.synchronize(dev)

    sampler.start()
    time.sleep(0.3)  # let the sampler start before the timed region
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t_wall = time.perf_counter()
    ev0.record(stream)
    for g in graphs:
        g.replay()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    t_wall = time.perf_counter() - t_wall
    if ws > 1:
        dist.barrier()
    # the same K steps launched call by call from Python: device time, and the
    # host's enqueue time per call (the loop returns before the device is done
    # as long as the host keeps ahead of it)
    ed0, ed1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ed0.record(stream)
    t_host = time.perf_counter()
    for i in range(args.steps):
        step(i)
    t_host = time.perf_counter() - t_host
    ed1.record(stream)
    torch.cuda.synchronize(dev)
    ms_direct = ed0.elapsed_time(ed1)
    # keep the GPU busy (untimed) until the sampler has seen ~1 s under load
    t_extra = time.perf_counter()
    while t_wall + (time.perf_counter() - t_extra) < args.clock_window:
        for g in graphs:
            g.replay()
        torch.cuda.synchronize(dev)
    sampler.stop()
    ms = ev0.elapsed_time(ev1)

    # one call at a time, cold: a graph of one step per input copy, the L2
    # flushed (a 2 x L2 buffer written) before each replay, the median of the
    # replays' event-timed durations
    single = None
    if not args.diagnostics and args.single_replays > 0:
        one_graphs = []
        for s_ in range(nsets):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g):
                step(s_)
            one_graphs.append(g)
        flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
        durs = []
        for r in range(args.single_replays + 3):
            flush.fill_(float(r))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            one_graphs[r % nsets].replay()
            e1.record(stream)
            torch.cuda.synchronize(dev)
            if r >= 3:
                durs.append(e0.elapsed_time(e1))
        del flush
        single = {"median_us": 1e3 * statistics.median(durs), "min_us": 1e3 * min(durs),
                  "replays": len(durs),
                  "protocol": "CUDA graph of one call, L2 flushed (2 x L2 written) before each "
                              "replay, CUDA events, median"}

    # the dominant kernel alone: the same K steps again, with CUDA events that
    # the library records around each stream-pass launch
    n_mark = args.steps
    marks = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
             for _ in range(n_mark)]
    for a, b in marks:  # torch creates the CUDA events on their first record
        a.record(stream)
        b.record(stream)
    torch.cuda.synchronize(dev)
    for i in range(n_mark):
        ver.mark_next(*marks[i])
        step(i)
    torch.cuda.synchronize(dev)
    stream_ms = sum(a.elapsed_time(b) for a, b in marks) / n_mark
    el = torch.tensor([ms], dtype=torch.float64)
    if ws > 1:
        el_t = el.to(dev)
        dist.all_reduce(el_t, op=dist.ReduceOp.MAX)
        el = el_t.cpu()
    ms_total = float(el[0])
    sec = ms_total / 1e3
    positions = ws * args.steps * B * k
    value = positions / sec
    logits_bytes = per_set  # per step per rank
    step_gbs = logits_bytes / (sec / args.steps) / 1e9
    achieved_gbs = logits_bytes / (stream_ms / 1e3) / 1e9
    peak, peak_kind = measured_peaks()

    # e2e through the host-buffer entry point: pinned inputs, H2D + verify + D2H per step
    e2e = None
    if (rank == 0 or ws > 1) and not args.diagnostics:
        wh = sets[0]
        Lt_h = wh.Lt.cpu().pin_memory()
        Ld_h = wh.Ld.cpu().pin_memory()
        D_h = wh.D.cpu().pin_memory()
        g_h = wh.gate.cpu().pin_memory()
        tau_h = wh.tau.cpu().pin_memory()
        out_h = dict(accepted_len=torch.empty(B, dtype=torch.int32).pin_memory(),
                     tokens=torch.empty(B, k + 1, dtype=torch.int32).pin_memory(),
                     accept_prob=torch.empty(B, k, dtype=torch.float32).pin_memory(),
                     flags=torch.empty(B, k, dtype=torch.int8).pin_memory())

        ga = gate_args(args, wh, cfg, sv)
        per_seq = "gate_per_seq" in ga
        if per_seq:
            ga = dict(ga, gate_per_seq=g_h, threshold_per_seq=tau_h)

        def hstep():
            ver.run_host(Lt_h, Ld_h, D_h, wh.T, seed=wh.philox_seed, out=out_h, **ga)
        for _ in range(3):
            hstep()
        n_e2e = max(1, args.e2e_steps)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            hstep()
        e2e_s = (time.perf_counter() - t0) / n_e2e
        h2d = (Lt_h.numel() * Lt_h.element_size() + Ld_h.numel() * Ld_h.element_size() +
               D_h.numel() * 4 + ((g_h.numel() + tau_h.numel() * 4) if per_seq else 0))
        d2h = sum(t.numel() * t.element_size() for t in out_h.values())
        e2e = {"value": ws * B * k / e2e_s, "unit": "positions/s", "h2d_bytes_per_step": h2d,
               "d2h_bytes_per_step": d2h}

    cpu = None
    if rank == 0 and args.diagnostics:
        cores = os.cpu_count() or 1
        small = make_workload(args, args.seed, "cpu", B=min(B, 16 if V > 100000 else B))
        rate, reps, cel = cpu_diag_rate(small, args.cpu_seconds, cores, sched, cum, filters_of(args))
        cpu = {"value": rate, "unit": "positions/s", "cores": cores, "kind": "oracle",
               "sample": f"oracle_diagnostics on {small.B} sequences of {args.workload} x {reps} "
                         f"repetitions ({cel:.1f} s)"}
    elif rank == 0:
        cores = os.cpu_count() or 1
        small = make_workload(args, args.seed, "cpu", B=min(B, 16 if V > 100000 else B))
        rate, reps, cel = cpu_oracle_rate(small, args.cpu_seconds, cores, sched, cum, filters_of(args))
        # the same oracle on one thread, on a quarter of the time
        rate1, _, _ = cpu_oracle_rate(small, max(args.cpu_seconds / 4, 0.1), 1, sched, cum, filters_of(args))
        cpu = {"value": rate, "unit": "positions/s", "cores": cores, "kind": "oracle",
               "single_thread_value": rate1,
               "sample": f"{small.B} sequences of {args.workload} x {reps} repetitions "
                         f"({cel:.1f} s)"}

    if rank == 0:
        clocks = sampler.summary()
        # the committed ncu summary covers the default configuration only
        traffic = (profile_traffic() if args.workload == DEFAULT_WORKLOAD and not overridden(args)
                   else None)
        line = {
            "metric": METRIC, "value": value, "unit": "positions/s", "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_total / args.steps,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
            "data": "synthetic",
            "config": {"workload": args.workload, "B_per_gpu": B, "k": k, "V": V,
                       "logits_dtype": w0.dtype, "T": w0.T, "gate": args.gate or cfg["gate"],
                       "gate_schedule": sched, "min_cum": cum, "filters": filt,
                       "gate_args": "per-sequence arrays" if "gate_per_seq" in gargs[0] else "scalars",
                       "call": "spec_verify_diagnostics" if args.diagnostics else "spec_verify_run",
                       "threshold": cfg["tau"],
                       "l2": f"inputs larger than L2: {nsets} rotated copies of "
                             f"{per_set / 1e6:.1f} MB logits",
                       "parallelism": f"replicas x{ws} (sequence shards)"},
            "timing": {"steps": "CUDA graph replays of the K calls (graphs of <= 500 calls), "
                                 "CUDA events around them",
                       "ms_per_step_direct": ms_direct / args.steps,
                       "host_enqueue_us_per_call": 1e6 * t_host / args.steps,
                       "single_call": single},
            "logits_gbs": step_gbs,
            "logits_frac_of_8tbs": step_gbs / NOMINAL_HBM_GBS,
            "logits_frac_of_measured": step_gbs / peak,
            "roofline": {"bound": "hbm", "achieved": achieved_gbs, "peak": peak, "unit": "GB/s",
                         "frac": achieved_gbs / peak, "peak_kind": peak_kind,
                         "traffic": traffic, "kernel": "stream_kernel",
                         "kernel_ms": stream_ms,
                         "algorithmic_bytes_per_launch": logits_bytes,
                         "timing": "CUDA events around each stream-pass launch, second pass of "
                                   "the K steps"},
            "cpu_baseline": cpu,
            "e2e": e2e,
            # the diagnostics launch 4 kernels per call (2 at temperature 0);
            # sampler filters add the launches of filter_launches in front
            "gpu_launches": args.steps * (((2 if w0.T == 0 else 4) if args.diagnostics
                                           else sv.spec_verify_launches_per_run())
                                          + (filter_launches(filt, w0.V, (w0.dtype, w0.dtype))
                                             if filt is not None and w0.T > 0 else 0)),
            "clocks": clocks,
        }
        print(json.dumps(line), flush=True)
    ver.close()
    if ws > 1:
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
