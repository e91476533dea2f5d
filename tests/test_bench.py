"""Host logic of bench.py (no GPU): the ncu summary parser that feeds
roofline.traffic, and the reference arm's JSON line."""
import json
import os
import runpy
import subprocess
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _bench():
    return runpy.run_path(os.path.join(ROOT, "bench.py"))


def test_profile_traffic_reads_the_summary_only_for_the_current_sources(tmp_path):
    b = _bench()
    p = tmp_path / "summary.md"
    p.write_text("# x\n\n- kernel_hash: `abc123`\n- traffic_bytes_per_launch: `184297984`\n")
    assert b["profile_traffic"](str(p), current_hash="abc123") == 184297984
    assert b["profile_traffic"](str(p), current_hash="other") is None
    assert b["profile_traffic"](str(tmp_path / "missing.md"), current_hash="abc123") is None
    # the committed summary names a 16-hex-digit hash and an integer byte count
    text = open(os.path.join(ROOT, "profiles", "stream_kernel_b64_v128256_zipf_gated.md")).read()
    assert "- kernel_hash: `" in text and "- traffic_bytes_per_launch: `" in text


def test_reference_arm_prints_one_json_line():
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0", "--workload", "tiny_v8_f32"],
                         capture_output=True, text=True, check=True, cwd=ROOT, timeout=300)
    lines = [ln for ln in out.stdout.splitlines() if ln.strip()]
    assert len(lines) == 1
    d = json.loads(lines[0])
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["cpu_baseline"]["kind"] == "oracle"
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["value"] > 0


def test_cpu_oracle_rate_on_one_thread_and_a_pool():
    # the CPU-baseline leg: the oracle timed on the workload's sequences, with
    # the pool of host cores and on a single thread
    import workloads
    b = _bench()
    w = workloads.make("b16_v32000_bf16", seed=1, device="cpu", B=2)
    for threads in (1, 2):
        rate, reps, el = b["cpu_oracle_rate"](w, 0.05, threads)
        assert rate > 0 and reps >= 1 and el >= 0.05
        assert abs(rate - reps * w.B * w.k / el) < 1e-9 * rate


def test_filter_launch_counts_follow_the_selection_route():
    # the launches a filtered call adds in front of its own (the bench line's
    # gpu_launches counts them): the histogram selection (1) when every
    # filtered side is bf16 and none is top_k = 1, else the statistics pass
    # and select_kernel (2), plus bound, gathering and list selection (3) when
    # a side gathers its top-k set (2 <= top_k <= chunks <= 512); within the
    # header's bound of 7 launches per filtered verifying call
    fl = _bench()["filter_launches"]
    OFF = (0, 1.0, 0.0)
    V = 128256  # 63 chunks
    assert fl(((50, 0.9, 0.0), (40, 0.95, 0.0)), V, ("bf16", "bf16")) == 1
    assert fl(((0, 0.9, 0.0), OFF), V, ("bf16", "f32")) == 1  # the f32 side is unfiltered
    assert fl(((0, 1.0, 0.05), OFF), V, ("bf16", "bf16")) == 1
    assert fl(((1, 1.0, 0.0), OFF), V, ("bf16", "bf16")) == 2  # top_k = 1: select_kernel's kept index
    assert fl(((0, 0.9, 0.0), OFF), V, ("f32", "f32")) == 2
    assert fl(((50, 0.9, 0.0), OFF), V, ("f32", "f32")) == 5  # gathered top-k
    assert fl(((64, 0.9, 0.0), OFF), V, ("f32", "f32")) == 2  # k above the 63 chunks: not gathered
    assert fl(((50, 0.9, 0.0), (1, 1.0, 0.0)), V, ("bf16", "bf16")) == 5
    for filt in (((50, 0.9, 0.0), (40, 0.95, 0.0)), ((1, 1.0, 0.0), (3, 1.0, 0.0))):
        for dts in (("bf16", "bf16"), ("f32", "bf16"), ("f32", "f32")):
            assert fl(filt, V, dts) + 2 <= 7
