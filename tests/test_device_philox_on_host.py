"""The library's device-side Philox4x32-10 (csrc/philox.cuh), built as host
C++ by ``device_philox_host_driver.cpp``, against the published known answers
and, on 10^6 random (seed, sequence, position, draw) requests, against the
oracle's separately written generator: both must give the same uniform bit for
bit.  No GPU is needed; the GPU parity tests check the same generator in use."""
from __future__ import annotations

import os
import shutil
import subprocess

import numpy as np
import pytest

from oracle import oracle as O

HERE = os.path.dirname(os.path.abspath(__file__))
CSRC = os.path.join(os.path.dirname(HERE), "speculative_decoding_verification_online_gb300", "csrc")


@pytest.fixture(scope="module")
def driver(tmp_path_factory):
    if shutil.which("g++") is None:
        pytest.skip("g++ not found")
    exe = str(tmp_path_factory.mktemp("philox") / "device_philox_host_driver")
    subprocess.run(["g++", "-std=c++17", "-O2", "-Wall", "-Wextra", "-Werror", "-Wno-unknown-pragmas",
                    "-I", CSRC, os.path.join(HERE, "device_philox_host_driver.cpp"), "-o", exe],
                   check=True)
    return exe


def test_device_philox_meets_the_known_answers(driver):
    rows = []
    with open(os.path.join(HERE, "golden", "philox4x32_10_kat.txt")) as f:
        for line in f:
            if line.strip() and not line.startswith("#"):
                rows.append(line.split())
    request = "".join(" ".join(r[:6]) + "\n" for r in rows)
    out = subprocess.run([driver, "kat"], input=request, capture_output=True, text=True, check=True)
    got = out.stdout.split()
    assert got == [r[6] for r in rows]


def test_device_philox_uniforms_equal_the_oracle_on_a_million_requests(driver, tmp_path):
    n = 1_000_000
    rng = np.random.default_rng(2024)
    rec = np.zeros(n, dtype=[("seed", "<u8"), ("seq", "<u8"), ("pos", "<u4"), ("draw", "<u4")])
    rec["seed"] = rng.integers(0, 2 ** 63, n, dtype=np.uint64) * 2 + rng.integers(0, 2, n, dtype=np.uint64)
    rec["seq"] = rng.integers(0, 2 ** 40, n, dtype=np.uint64)
    rec["pos"] = rng.integers(0, 64, n, dtype=np.uint32)
    rec["draw"] = rng.integers(0, 2, n, dtype=np.uint32)
    src, dst = tmp_path / "req.bin", tmp_path / "u.bin"
    rec.tofile(src)
    subprocess.run([driver, "grid", str(src), str(dst)], check=True)
    dev = np.fromfile(dst, dtype=np.float32)
    assert dev.shape == (n,)
    ref = np.array([O.uniform(int(s), int(q), int(p), int(d))
                    for s, q, p, d in zip(rec["seed"], rec["seq"], rec["pos"], rec["draw"])])
    assert np.array_equal(dev.astype(np.float64), ref)
    # the uniforms are 24-bit grid points in [0, 1)
    assert dev.min() >= 0.0 and dev.max() < 1.0
    assert np.all(dev * 2.0 ** 24 == np.floor(dev * 2.0 ** 24))
