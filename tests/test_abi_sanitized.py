"""The host side of the C ABI under AddressSanitizer and UndefinedBehaviorSanitizer.

Every translation unit of ``csrc/`` is compiled with both sanitizers on its
host code (the device code as PTX only: no kernel runs here) and linked with
``abi_sanitize_driver.c``, which calls every entry point on the paths a host
without a usable GPU reaches: status strings, launch counts, argument
validation, a NULL handle, sizes beyond the limits, the allocation-free entry
point's size checks, and device calls that fail.  Any out-of-bounds access,
leak or undefined operation on those paths, or an unexpected status code,
fails the test.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(ROOT, "speculative_decoding_verification_online_gb300", "csrc")
INCLUDE = os.path.join(ROOT, "include")
SANITIZE = ["-fsanitize=address", "-fsanitize=undefined", "-fno-sanitize-recover=all",
            "-fno-omit-frame-pointer"]


def _cuda_home():
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    return os.path.dirname(os.path.dirname(nvcc)) if os.path.exists(nvcc) else None


def test_host_abi_is_clean_under_address_and_undefined_behaviour_sanitizers(tmp_path):
    cuda = _cuda_home()
    if cuda is None or shutil.which("gcc") is None or shutil.which("g++") is None:
        pytest.skip("nvcc or gcc not found")
    libdir = os.path.join(cuda, "lib64")
    if not os.path.exists(os.path.join(libdir, "libcudart.so")):
        pytest.skip("no shared CUDA runtime under " + libdir)
    drv_o, exe = str(tmp_path / "driver.o"), str(tmp_path / "abi_sanitized")
    xc = [a for f in SANITIZE for a in ("-Xcompiler", f)]
    # every translation unit of the library (in parallel), then the driver
    units = sorted(f for f in os.listdir(CSRC) if f.endswith(".cu"))
    objs = [str(tmp_path / (u[:-3] + ".o")) for u in units]
    procs = [subprocess.Popen([os.path.join(cuda, "bin", "nvcc"), "-gencode", "arch=compute_103a,code=compute_103a",
                               "-O1", "-g", "-std=c++17", *xc, "-I", INCLUDE, "-I", CSRC, "-c",
                               os.path.join(CSRC, u), "-o", o], stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                              text=True) for u, o in zip(units, objs)]
    for u, pr in zip(units, procs):
        out, err = pr.communicate()
        assert pr.returncode == 0, u + "\n" + err
    steps = [
        ["gcc", "-std=c11", "-O1", "-g", *SANITIZE, "-Wall", "-Wextra", "-Werror", "-I", INCLUDE, "-c",
         os.path.join(HERE, "abi_sanitize_driver.c"), "-o", drv_o],
        ["g++", *SANITIZE, drv_o, *objs, "-L", libdir, "-lcudart", "-Wl,-rpath," + libdir, "-o", exe],
    ]
    for cmd in steps:
        r = subprocess.run(cmd, capture_output=True, text=True)
        if r.returncode != 0 and ("lasan" in r.stderr or "lubsan" in r.stderr):
            pytest.skip("no sanitizer runtime on this host")
        assert r.returncode == 0, " ".join(cmd) + "\n" + r.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:halt_on_error=1",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    run = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "runtime error" not in run.stderr, run.stderr
    assert "0 failed checks" in run.stdout, run.stdout
