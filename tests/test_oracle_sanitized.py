"""The CPU oracle under AddressSanitizer and UndefinedBehaviorSanitizer.

``oracle_sanitize_driver.c`` calls every oracle entry point -- Philox, the
softmax row, the inverse CDF, the sampler filters, verification with and
without a gate policy or filters, every control rule, the diagnostics -- on
float32 and bfloat16 rows of 1 to 300 tokens, temperatures 1, 0.7 and 0, the
largest k, explicit uniforms at 0 and 1 - 2^-24, and invalid rows and tokens.
It is compiled together with the oracle's own source with both sanitizers
(leak checking included, every report fatal), so an out-of-bounds access, a
leak, a signed overflow or another undefined operation anywhere in the oracle
fails this test.  The arithmetic itself is pinned by the other oracle tests.
"""
from __future__ import annotations

import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ORACLE = os.path.join(os.path.dirname(HERE), "oracle")


def test_oracle_is_clean_under_address_and_undefined_behaviour_sanitizers(tmp_path):
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not found")
    exe = str(tmp_path / "oracle_sanitized")
    build = subprocess.run(
        [gcc, "-std=c11", "-O1", "-g", "-fno-omit-frame-pointer", "-ffp-contract=off",
         "-fsanitize=address,undefined", "-fno-sanitize-recover=all", "-Wall", "-Wextra", "-Werror",
         "-I", ORACLE, os.path.join(HERE, "oracle_sanitize_driver.c"),
         os.path.join(ORACLE, "spec_verify_oracle.c"), "-o", exe, "-lm", "-lpthread"],
        capture_output=True, text=True)
    if build.returncode != 0 and ("lasan" in build.stderr or "lubsan" in build.stderr):
        pytest.skip("no sanitizer runtime on this host: " + build.stderr.strip().splitlines()[-1])
    assert build.returncode == 0, build.stderr
    env = dict(os.environ, ASAN_OPTIONS="detect_leaks=1:halt_on_error=1",
               UBSAN_OPTIONS="print_stacktrace=1:halt_on_error=1")
    run = subprocess.run([exe], capture_output=True, text=True, env=env, timeout=300)
    assert run.returncode == 0, run.stdout + run.stderr
    assert "runtime error" not in run.stderr, run.stderr
    assert "0 failed checks" in run.stdout, run.stdout
