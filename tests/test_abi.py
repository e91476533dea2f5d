"""The C-ABI library builds, loads without a GPU and exports every symbol the
header declares; host-side helpers behave.  No compute call is made here."""
import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "spec_verify.h")


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(spec_verify_\w+)\s*\(", text)))


@pytest.fixture(scope="module")
def library():
    from speculative_decoding_verification_online_gb300 import build as B
    return B.build()


def test_header_declares_the_boundary():
    names = _declared_functions()
    for must in ("spec_verify_init", "spec_verify_run", "spec_verify_free"):
        assert must in names


def test_library_exports_every_declared_symbol(library):
    lib = ctypes.CDLL(library)
    for name in _declared_functions():
        assert hasattr(lib, name), name
    out = subprocess.run(["nm", "-D", "--defined-only", library], capture_output=True, text=True,
                         check=True).stdout
    exported = set(re.findall(r"\bT\s+(spec_verify_\w+)", out))
    assert set(_declared_functions()) <= exported


def test_status_strings_and_launch_count(library):
    import speculative_decoding_verification_online_gb300 as sv
    assert sv.spec_verify_status_string(0) == "ok"
    assert sv.spec_verify_status_string(1) == "invalid argument"
    assert "unknown" in sv.spec_verify_status_string(99)
    assert sv.spec_verify_launches_per_run() == 2


def test_init_rejects_bad_sizes_before_touching_the_device(library):
    import speculative_decoding_verification_online_gb300 as sv
    lib = sv.load()
    h = ctypes.c_void_p()
    assert lib.spec_verify_init(ctypes.byref(h), 0, 4, 100, 0) == sv.spec_verify.SV_EINVAL
    assert lib.spec_verify_init(ctypes.byref(h), 4, 0, 100, 0) == sv.spec_verify.SV_EINVAL
    assert lib.spec_verify_init(ctypes.byref(h), 4, 33, 100, 0) == sv.spec_verify.SV_EUNSUPPORTED
    assert lib.spec_verify_init(ctypes.byref(h), 4, 4, (1 << 22) + 1, 0) == \
        sv.spec_verify.SV_EUNSUPPORTED
    assert h.value is None
    assert lib.spec_verify_init(None, 4, 4, 100, 0) == sv.spec_verify.SV_EINVAL


def test_run_rejects_a_null_handle(library):
    import speculative_decoding_verification_online_gb300 as sv
    lib = sv.load()
    rc = lib.spec_verify_run(None, None, 0, None, 0, None, 1, 1.0, 0, 0.5, None, None, 0, None,
                             None, None, None, None, None)
    assert rc == sv.spec_verify.SV_EINVAL
    assert lib.spec_verify_free(None) == 0


def test_product_path_has_no_cpu_fallback(monkeypatch, tmp_path):
    import speculative_decoding_verification_online_gb300.spec_verify as m
    monkeypatch.setattr(m, "_lib", None)
    monkeypatch.setattr(m, "LIBRARY", str(tmp_path / "missing.so"))
    with pytest.raises(RuntimeError, match="not built"):
        m.load()


def test_product_package_does_not_reach_the_oracle():
    pkg = os.path.join(ROOT, "speculative_decoding_verification_online_gb300")
    for dirpath, _, files in os.walk(pkg):
        for f in files:
            if f.endswith((".py", ".cu", ".cuh", ".h")):
                text = open(os.path.join(dirpath, f)).read()
                assert not re.search(r"\b(from|import)\s+oracle|liboracle", text), f
