"""Build step for the CUDA library: one nvcc invocation for sm_103a.

``python -m speculative_decoding_verification_online_gb300.build`` (or
``build()``) compiles the translation units of ``csrc/`` (one nvcc process
each, in parallel: the C ABI, and the kernels of each pair of logits types)
and links them into ``libspec_verify.so`` next to this file.  The build is in-tree and skipped when the library is newer
than every source.
"""
from __future__ import annotations

import glob
import os
import subprocess
import sys

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)
CSRC = os.path.join(HERE, "csrc")
INCLUDE = os.path.join(ROOT, "include")
LIBRARY = os.path.join(HERE, "libspec_verify.so")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources():
    return sorted(glob.glob(os.path.join(CSRC, "*.cu")) + glob.glob(os.path.join(CSRC, "*.cuh")) +
                  glob.glob(os.path.join(INCLUDE, "*.h")))


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.isabs(cand) and os.path.exists(cand) or not os.path.isabs(cand)):
            return cand
    return "nvcc"


def build(force: bool = False, verbose: bool = False) -> str:
    """Compile every translation unit of csrc/ (in parallel) and link the library."""
    srcs = sources()
    if not force and os.path.exists(LIBRARY) and os.path.getmtime(LIBRARY) >= max(
            os.path.getmtime(s) for s in srcs):
        return LIBRARY
    objdir = os.path.join(HERE, "_build")
    os.makedirs(objdir, exist_ok=True)
    units = sorted(glob.glob(os.path.join(CSRC, "*.cu")))
    procs = []
    for cu in units:
        obj = os.path.join(objdir, os.path.basename(cu)[:-3] + f".{os.getpid()}.o")
        cmd = [nvcc(), *ARCH, "-lineinfo", "-O3", "-std=c++17", "-Xcompiler", "-fPIC",
               "-I", INCLUDE, "-I", CSRC, "-c", cu, "-o", obj]
        if verbose:
            cmd.insert(1, "-Xptxas=-v")
        procs.append((subprocess.Popen(cmd), obj, cmd))
    try:
        failed = [cmd for p, _, cmd in procs if p.wait() != 0]
        if failed:
            raise subprocess.CalledProcessError(1, failed[0])
        tmp = LIBRARY + f".tmp{os.getpid()}"
        subprocess.run([nvcc(), *ARCH, "-shared", *[o for _, o, _ in procs], "-o", tmp], check=True)
        os.replace(tmp, LIBRARY)
    finally:
        for _, obj, _ in procs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIBRARY


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
