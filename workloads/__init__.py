"""Seeded synthetic inputs for the verification workloads.

This package holds input generators only (target/draft logits, drafted tokens,
per-sequence gate settings).  It contains none of the verification arithmetic
and serves both the CUDA path's tests/benchmark and the oracle's tests.
"""
from .synthetic import CONFIGS, Workload, make, to_numpy_logits  # noqa: F401
