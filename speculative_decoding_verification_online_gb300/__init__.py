"""GB300 (sm_103a) batched speculative-decoding verification.

Modified rejection sampling in plain and mu/NULL-gated modes: a streaming
kernel and a per-sequence finishing kernel behind the C ABI of
``include/spec_verify.h``.  This package holds the CUDA sources (``csrc/``),
the build step, the ctypes binding, the sequence-sharding helper and the
acceptance summary over the batch counters (``metrics``).
"""
from .spec_verify import (  # noqa: F401
    COUNTER_NAMES, SV_BF16, SV_CNT_ACCEPTED, SV_CNT_BONUS, SV_CNT_BOUNDARY, SV_CNT_DEGENERATE, SV_CNT_INVALID,
    SV_CNT_NULL, SV_CNT_REJECTED, SV_CNT_TESTED, SV_F32, SV_FLAG_ACCEPT, SV_FLAG_INVALID, SV_FLAG_NULL, SV_FLAG_REJECT,
    SV_FLAG_UNREACHED, SV_GATED_MU, SV_PLAIN, SpecVerifier, SpecVerifyError, load,
    spec_verify_diagnostics, spec_verify_free, spec_verify_init, spec_verify_launches_per_run, spec_verify_mark_next,
    spec_verify_run, spec_verify_run_ex, spec_verify_run_host, spec_verify_run_noalloc,
    spec_verify_set_filters, spec_verify_set_gate_policy, spec_verify_status_string, run_noalloc,
    spec_verify_launches_per_filtered_run)
from .metrics import acceptance_summary, rule_id, summary_line  # noqa: F401,E402
