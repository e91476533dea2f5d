"""Bounded waits of the verifying stream pass.

The stream pass takes its work units from CTAs that have not started (cluster
launch control), waiting for each answer in shared memory.  Every such wait
has an iteration limit; a test hook makes each CTA's first wait use a barrier
that nothing completes, so the limit runs out.  The call must then return
normally with every sequence failed closed (a unit of work may have been
lost), and later calls on the handle must be unaffected."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from tests.gpu_helpers import compare, oracle_for, peaked_workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def sv():
    import speculative_decoding_verification_online_gb300 as pkg
    from speculative_decoding_verification_online_gb300 import build as B
    B.build()
    pkg.load()
    return pkg


def _call(sv, ver, w, T=None):
    cnt = torch.zeros(8, dtype=torch.int64, device="cuda")
    out = ver.run(w.Lt, w.Ld, w.D, w.T if T is None else T, gate_mode=sv.SV_GATED_MU, threshold=0.5,
                  seed=w.philox_seed, counters=cnt)
    torch.cuda.synchronize()
    return out, cnt.cpu().numpy()


@pytest.mark.parametrize("T", [1.0, 0.0])
def test_a_wait_that_gives_up_fails_the_call_closed(sv, T):
    B, k, V = 24, 3, 70000  # 5 units per row: most CTAs wait for a second unit
    w = peaked_workload(B, k, V, "bf16", seed=404, gate=1, tau=0.5, T=T)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_test_hooks(wait_limit=4096, stall_first_request=True)
    out, cnt = _call(sv, ver, w)
    assert torch.all(out["accepted_len"] == -1)
    assert torch.all(out["tokens"] == -1)
    assert torch.all(out["flags"] == sv.SV_FLAG_INVALID)
    assert torch.all(out["accept_prob"] == 0)
    assert cnt[6] == B and cnt[1] == 0
    # hooks off: the next calls (which use the other error word, then the
    # failed call's word again) are correct
    ver.set_test_hooks(0, False)
    ref = oracle_for(w)
    for i in range(2):
        out, cnt = _call(sv, ver, w)
        compare(w, out, ref, what=f"after a wait gave up, call {i + 1} (T={T})")
        assert cnt[6] == 0
    ver.close()


def test_a_small_limit_without_the_stall_still_verifies(sv):
    # a limit far below the default, with answers that arrive in time
    B, k, V = 32, 4, 90000
    w = peaked_workload(B, k, V, "bf16", seed=405, gate=1, tau=0.5)
    ver = sv.SpecVerifier(B, k, V, device=0)
    ver.set_test_hooks(wait_limit=1 << 16, stall_first_request=False)
    out, cnt = _call(sv, ver, w)
    compare(w, out, oracle_for(w), what="small wait limit")
    assert cnt[6] == 0
    ver.close()
