"""The device-side timeout path of the tensor-core partials kernel.

Every wait inside that kernel is bounded; when one runs out the kernel raises an abort
flag, lets the copies and MMAs it already started finish, frees its tensor memory,
returns and records TVA_ERR_TIMEOUT in the caller's status word ("Faster decoding",
"Correctness & fault tests": failures must be detected and reported, not hang).
Here the wait is made to run out on purpose, through the library's diagnostic hook:
the MMA-issuing thread waits on a barrier that nothing completes, with a short limit.
Nothing faults or hangs; the next normal call on the same stream must then match the
oracle, which shows that the aborted launch left no tensor memory allocated and no
copy in flight.
"""
import pytest
import torch

from tree_verification_attention_gb300 import api, workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()
    yield
    api.diag_set_wait_limit(0, False)


@pytest.mark.parametrize("cfg,over", [(3, dict(prefix=1500, m=40)), (6, dict(prefix=700, batch=3)),
                                      (1, dict(d=64, Hq=8, Hkv=2, prefix=600, m=20, dtype="bf16")),
                                      (5, dict(prefix=900))],
                         ids=["bf16-d128-two-mtiles", "fp16-d128-batch", "bf16-d64", "bf16-shared-kv-teams"])
def test_expired_wait_reports_timeout_and_the_next_call_is_exact(cfg, over):
    w = workloads.make_workload(cfg, **over)
    t = _gpu.to_device(w)
    try:
        api.diag_set_wait_limit(50_000, True)   # 50 us, and a wait nothing completes
        _, _, st = _gpu.run_attention(w, t)
    finally:
        api.diag_set_wait_limit(0, False)
    assert st == 6, api.STATUS.get(st, st)
    out, lse, st2 = _gpu.run_attention(w, t)
    assert st2 == 0
    o_ref, l_ref = _gpu.oracle_attention(w)
    _gpu.assert_close(w, out, lse, o_ref, l_ref, f"after a timeout, {w.name}")


def test_short_limit_without_a_stall_still_completes():
    """A limit shorter than the default but far above any real wait changes nothing."""
    w = workloads.make_workload(3, prefix=2000, m=64)
    t = _gpu.to_device(w)
    try:
        api.diag_set_wait_limit(20_000_000, False)   # 20 ms
        out, lse, st = _gpu.run_attention(w, t)
    finally:
        api.diag_set_wait_limit(0, False)
    assert st == 0
    o_ref, l_ref = _gpu.oracle_attention(w)
    _gpu.assert_close(w, out, lse, o_ref, l_ref)
    torch.cuda.synchronize()
