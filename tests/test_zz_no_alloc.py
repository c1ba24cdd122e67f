"""The allocation-free entry point (tree_verify_attn_varlen_noalloc).

Callers that may not allocate device memory - an engine that owns every allocation
and forbids cudaMalloc on its execution path, or a plugin interface with no workspace
argument - call this form; its scratch is a fixed 32 MiB array inside the library.
This file is collected last on purpose.  It checks, through the C ABI, that two calls
in a row (on different problems, so the second one starts from the first one's
leftover scratch) match the float64 oracle within the parity tolerances and are bit
for bit the workspace form's results (the same kernels, layout and reduction order run
on both, so any difference would be stale scratch leaking in), and that a problem too
large for the fixed scratch is refused before anything runs.
"""
import ctypes

import pytest
import torch

from tree_verification_attention_gb300 import api, workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _both(w):
    t = _gpu.to_device(w)
    args = (t["q"], t["k_cache"], t["v_cache"], t["tree_k"], t["tree_v"], t["parent"], t["cu_prefix"],
            t["cu_nodes"], max(1, int(w.prefix_lens.max())), int(w.tree_sizes.max()))
    st_ref = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    st_new = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    o_new, l_new = api.tree_verify_attn_varlen_noalloc(*args, dev_status=st_new)
    o_ws, l_ws = api.tree_verify_attn_varlen(*args, dev_status=st_ref)
    torch.cuda.synchronize()
    assert int(st_ref.item()) == 0 and int(st_new.item()) == 0
    return o_new, l_new, o_ws, l_ws


def test_two_calls_in_a_row_match_the_oracle_and_the_workspace_form():
    for w in (workloads.make_workload(3, prefix=1500), workloads.make_workload(4, prefix=(200, 1300))):
        o_new, l_new, o_ws, l_ws = _both(w)
        o_ref, l_ref = _gpu.oracle_attention(w)
        _gpu.assert_close(w, o_new.double().cpu().numpy(), l_new.double().cpu().numpy(), o_ref, l_ref, w.name)
        assert torch.equal(o_new, o_ws) and torch.equal(l_new, l_ws), w.name


def test_too_large_for_the_static_scratch_is_refused():
    lib = api.load_library()
    fn = lib.tree_verify_attn_varlen_noalloc
    fn.restype = ctypes.c_int
    fn.argtypes = [ctypes.POINTER(api.Params)] + [ctypes.c_void_p] * 10
    w = workloads.make_workload(3, prefix=256, m=8)
    t = _gpu.to_device(w)
    p = api.make_params(t["q"], t["k_cache"], t["cu_prefix"], t["cu_nodes"], 8, 256, 8)
    p.batch, p.max_nodes = 1024, 128       # bound-driven scratch far beyond 32 MiB
    assert api.workspace_size(p) > (32 << 20)
    out = torch.empty_like(t["q"])
    lse = torch.empty(t["q"].shape[:2], dtype=torch.float32, device="cuda:0")
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    ptr = lambda x: ctypes.c_void_p(x.data_ptr())  # noqa: E731
    code = fn(ctypes.byref(p), ptr(t["q"]), ptr(t["k_cache"]), ptr(t["v_cache"]), ptr(t["tree_k"]),
              ptr(t["tree_v"]), ptr(t["parent"]), ptr(out), ptr(lse), ptr(st),
              ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert code == 4
    assert b"static buffer" in lib.tva_last_error()
    torch.cuda.synchronize()
    assert int(st.item()) == 0
