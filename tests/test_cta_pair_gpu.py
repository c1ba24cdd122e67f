"""GPU parity of the CTA-pair attention partials kernel (selected through the
tva_diag_use_cta_pair diagnostic), against the float64 oracle.

The pair kernel applies to bf16 / fp16 problems at head_dim 128 whose row groups hold two
M-tiles (max_nodes * G > 128; a single sequence whose tree one-M-tile groups cover with
fewer M-tiles gets those instead, and no pair).  Each case first checks that the selection took effect: the
pair kernel runs one worker per two SMs.
"""
import numpy as np
import pytest
import torch

from tree_verification_attention_gb300 import api, workloads
from tests import _gpu

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _pair():
    import __graft_entry__
    __graft_entry__.build()
    api.diag_use_cta_pair(True)
    yield
    api.diag_use_cta_pair(False)


def _workers(w, t):
    prm = api.make_params(t["q"], t["k_cache"], t["cu_prefix"], t["cu_nodes"], w.num_kv_heads,
                          max(1, int(w.prefix_lens.max())), int(w.tree_sizes.max()))
    return api.num_workers(prm)


CASES = [
    (3, dict(prefix=1500)),                                   # 64-node best-first tree
    (5, dict(prefix=900)),                                    # G = 8, 128 nodes: 4 row groups
    (6, dict(prefix=700, batch=3)),                           # fp16 beam trees, 68 nodes
    (1, dict(batch=2, Hq=12, Hkv=4, d=128, prefix=(77, 200), m=50, tree="random", dtype="bf16",
             vocab=8, seed=77)),                              # 126-row M-tiles
    (1, dict(batch=1, Hq=32, Hkv=8, d=128, prefix=300, m=128, tree="random", dtype="fp16",
             vocab=8, seed=77)),
    (1, dict(batch=6, Hq=32, Hkv=8, d=128, prefix=(0, 900), m=40, tree="random", dtype="bf16",
             vocab=8, seed=5)),                               # empty prefixes, many segments
]


@pytest.mark.parametrize("cfg,over", CASES, ids=[f"pair{i}" for i in range(len(CASES))])
def test_pair_kernel_matches_oracle(cfg, over):
    w = workloads.make_workload(cfg, **over)
    t = _gpu.to_device(w)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert _workers(w, t) == sms // 2
    out, lse, st = _gpu.run_attention(w, t)
    assert st == 0
    o_ref, l_ref = _gpu.oracle_attention(w)
    _gpu.assert_close(w, out, lse, o_ref, l_ref, f"pair kernel, config {cfg} {over}")


def test_pair_kernel_full_size_64k_prefix(record_property):
    """The 64k-prefix, 64-node best-first workload at full size, every row of every KV
    head, through the single-sequence entry point the bench uses."""
    from tests.test_parity_gpu import _oracle_heads
    w = workloads.make_workload(3)
    t = _gpu.to_device(w)
    o, l = api.tree_verify_attn(t["q"], t["k_cache"], t["v_cache"], t["tree_k"], t["tree_v"], t["parent"])
    torch.cuda.synchronize()
    out, lse = o.double().cpu().numpy(), l.double().cpu().numpy()
    assert api.read_device_status() == 0
    del t, o, l
    G = w.num_q_heads // w.num_kv_heads
    worst = (0.0, 0.0)
    for g, (o_ref, l_ref) in _oracle_heads(w, range(w.num_kv_heads)).items():
        e = _gpu.assert_close(w, out[:, g * G:(g + 1) * G], lse[:, g * G:(g + 1) * G], o_ref, l_ref,
                              f"pair kernel, full 64k workload, KV head {g}")
        worst = (max(worst[0], e[0]), max(worst[1], e[1]))
    record_property("max_abs_out", worst[0])
    record_property("max_rel_lse", worst[1])
    print(f"\npair kernel, full 64k workload: max-abs(out) {worst[0]:.3e}, rel(lse) {worst[1]:.3e}")


@pytest.mark.parametrize("cfg,over", [(3, dict(prefix=1500, m=40)), (6, dict(prefix=700, batch=3))],
                         ids=["bf16", "fp16-batch"])
def test_pair_kernel_expired_wait_reports_timeout_and_the_next_call_is_exact(cfg, over):
    """The pair's timeout path: the MMA-issuing warp of each pair's first CTA waits on a
    barrier nothing completes (a 50 us limit), both CTAs abort, the first CTA drains the
    copies of both, they free their tensor memory together and TVA_ERR_TIMEOUT is
    recorded; the next normal call on the same stream must match the oracle."""
    w = workloads.make_workload(cfg, **over)
    t = _gpu.to_device(w)
    try:
        api.diag_set_wait_limit(50_000, True)
        _, _, st = _gpu.run_attention(w, t)
    finally:
        api.diag_set_wait_limit(0, False)
    assert st == 6, api.STATUS.get(st, st)
    out, lse, st2 = _gpu.run_attention(w, t)
    assert st2 == 0
    o_ref, l_ref = _gpu.oracle_attention(w)
    _gpu.assert_close(w, out, lse, o_ref, l_ref, f"pair kernel after a timeout, {w.name}")


def test_default_kernel_restored_after_deselect():
    w = workloads.make_workload(3, prefix=1500)
    t = _gpu.to_device(w)
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    api.diag_use_cta_pair(False)
    try:
        assert _workers(w, t) == sms
        out, lse, st = _gpu.run_attention(w, t)
        assert st == 0
        o_ref, l_ref = _gpu.oracle_attention(w)
        _gpu.assert_close(w, out, lse, o_ref, l_ref, "default kernel after deselect")
    finally:
        api.diag_use_cta_pair(True)
    assert np.isfinite(out).all()
