"""GPU Gated DeltaNet tree verification against the per-path recurrence oracle (fp64).

The kernel computes in fp32: K S0 / Q S0 dot products of length d, a forward
substitution along each path (|X_ij| <= beta <= 1 with unit keys) and the output sum,
so errors stay a few 1e-6 of |o| (~1-10 here); the bar is max-abs 2e-4 + 1e-4 |o|.
With bf16 q, k, v (the page's precision) the oracle consumes the same bf16 values, the
arithmetic is still fp32, and the output is rounded to bf16 once: at most half a bf16
spacing, 2^-8 |o|, more, so the bar is 2e-4 + (1e-4 + 2^-8) |o|."""
import numpy as np
import pytest
import torch

import oracle
from tree_verification_attention_gb300 import api, workloads

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _run(c, max_nodes=None, expect_status=0, bf16=False):
    t = {n: torch.from_numpy(np.ascontiguousarray(x)).cuda() for n, x in c.items()}
    if bf16:   # exact: the case holds bf16 values
        for n in ("q", "k", "v"):
            t[n] = t[n].to(torch.bfloat16)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    out = api.gdn_tree_verify(t["cu_nodes"], t["parent"], t["q"], t["k"], t["v"], t["beta"], t["alpha"], t["S0"],
                              max_nodes=max_nodes, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == expect_status
    assert out.dtype == (torch.bfloat16 if bf16 else torch.float32)
    return out.float().cpu().numpy()


def _check(c, bf16=False):
    got = _run(c, bf16=bf16)
    ref = oracle.gdn_tree_outputs(c["q"], c["k"], c["v"], c["beta"], c["alpha"], c["S0"], c["parent"],
                                  c["cu_nodes"])
    err = np.abs(got - ref)
    rel = 1e-4 + (2.0 ** -8 if bf16 else 0.0)
    assert (err <= 2e-4 + rel * np.abs(ref)).all(), (err.max(), np.abs(ref).max())
    return err.max()


@pytest.mark.parametrize("d", [64, 128])
def test_random_trees_match_the_recurrence(d):
    _check(workloads.make_gdn_case(batch=3, heads=4, d=d, m=40, tree="random", seed=d))


def test_workload_shape_best_first():
    _check(workloads.make_gdn_case(batch=1, heads=32, d=128, m=64, tree="best_first", seed=7))


def test_beam_tree_and_ragged_batch():
    rng = np.random.default_rng(8)
    pars = [workloads.beam_tree(rng, (4, 16, 16, 16, 16)), workloads.random_tree(rng, 5),
            workloads.chain_tree(1), workloads.best_first_tree(rng, 30, 4, 8)]
    _check(workloads.make_gdn_case(batch=4, heads=3, d=128, seed=9, parents=pars))


@pytest.mark.parametrize("d", [64, 128])
def test_deepest_tree_a_chain_of_128(d):
    _check(workloads.make_gdn_case(batch=1, heads=2, d=d, m=128, tree="chain", seed=10 + d))


def test_full_random_tree_of_128_nodes():
    _check(workloads.make_gdn_case(batch=2, heads=2, d=128, m=128, tree="random", seed=12))


def test_non_topological_parent_is_reported():
    c = workloads.make_gdn_case(batch=2, heads=2, d=64, m=10, tree="random", seed=13)
    c["parent"] = c["parent"].copy()
    c["parent"][10 + 4] = 6          # second sequence: node 4 claims a later parent
    _run(c, expect_status=3)


def test_tree_larger_than_max_nodes_is_reported():
    c = workloads.make_gdn_case(batch=1, heads=2, d=64, m=20, tree="random", seed=14)
    _run(c, max_nodes=16, expect_status=1)


@pytest.mark.parametrize("d", [64, 128])
def test_bf16_inputs_random_trees(d):
    _check(workloads.make_gdn_case(batch=3, heads=4, d=d, m=40, tree="random", seed=20 + d, dtype="bf16"), bf16=True)


def test_bf16_workload_shape_and_deep_chain():
    _check(workloads.make_gdn_case(batch=1, heads=32, d=128, m=64, tree="best_first", seed=27, dtype="bf16"), bf16=True)
    _check(workloads.make_gdn_case(batch=1, heads=2, d=128, m=128, tree="chain", seed=28, dtype="bf16"), bf16=True)


def test_bf16_rounding_is_the_only_difference_from_fp32():
    """The same bf16-valued inputs through the fp32 and the bf16 entry points: the bf16
    output is the fp32 output rounded once (within one bf16 spacing)."""
    c = workloads.make_gdn_case(batch=2, heads=4, d=128, m=50, tree="random", seed=29, dtype="bf16")
    f32 = _run(c)
    b16 = _run(c, bf16=True)
    assert (np.abs(b16 - f32) <= 2.0 ** -7 * np.abs(f32) + 1e-30).all()
