"""Pins for oracle.tree_attention: the oracle against facts fixed outside itself."""
import numpy as np
import pytest

from oracle import ancestor_mask, tree_verify_attention, tree_verify_attention_rows
from tests import _pins


def test_ancestor_mask_small_tree():
    # tree: 0 and 3 hang off the prefix end, 1 under 0, 2 under 1, 4 under 3
    vis = ancestor_mask(np.array([-1, 0, 1, -1, 3]))
    expect = np.array([
        [1, 0, 0, 0, 0],
        [1, 1, 0, 0, 0],
        [1, 1, 1, 0, 0],
        [0, 0, 0, 1, 0],
        [0, 0, 0, 1, 1]], dtype=bool)
    np.testing.assert_array_equal(vis, expect)


@pytest.mark.parametrize("bad", [[0], [-1, 1], [-1, 0, 5], [-2]])
def test_rejects_non_topological_parent(bad):
    with pytest.raises(ValueError):
        ancestor_mask(np.array(bad))


@pytest.mark.parametrize("P", [0, 1, 37])
def test_every_tree_up_to_six_nodes_equals_path_causal_attention(P):
    """Node i == causal attention at the end of prefix ++ path(root -> i), for every
    topologically ordered parent array with m <= 6 (1 + 1 + 2 + 6 + 24 + 120 + 720 trees)."""
    rng = np.random.default_rng(100 + P)
    ntrees = 0
    for m in range(1, 7):
        for parent in _pins.all_parent_arrays(m):
            prob = _pins.random_problem(rng, P, m, Hq=4, Hkv=2, d=8, parent=parent)
            _pins.check_path_bruteforce(tree_verify_attention, prob)
            ntrees += 1
    assert ntrees == 1 + 2 + 6 + 24 + 120 + 720


def test_chain_equals_causal_attention():
    _pins.check_chain_is_causal(tree_verify_attention, np.random.default_rng(1))
    _pins.check_chain_is_causal(tree_verify_attention, np.random.default_rng(2), P=0, m=5, Hq=3, Hkv=1)


def test_single_node_equals_decode_attention():
    _pins.check_single_node_is_decode(tree_verify_attention, np.random.default_rng(3))
    _pins.check_single_node_is_decode(tree_verify_attention, np.random.default_rng(4), P=0)


def test_all_roots_see_prefix_and_self_only():
    rng = np.random.default_rng(5)
    m = 6
    prob = _pins.random_problem(rng, 11, m, parent=[-1] * m)
    _pins.check_path_bruteforce(tree_verify_attention, prob)
    # a root's result does not depend on any other node's key/value
    out, lse = tree_verify_attention(**prob)
    prob["tree_k"][1:] = 0.0
    prob["tree_v"][1:] = 0.0
    out2, lse2 = tree_verify_attention(**prob)
    assert np.array_equal(out[0], out2[0]) and np.array_equal(lse[0], lse2[0])


def test_uniform_keys_closed_form():
    _pins.check_uniform_closed_form(tree_verify_attention, np.random.default_rng(6))


def test_sibling_independence():
    _pins.check_sibling_independence(tree_verify_attention, np.random.default_rng(7))


def test_relabeling_permutes_outputs():
    _pins.check_relabeling(tree_verify_attention, np.random.default_rng(8))


def test_batch_equals_separate_sequences():
    """A ragged batch is the concatenation of independent single-sequence problems."""
    rng = np.random.default_rng(9)
    probs = [_pins.random_problem(rng, P, m) for P, m in [(7, 3), (0, 5), (20, 1), (3, 6)]]
    cat = lambda k: np.concatenate([p[k] for p in probs], 0)  # noqa: E731
    batch = dict(q=cat("q"), k_cache=cat("k_cache"), v_cache=cat("v_cache"), tree_k=cat("tree_k"),
                 tree_v=cat("tree_v"), parent=cat("parent"), num_kv_heads=2,
                 cu_prefix=np.cumsum([0] + [p["k_cache"].shape[0] for p in probs]),
                 cu_nodes=np.cumsum([0] + [p["q"].shape[0] for p in probs]))
    out, lse = tree_verify_attention(**batch)
    n = 0
    for p in probs:
        o1, l1 = tree_verify_attention(**p)
        m = p["q"].shape[0]
        np.testing.assert_allclose(out[n:n + m], o1, rtol=1e-13, atol=1e-13)
        np.testing.assert_allclose(lse[n:n + m], l1, rtol=1e-13, atol=1e-13)
        n += m


def test_rows_form_matches_full_form():
    rng = np.random.default_rng(10)
    prob = _pins.random_problem(rng, 17, 9, Hq=6, Hkv=3, d=8)
    out, lse = tree_verify_attention(**prob)
    rows = [(n, h) for n in range(9) for h in range(6)]
    o2, l2 = tree_verify_attention_rows(rows, **prob)
    np.testing.assert_allclose(o2, out.reshape(-1, 8), rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(l2, lse.reshape(-1), rtol=1e-12, atol=1e-13)


def test_large_logits_do_not_overflow():
    """Keys scaled x40 give logits in the hundreds: result must stay finite and equal
    the path brute force (which evaluates the same softmax through the library)."""
    rng = np.random.default_rng(11)
    prob = _pins.random_problem(rng, 8, 4, parent=[-1, 0, 0, 2])
    prob["k_cache"] *= 40.0
    prob["tree_k"] *= 40.0
    out, lse = tree_verify_attention(**prob)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse))
    _pins.check_path_bruteforce(tree_verify_attention, prob, rtol=1e-10, atol=1e-10)
