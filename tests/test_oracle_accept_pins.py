"""Pins for oracle.acceptance and oracle.expected_tokens."""
import os

import numpy as np
import pytest

from oracle import accept_longest_path, expected_tokens, iid_expected_tokens, survival_from_conditional
from tests import _pins

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "expected_tokens_worked_example.txt")


def _golden():
    vals = {}
    with open(GOLDEN) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            key, *nums = line.split()
            vals[key] = [float(x) for x in nums]
    return vals


def test_worked_example_survival_and_expected_tokens():
    g = _golden()
    s = survival_from_conditional(g["conditional"])
    np.testing.assert_allclose(s, g["survival"], rtol=0, atol=1e-15)
    assert abs(expected_tokens(s) - g["expected_tokens"][0]) < 1e-12
    assert f"{expected_tokens(s):.4f}" == "3.0230"


def test_worked_example_iid_estimate_differs():
    g = _golden()
    alpha = float(np.mean(g["conditional"]))
    assert abs(alpha - g["iid_alpha"][0]) < 1e-15
    iid = iid_expected_tokens(alpha, len(g["conditional"]))
    assert abs(iid - g["iid_expected_tokens"][0]) < 1e-12
    assert abs(iid - sum(alpha ** k for k in range(5))) < 1e-12
    assert f"{iid:.4f}" == "2.5256"
    assert abs(iid - g["expected_tokens"][0]) > 0.4
    assert iid_expected_tokens(1.0, 4) == 5.0


def test_walk_reproduces_expected_tokens_by_enumeration():
    """Exhaustive 2^4 accept patterns on a chain, weighted by the page's conditional
    probabilities: sum Pr * (accept_len + 1) must equal E[Y] = 3.0230."""
    g = _golden()
    ey = _pins.chain_expected_tokens_by_enumeration(accept_longest_path, g["conditional"])
    assert abs(ey - g["expected_tokens"][0]) < 1e-12


def _chain_case(matches, gamma=5):
    parent = np.arange(-1, gamma - 1, dtype=np.int32)
    slot = np.arange(10, 10 + gamma + 1, dtype=np.int32)
    draft = np.array([slot[k] if matches[k] else 999 for k in range(gamma)], np.int32)
    return accept_longest_path(parent, draft, slot, np.array([0, gamma], np.int32))


def test_forced_first_rejection_late_rejection_all_accept():
    alen, path, nxt = _chain_case([0, 1, 1, 1, 1])
    assert alen[0] == 0 and nxt[0] == 10 and all(path == -1)
    alen, path, nxt = _chain_case([1, 1, 1, 0, 1])
    assert alen[0] == 3 and list(path[:3]) == [0, 1, 2] and nxt[0] == 13
    alen, path, nxt = _chain_case([1, 1, 1, 1, 1])
    assert alen[0] == 5 and list(path) == [0, 1, 2, 3, 4] and nxt[0] == 15   # bonus token


def test_wide_tree_fully_rejected():
    m = 16
    parent = np.full(m, -1, np.int32)
    slot = np.full(m + 1, 7, np.int32)
    draft = np.arange(100, 100 + m, dtype=np.int32)
    alen, path, nxt = accept_longest_path(parent, draft, slot, np.array([0, m], np.int32))
    assert alen[0] == 0 and nxt[0] == 7 and all(path == -1)


def test_tie_goes_to_smaller_index():
    # two accepted siblings of depth 1: node 0 and node 1 both match slot[0]
    parent = np.array([-1, -1, 1], np.int32)
    slot = np.array([5, 6, 8, 9], np.int32)
    draft = np.array([5, 5, 1], np.int32)
    alen, path, nxt = accept_longest_path(parent, draft, slot, np.array([0, 3], np.int32))
    assert alen[0] == 1 and path[0] == 0 and nxt[0] == 6


def test_every_tree_up_to_six_nodes_against_forward_enumeration():
    _pins.check_accept_bruteforce(accept_longest_path, np.random.default_rng(0), max_m=6, vocab=2, draws=2)


def test_ragged_batch_keeps_order_and_offsets():
    rng = np.random.default_rng(1)
    sizes = [3, 0, 7, 1, 5]
    parents, drafts, slots = [], [], []
    for m in sizes:
        parents.append(np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, m)], np.int32)[:m])
        slots.append(rng.integers(0, 2, m + 1).astype(np.int32))
        drafts.append(rng.integers(0, 2, m).astype(np.int32))
    cu = np.cumsum([0] + sizes).astype(np.int32)
    alen, path, nxt = accept_longest_path(np.concatenate(parents), np.concatenate(drafts),
                                          np.concatenate(slots), cu)
    for b, m in enumerate(sizes):
        L, p, tok = _pins.bruteforce_accept(parents[b], drafts[b], slots[b])
        assert alen[b] == L and nxt[b] == tok
        assert list(path[cu[b]:cu[b] + L]) == p
        assert all(path[cu[b] + L:cu[b + 1]] == -1)


def test_rejects_bad_parent():
    with pytest.raises(ValueError):
        accept_longest_path(np.array([-1, 1], np.int32), np.zeros(2, np.int32), np.zeros(3, np.int32),
                            np.array([0, 2], np.int32))
