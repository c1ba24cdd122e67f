"""Pins for oracle.kv_commit: the oracle against facts fixed outside itself.

"Faster decoding", section "The scheduler must plan speculative work": only the
accepted draft prefix's target KV is committed.  The strongest pin ties the commit to
the attention definition (LongSpec, "Fast Tree Attention": a tree node sees the
prefix, its ancestors and itself): the committed sequence, read causally, must give
every path node exactly its tree-attention output."""
import numpy as np

from oracle import accept_longest_path, commit_accepted_kv, tree_verify_attention
from tests import _pins
from tree_verification_attention_gb300 import workloads


def test_committed_path_read_causally_equals_tree_attention():
    _pins.check_commit_causal(commit_accepted_kv, tree_verify_attention, np.random.default_rng(11))


def test_only_the_committed_rows_change():
    _pins.check_commit_touches_only_the_path_rows(commit_accepted_kv, np.random.default_rng(12))


def test_empty_path_writes_nothing():
    _pins.check_commit_empty_path_writes_nothing(commit_accepted_kv, np.random.default_rng(13))


def test_fully_accepted_chain_commits_the_tree_rows_in_order():
    _pins.check_commit_full_chain(commit_accepted_kv, np.random.default_rng(14))


def test_commit_of_the_greedy_walk_result():
    """The acceptance walk's own output feeds the commit: each sequence's committed rows
    are the tree rows of the root -> last-accepted-node path, found here by walking the
    parent array up from the last node."""
    w = workloads.make_workload(4, batch=3, prefix=(5, 20), m=12, dtype="fp32")
    alen, apath, _ = accept_longest_path(w.parent, w.draft_tok, w.target_argmax, w.cu_nodes)
    assert alen.max() > 0
    room = 12
    dst = np.array([int(w.cu_prefix[-1]) + room * b for b in range(w.batch)], dtype=np.int32)
    kc = np.zeros((int(w.cu_prefix[-1]) + room * w.batch,) + w.k_cache.shape[1:], dtype=w.k_cache.dtype)
    k_new, _ = commit_accepted_kv(kc, kc, w.tree_k, w.tree_v, w.cu_nodes, alen, apath, dst)
    for b in range(w.batch):
        n0, L = int(w.cu_nodes[b]), int(alen[b])
        if L == 0:
            continue
        last = int(apath[n0 + L - 1])
        path = _pins.path_to(w.parent[n0:int(w.cu_nodes[b + 1])], last)
        np.testing.assert_array_equal(k_new[dst[b]:dst[b] + L], w.tree_k[n0 + np.array(path)])
