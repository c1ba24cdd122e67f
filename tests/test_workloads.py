"""The seeded input generators: shapes, determinism, tree structure, bf16 rounding."""
import numpy as np
import pytest
import torch

from tree_verification_attention_gb300 import workloads as W
from tree_verification_attention_gb300 import workloads


def test_bf16_rounding_matches_torch():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(100000).astype(np.float32) * 10,
                        np.array([1.0 + 2 ** -8, 1.0 + 3 * 2 ** -8, -0.0, 65504.0, 1e-30], np.float32)])
    ours = W.bf16_round_bits(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(ours, ref)
    back = W.bits_to_f64(ours)
    np.testing.assert_array_equal(back, torch.from_numpy(x).to(torch.bfloat16).double().numpy())


@pytest.mark.parametrize("config", [1, 2, 3, 4, 5])
def test_small_variants_have_the_right_structure(config):
    over = dict(prefix=300) if config != 4 else dict(prefix=(100, 400))
    w = W.make_workload(config, **over)
    d = W.workload_defaults(config)
    B, m = d["batch"], d["m"]
    assert w.batch == B and w.num_nodes == B * m
    assert w.q.shape == (B * m, d["Hq"], d["d"])
    assert w.k_cache.shape == (int(w.cu_prefix[-1]), d["Hkv"], d["d"])
    assert w.tree_k.shape == (B * m, d["Hkv"], d["d"])
    assert w.target_argmax.shape == (B * m + B,)
    assert w.q.dtype == (np.float32 if config == 1 else np.uint16)
    for b in range(B):
        par = w.parent[w.cu_nodes[b]:w.cu_nodes[b + 1]]
        assert all(-1 <= p < i for i, p in enumerate(par))
        depth = W.tree_depths(par)
        if "max_depth" in d:
            assert depth.max() <= d["max_depth"]
    if config == 2:
        assert list(w.parent) == list(range(-1, 7))
    if config == 4:
        assert np.all((w.prefix_lens >= 100) & (w.prefix_lens <= 400))


def test_deterministic():
    a = W.make_workload(3, prefix=256)
    b = W.make_workload(3, prefix=256)
    for k in ("parent", "draft_tok", "target_argmax", "q", "k_cache", "v_cache", "tree_k", "tree_v"):
        np.testing.assert_array_equal(getattr(a, k), getattr(b, k))
    c = W.make_workload(3, seed=7, prefix=256)
    assert not np.array_equal(a.q, c.q)


def test_full_size_trees():
    """The full-size tree shapes (only the tree part is drawn here, cheaply)."""
    rng = np.random.Generator(np.random.PCG64(1003))
    par = W.best_first_tree(rng, 64, width=4, max_depth=8)
    assert len(par) == 64 and W.tree_depths(par).max() <= 8
    assert all(-1 <= p < i for i, p in enumerate(par))
    rng = np.random.Generator(np.random.PCG64(1005))
    par = W.best_first_tree(rng, 128, width=8, max_depth=10)
    assert len(par) == 128 and W.tree_depths(par).max() <= 10
    # every node's child count is at most the branch bound
    counts = np.bincount(par[par >= 0], minlength=128)
    assert counts.max() <= 4 and np.sum(par == -1) <= 4


def test_best_first_degenerate_shapes():
    """One child per expansion and width 1 gives a chain; running out of expandable
    nodes before m nodes is an error, not a short tree."""
    rng = np.random.default_rng(0)
    assert list(W.best_first_tree(rng, 5, width=1, max_depth=5, max_branch=1)) == [-1, 0, 1, 2, 3]
    par = W.best_first_tree(np.random.default_rng(1), 1, width=8, max_depth=1, max_branch=4)
    assert list(par) == [-1]
    with pytest.raises(ValueError):
        W.best_first_tree(np.random.default_rng(0), 5, width=1, max_depth=2, max_branch=1)


def test_match_probability_and_sink_scaling():
    w = W.make_workload(3, prefix=128, m=64, vocab=1000)
    slots = w.target_argmax[:65]
    match = w.draft_tok == slots[w.parent + 1]
    assert 0.5 < match.mean() < 0.9
    w5 = W.make_workload(5, prefix=1000, m=16)
    k = W.bits_to_f64(w5.k_cache)
    norms = np.linalg.norm(k[:, 0, :], axis=1)
    assert np.sum(norms > 2.5 * np.median(norms)) == 10     # 1% of 1000 keys boosted x4


def test_beam_tree_levels_follow_the_widths():
    """LongSpec's beam widths [4, 16, 16, 16, 16]: step s holds widths[s] nodes whose
    parents are nodes of step s - 1, and a surviving candidate outscores every dropped one
    (checked on the returned structure: level sizes and parent levels)."""
    rng = np.random.default_rng(0)
    for widths in ([4, 16, 16, 16, 16], [2, 3, 5], [1, 1, 1, 1], [7]):
        par = workloads.beam_tree(rng, widths)
        assert len(par) == sum(widths)
        depth = workloads.tree_depths(par)
        np.testing.assert_array_equal(np.bincount(depth)[1:], widths)
        start = np.concatenate([[0], np.cumsum(widths)])
        for lvl in range(1, len(widths)):
            kids = par[start[lvl]:start[lvl + 1]]
            assert ((kids >= start[lvl - 1]) & (kids < start[lvl])).all()


def test_fp16_storage_is_ieee_half_rounding():
    import torch
    x = np.random.default_rng(1).standard_normal(10000).astype(np.float32) * 100
    bits = workloads.f16_round_bits(x)
    ref = torch.from_numpy(x).to(torch.float16).view(torch.int16).numpy().view(np.uint16)
    np.testing.assert_array_equal(bits, ref)
    np.testing.assert_array_equal(workloads.f16_bits_to_f64(bits), torch.from_numpy(x).to(torch.float16).double().numpy())
    w = workloads.make_workload(6, prefix=64)
    assert w.dtype == "fp16" and w.q.dtype == np.uint16 and w.num_nodes == 68
