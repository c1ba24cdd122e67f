"""Pins for oracle.lse_merge: the aggregation proposition as an fp64 identity."""
import numpy as np
import torch
import torch.nn.functional as F
from scipy.special import logsumexp

from oracle import attention_partial, merge_partials


def _sdpa_one(q, K, V, scale):
    o = F.scaled_dot_product_attention(torch.from_numpy(q)[None, None], torch.from_numpy(K)[None],
                                       torch.from_numpy(V)[None], scale=scale)
    return o[0, 0].numpy(), logsumexp(scale * (K @ q))


def test_partial_matches_library_attention():
    rng = np.random.default_rng(0)
    for n in (1, 2, 17, 300):
        q, K, V = rng.standard_normal(16), rng.standard_normal((n, 16)), rng.standard_normal((n, 16))
        o, lse = attention_partial(q, K, V, 0.25)
        o_ref, l_ref = _sdpa_one(q, K, V, 0.25)
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
        np.testing.assert_allclose(lse, l_ref, rtol=1e-13)


def test_merge_of_any_split_equals_unsplit_softmax():
    """Split the concatenated keys at random points into 1..8 groups; merging the
    groups' partials reproduces attention over all keys (relative 1e-12)."""
    rng = np.random.default_rng(1)
    for trial in range(200):
        n = int(rng.integers(1, 120))
        d = int(rng.choice([4, 8, 16]))
        q, K, V = rng.standard_normal(d) * 2, rng.standard_normal((n, d)), rng.standard_normal((n, d))
        k = int(rng.integers(1, 9))
        cuts = np.sort(rng.integers(0, n + 1, size=k - 1))
        bounds = np.concatenate([[0], cuts, [n]])
        parts = [attention_partial(q, K[a:b], V[a:b], 1 / np.sqrt(d)) for a, b in zip(bounds[:-1], bounds[1:])]
        o, lse = merge_partials(np.stack([p[0] for p in parts]), np.array([p[1] for p in parts]))
        o_ref, l_ref = _sdpa_one(q, K, V, 1 / np.sqrt(d))
        np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-12)
        np.testing.assert_allclose(lse, l_ref, rtol=1e-12)


def test_two_way_merge_is_the_papers_formula():
    """In a range where exp does not overflow, the stable form equals the page's
    literal log(exp(a) + exp(b)) and weights exp(LSE_x - LSE_merge)."""
    rng = np.random.default_rng(2)
    oc, os_ = rng.standard_normal(8), rng.standard_normal(8)
    a, b = 1.3, -0.4
    lm = np.log(np.exp(a) + np.exp(b))
    o, lse = merge_partials(np.stack([oc, os_]), np.array([a, b]))
    np.testing.assert_allclose(lse, lm, rtol=1e-15)
    np.testing.assert_allclose(o, oc * np.exp(a - lm) + os_ * np.exp(b - lm), rtol=1e-14)


def test_empty_group_drops_out_and_order_is_irrelevant():
    rng = np.random.default_rng(3)
    q, K, V = rng.standard_normal(8), rng.standard_normal((10, 8)), rng.standard_normal((10, 8))
    full = attention_partial(q, K, V, 0.3)
    empty = attention_partial(q, K[:0], V[:0], 0.3)
    assert empty[1] == -np.inf and np.all(empty[0] == 0)
    o, lse = merge_partials(np.stack([empty[0], full[0], empty[0]]), np.array([empty[1], full[1], empty[1]]))
    np.testing.assert_allclose(o, full[0], rtol=1e-15)
    assert lse == full[1]
    o_all, l_all = merge_partials(np.zeros((2, 8)), np.array([-np.inf, -np.inf]))
    assert l_all == -np.inf and np.all(o_all == 0)


def test_huge_lse_offsets_are_stable():
    rng = np.random.default_rng(4)
    o1, o2 = rng.standard_normal(4), rng.standard_normal(4)
    o, lse = merge_partials(np.stack([o1, o2]), np.array([1000.0, 1000.0]))
    # ulp(1000) ~ 1.1e-13 bounds how exactly LSE - LSE_merge can be formed here
    np.testing.assert_allclose(lse, 1000.0 + np.log(2.0), rtol=1e-15)
    np.testing.assert_allclose(o, 0.5 * (o1 + o2), rtol=1e-12)
    o, lse = merge_partials(np.stack([o1, o2]), np.array([-1e4, 0.0]))
    np.testing.assert_allclose(o, o2, rtol=1e-15)
