"""GPU stochastic chain verification: bit-exact against the oracle on the same uniforms,
and the frequency pins of the oracle applied to the GPU's own outputs."""
import numpy as np
import pytest
import torch

import oracle
from tree_verification_attention_gb300 import api
from tests import _pins

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _gpu_verify(p, q, draft, ua, us, cu, max_draft=None, status=None):
    f = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()  # noqa: E731
    i = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()    # noqa: E731
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    q2 = np.asarray(q, np.float32).reshape(-1, np.asarray(p).shape[1])
    alen, out = api.verify_chain_sampling(i(cu), f(p), f(q2), i(draft), f(ua), f(us), max_draft=max_draft,
                                          dev_status=st)
    torch.cuda.synchronize()
    if status is not None:
        status.append(int(st.item()))
    else:
        assert int(st.item()) == 0
    return alen.cpu().numpy(), out.cpu().numpy()


def _softmax_rows(rng, rows, V, temp):
    z = rng.standard_normal((rows, V)) * temp
    e = np.exp(z - z.max(1, keepdims=True))
    return (e / e.sum(1, keepdims=True)).astype(np.float32)


def _random_case(rng, B, V, max_gamma=8, temp=3.0):
    gam = rng.integers(0, max_gamma + 1, B)
    cu = np.concatenate([[0], np.cumsum(gam)]).astype(np.int32)
    p = _softmax_rows(rng, int(cu[-1]) + B, V, temp)
    q = _softmax_rows(rng, max(int(cu[-1]), 1), V, temp)[: int(cu[-1])]
    # drafts ~ q; p correlated with q so that acceptances happen
    p_mix = p.copy()
    for b in range(B):
        for k in range(int(gam[b])):
            r = int(cu[b]) + b + k
            p_mix[r] = (0.7 * q[int(cu[b]) + k] + 0.3 * p[r]).astype(np.float32)
    draft = np.array([rng.choice(V, p=q[g].astype(np.float64) / q[g].astype(np.float64).sum())
                      for g in range(int(cu[-1]))], dtype=np.int32)
    ua = rng.random(int(cu[-1])).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    return p_mix, q, draft, ua, us, cu


@pytest.mark.parametrize("B,V", [(64, 7), (16, 1000), (3, 128256)])
def test_bit_exact_against_oracle(B, V):
    rng = np.random.default_rng(B * 7 + V)
    case = _random_case(rng, B, V)
    a_gpu, o_gpu = _gpu_verify(*case)
    a_ref, o_ref = oracle.verify_chain_sampling(*case)
    np.testing.assert_array_equal(a_gpu, a_ref)
    np.testing.assert_array_equal(o_gpu, o_ref)
    assert (a_ref < np.diff(case[5])).any() and (a_ref > 0).any()   # both outcomes occur


@pytest.mark.parametrize("V", [600000, 600001])
def test_large_vocabulary_multi_group_pieces(V):
    """A vocabulary above about 262 K tokens gives each thread of the drawing CTA a piece
    of more than one group of 4 entries (its walk reads the later groups again); V not a
    multiple of 4 takes the scalar loads."""
    rng = np.random.default_rng(V % 7)
    case = _random_case(rng, 3, V, max_gamma=4, temp=4.0)
    a_gpu, o_gpu = _gpu_verify(*case)
    a_ref, o_ref = oracle.verify_chain_sampling(*case)
    np.testing.assert_array_equal(a_gpu, a_ref)
    np.testing.assert_array_equal(o_gpu, o_ref)
    assert (a_ref < np.diff(case[5])).any() and (a_ref == np.diff(case[5])).any()   # residual and bonus draws


def test_masses_outside_the_fast_split_range_are_exact():
    """Unnormalised nonnegative masses with entries planted at 2 and above: the slice sums
    take the split fp32 form only for rounds whose masses all lie in [0, 2) and sum the
    other rounds again on the integer path, so the draws stay bit-exact."""
    rng = np.random.default_rng(57)
    p, q, draft, ua, us, cu = _random_case(rng, 5, 128256)
    p, q = (4 * p).astype(np.float32), (4 * q).astype(np.float32)
    for rows in (p, q):
        for r in range(rows.shape[0]):
            at = rng.choice(rows.shape[1], 6, replace=False)
            rows[r, at] = rng.uniform(2.0, 300.0, 6).astype(np.float32)
    a_gpu, o_gpu = _gpu_verify(p, q, draft, ua, us, cu)
    a_ref, o_ref = oracle.verify_chain_sampling(p, q, draft, ua, us, cu)
    np.testing.assert_array_equal(a_gpu, a_ref)
    np.testing.assert_array_equal(o_gpu, o_ref)


def test_gpu_outputs_follow_the_target_distribution():
    _pins.check_sampling_marginals(_gpu_verify, np.random.default_rng(51), n=60000)


def test_gpu_forced_first_late_and_no_rejection():
    _pins.check_sampling_forced_cases(_gpu_verify, np.random.default_rng(52), n=4000)


def test_empty_residual_falls_back_to_p():
    rng = np.random.default_rng(53)
    V, B = 50, 200
    q = _softmax_rows(rng, B, V, 1.0)
    p = np.concatenate([0.5 * q, _softmax_rows(rng, B, V, 1.0)]).astype(np.float32)
    # sequence b: one draft at q row b; p rows: [b] (half of q, so the residual is empty) ...
    p_rows = np.empty((2 * B, V), np.float32)
    p_rows[0::2] = p[:B]
    p_rows[1::2] = p[B:]
    cu = np.arange(B + 1, dtype=np.int32)
    draft = np.array([rng.choice(V, p=q[b].astype(np.float64) / q[b].astype(np.float64).sum()) for b in range(B)],
                     np.int32)
    ua = rng.random(B).astype(np.float32)
    us = rng.random(B).astype(np.float32)
    a_gpu, o_gpu = _gpu_verify(p_rows, q, draft, ua, us, cu)
    a_ref, o_ref = oracle.verify_chain_sampling(p_rows, q, draft, ua, us, cu)
    np.testing.assert_array_equal(a_gpu, a_ref)
    np.testing.assert_array_equal(o_gpu, o_ref)
    assert (a_ref == 0).sum() > 50


def test_sequences_without_drafts_draw_the_bonus():
    rng = np.random.default_rng(54)
    V, B = 40, 30
    p = _softmax_rows(rng, B, V, 2.0)
    cu = np.zeros(B + 1, np.int32)
    us = rng.random(B).astype(np.float32)
    empty_f, empty_i = np.zeros(0, np.float32), np.zeros(0, np.int32)
    a_gpu, o_gpu = _gpu_verify(p, np.zeros((0, V), np.float32), empty_i, empty_f, us, cu, max_draft=0)
    a_ref, o_ref = oracle.verify_chain_sampling(p, np.zeros((0, V), np.float32), empty_i, empty_f, us, cu)
    np.testing.assert_array_equal(a_gpu, a_ref)
    np.testing.assert_array_equal(o_gpu, o_ref)


@pytest.mark.parametrize("bad", ["token", "q_zero", "u_one", "gamma"])
def test_invalid_sequence_is_flagged_and_others_are_unaffected(bad):
    p, q, draft, ua, us, cu = _random_case(np.random.default_rng(56), 6, 30, max_gamma=5)
    b = int(np.argmax(np.diff(cu)))          # a sequence with the most drafts (at least one)
    g = int(cu[b])
    max_draft = int(np.diff(cu).max())
    p2, q2, d2, ua2 = p, q.copy(), draft.copy(), ua.copy()
    if bad == "token":
        d2[g] = 30
    elif bad == "q_zero":
        q2[g, d2[g]] = 0.0
    elif bad == "u_one":
        ua2[g] = 1.0
    else:
        max_draft -= 1
    st = []
    a_gpu, o_gpu = _gpu_verify(p2, q2, d2, ua2, us, cu, max_draft=max_draft, status=st)
    assert st[0] == 1
    assert a_gpu[b] == 0 and o_gpu[b] == -1
    # the other sequences' results do not depend on sequence b's inputs
    others = [i for i in range(6) if np.diff(cu)[i] <= max_draft and i != b]
    a_ref, o_ref = oracle.verify_chain_sampling(p, q, draft, ua, us, cu)
    np.testing.assert_array_equal(a_gpu[others], a_ref[others])
    np.testing.assert_array_equal(o_gpu[others], o_ref[others])
