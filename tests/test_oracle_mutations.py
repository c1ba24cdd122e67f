"""Each pin must catch a plausible mistake planted in the oracle (on the CPU).

The mutants below are the real oracle with one thing changed: the node's own key
masked out, a proper-ancestor slip, the wrong softmax scale, the wrong GQA mapping, the
tree K/V swapped, the prefix dropped, an LSE term dropped, ties broken the other way,
the bonus token read from the wrong slot.  Every one must make at least one pin fail."""
import numpy as np
import pytest

import oracle.tree_attention as ta
from oracle import accept_longest_path, attention_partial, merge_partials, tree_verify_attention
from tests import _pins


def _attention_pins_fail(fn):
    rng = np.random.default_rng(0)
    checks = [
        lambda: [_pins.check_path_bruteforce(fn, _pins.random_problem(rng, P, m, parent=par))
                 for P in (0, 5) for m in range(1, 5) for par in _pins.all_parent_arrays(m)],
        lambda: _pins.check_chain_is_causal(fn, rng),
        lambda: _pins.check_single_node_is_decode(fn, rng),
        lambda: _pins.check_uniform_closed_form(fn, rng),
        lambda: _pins.check_sibling_independence(fn, rng),
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except AssertionError:
            failed += 1
    return failed


def test_real_oracle_passes_all_attention_pins():
    assert _attention_pins_fail(tree_verify_attention) == 0


def test_mutant_self_not_visible(monkeypatch):
    real = ta.ancestor_mask

    def no_self(parent):
        v = real(parent)
        np.fill_diagonal(v, False)
        return v
    monkeypatch.setattr(ta, "ancestor_mask", no_self)
    with np.errstate(invalid="ignore", divide="ignore"):
        assert _attention_pins_fail(ta.tree_verify_attention) > 0


def test_mutant_parent_only_instead_of_all_ancestors(monkeypatch):
    def parent_and_self(parent):
        m = len(parent)
        v = np.eye(m, dtype=bool)
        for i, p in enumerate(parent):
            if p >= 0:
                v[i, p] = True
        return v
    monkeypatch.setattr(ta, "ancestor_mask", parent_and_self)
    assert _attention_pins_fail(ta.tree_verify_attention) > 0


def test_mutant_wrong_scale():
    fn = lambda **p: tree_verify_attention(**p, softmax_scale=1.0 / 8)  # 1/d instead of 1/sqrt(d)  # noqa: E731
    assert _attention_pins_fail(fn) > 0


def test_mutant_wrong_gqa_mapping():
    def fn(**p):
        Hq = p["q"].shape[1]
        Hkv = p["num_kv_heads"]
        G = Hq // Hkv
        # interleaved mapping h -> h % Hkv, emulated by permuting the query heads
        perm = np.array([(h % Hkv) * G + h // Hkv for h in range(Hq)])
        inv = np.argsort(perm)
        q2 = p["q"][:, inv, :]
        out, lse = tree_verify_attention(**{**p, "q": q2})
        return out[:, perm, :], lse[:, perm]
    assert _attention_pins_fail(fn) > 0


def test_mutant_tree_k_v_swapped():
    fn = lambda **p: tree_verify_attention(**{**p, "tree_k": p["tree_v"], "tree_v": p["tree_k"]})  # noqa: E731
    assert _attention_pins_fail(fn) > 0


def test_mutant_prefix_dropped():
    def fn(**p):
        z = p["k_cache"][:0]
        out, lse = tree_verify_attention(**{**p, "k_cache": z, "v_cache": z,
                                           "cu_prefix": np.zeros_like(p["cu_prefix"])})
        return out, lse
    assert _attention_pins_fail(fn) > 0


def test_mutant_merge_without_reweighting():
    rng = np.random.default_rng(1)
    q, K, V = rng.standard_normal(8), rng.standard_normal((30, 8)), rng.standard_normal((30, 8))
    parts = [attention_partial(q, K[a:b], V[a:b], 0.35) for a, b in [(0, 11), (11, 30)]]
    o_ref, l_ref = attention_partial(q, K, V, 0.35)
    o, lse = merge_partials(np.stack([p[0] for p in parts]), np.array([p[1] for p in parts]))
    assert np.allclose(o, o_ref, rtol=1e-12)
    bad = sum(p[0] for p in parts) / 2   # plain average: the planted mistake
    assert not np.allclose(bad, o_ref, rtol=1e-6)


def _accept_pins_fail(fn):
    failed = 0
    try:
        _pins.check_accept_bruteforce(fn, np.random.default_rng(0), max_m=5, vocab=2, draws=2)
    except AssertionError:
        failed += 1
    ey = _pins.chain_expected_tokens_by_enumeration(fn, [0.85, 0.75, 0.60, 0.40])
    if abs(ey - 3.023) > 1e-12:
        failed += 1
    return failed


def test_real_acceptance_passes_pins():
    assert _accept_pins_fail(accept_longest_path) == 0


def _walk_variant(parent, draft, slot, cu, tie_later=False, own_slot=False, bonus_shift=1):
    """A copy of the oracle's walk (one sequence) with switchable planted mistakes."""
    m = len(parent)
    best, bd = -1, 0
    for i in range(m):
        j, ok, depth = i, True, 0
        while j >= 0:
            want = slot[j] if own_slot else slot[parent[j] + 1]
            ok &= bool(draft[j] == want)
            depth += 1
            j = int(parent[j])
        if ok and (depth > bd or (tie_later and depth == bd)):
            best, bd = i, depth
    path = np.full(m, -1, np.int32)
    if best >= 0:
        pth = _pins.path_to(parent, best)
        path[: len(pth)] = pth
    nxt = slot[best + bonus_shift] if best >= 0 else slot[0]
    return np.array([bd], np.int32), path, np.array([nxt], np.int32)


def test_walk_copy_without_mistakes_passes():
    assert _accept_pins_fail(_walk_variant) == 0


@pytest.mark.parametrize("mistake", [dict(tie_later=True), dict(own_slot=True), dict(bonus_shift=0)])
def test_acceptance_mutants_are_caught(mistake):
    assert _accept_pins_fail(lambda *a: _walk_variant(*a, **mistake)) > 0


# ----------------------------------------------------------------------------- KV commit
def _commit_pins_fail(fn):
    checks = [
        lambda: _pins.check_commit_causal(fn, tree_verify_attention, np.random.default_rng(21)),
        lambda: _pins.check_commit_touches_only_the_path_rows(fn, np.random.default_rng(22)),
        lambda: _pins.check_commit_empty_path_writes_nothing(fn, np.random.default_rng(23)),
        lambda: _pins.check_commit_full_chain(fn, np.random.default_rng(24)),
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except (AssertionError, IndexError, ValueError):
            failed += 1
    return failed


def _commit_mutant(src_of, dst_of, copy_v=True):
    """The oracle's loop with the source row, destination row or V copy altered."""
    def fn(k_cache, v_cache, tree_k, tree_v, cu_nodes, accept_len, accept_path, dst_row):
        k_out, v_out = np.array(k_cache, copy=True), np.array(v_cache, copy=True)
        for b in range(len(cu_nodes) - 1):
            n0, L = int(cu_nodes[b]), int(accept_len[b])
            for j in range(L):
                s = src_of(accept_path, n0, j, L)
                t = dst_of(dst_row, b, j)
                k_out[t] = tree_k[s]
                if copy_v:
                    v_out[t] = tree_v[s]
        return k_out, v_out
    return fn


def test_real_commit_oracle_passes_all_commit_pins():
    from oracle import commit_accepted_kv
    assert _commit_pins_fail(commit_accepted_kv) == 0


def test_commit_mutant_leaf_first():
    fn = _commit_mutant(lambda ap, n0, j, L: n0 + int(ap[n0 + L - 1 - j]), lambda d, b, j: int(d[b]) + j)
    assert _commit_pins_fail(fn) > 0


def test_commit_mutant_destination_off_by_one():
    fn = _commit_mutant(lambda ap, n0, j, L: n0 + int(ap[n0 + j]), lambda d, b, j: int(d[b]) + j + 1)
    assert _commit_pins_fail(fn) > 0


def test_commit_mutant_local_id_used_as_global_row():
    fn = _commit_mutant(lambda ap, n0, j, L: int(ap[n0 + j]), lambda d, b, j: int(d[b]) + j)
    assert _commit_pins_fail(fn) > 0


def test_commit_mutant_values_not_copied():
    fn = _commit_mutant(lambda ap, n0, j, L: n0 + int(ap[n0 + j]), lambda d, b, j: int(d[b]) + j, copy_v=False)
    assert _commit_pins_fail(fn) > 0


# ----------------------------------------------------------------- stochastic verification
def _sampling_pins_fail(fn):
    checks = [
        lambda: _pins.check_sampling_marginals(fn, np.random.default_rng(41), n=20000),
        lambda: _pins.check_sampling_forced_cases(fn, np.random.default_rng(42), n=1500),
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except (AssertionError, ValueError, IndexError):
            failed += 1
    return failed


def _sampling_mutant(accept=None, resid=None, bonus_row=0, stop=True):
    """The oracle's loop with one rule altered."""
    from oracle import quantised_draw

    def fn(p, q, draft_tok, u_accept, u_sample, cu_draft):
        p = np.asarray(p, np.float32); q = np.asarray(q, np.float32)
        B = len(cu_draft) - 1
        alen = np.zeros(B, np.int32); out = np.zeros(B, np.int32)
        for b in range(B):
            g0, gamma = int(cu_draft[b]), int(cu_draft[b + 1] - cu_draft[b])
            k, first_rej = 0, None
            for i in range(gamma):
                x = int(draft_tok[g0 + i]); px, qx = p[g0 + b + i, x], q[g0 + i, x]
                u = np.float32(u_accept[g0 + i])
                ok = accept(px, qx, u) if accept else (px >= qx or np.float32(u * qx) < px)
                if ok:
                    k += 1              # (past a rejection only when the mutant does not stop)
                else:
                    if first_rej is None:
                        first_rej = i
                    if stop:
                        break
            alen[b] = k
            j = first_rej if first_rej is not None else gamma
            prow = p[g0 + b + j]
            if first_rej is not None:
                w = resid(prow, q[g0 + j]) if resid else np.maximum(np.float32(0), prow - q[g0 + j])
                t = quantised_draw(np.maximum(w, 0), u_sample[b])
                out[b] = t if t >= 0 else quantised_draw(prow, u_sample[b])
            else:
                out[b] = quantised_draw(p[g0 + b + j - bonus_row], u_sample[b])
        return alen, out
    return fn


def test_real_sampling_oracle_passes_its_pins():
    from oracle import verify_chain_sampling
    assert _sampling_pins_fail(verify_chain_sampling) == 0
    assert _sampling_pins_fail(_sampling_mutant()) == 0      # the mutant frame itself is faithful


def test_sampling_mutant_accept_test_reversed():
    assert _sampling_pins_fail(_sampling_mutant(accept=lambda px, qx, u: np.float32(u * qx) > px)) > 0


def test_sampling_mutant_correction_from_p():
    assert _sampling_pins_fail(_sampling_mutant(resid=lambda pr, qr: pr)) > 0


def test_sampling_mutant_residual_reversed():
    assert _sampling_pins_fail(_sampling_mutant(resid=lambda pr, qr: np.maximum(0, qr - pr))) > 0


def test_sampling_mutant_bonus_from_the_last_draft_position():
    assert _sampling_pins_fail(_sampling_mutant(bonus_row=1)) > 0


def test_sampling_mutant_accepts_past_the_first_rejection():
    assert _sampling_pins_fail(_sampling_mutant(stop=False)) > 0


# ----------------------------------------------------------------------------- GDN trees
def _gdn_pins_fail(fn):
    checks = [
        lambda: _pins.check_gdn_triangular_solve(fn, np.random.default_rng(71), trials=3),
        lambda: _pins.check_gdn_no_write(fn, np.random.default_rng(72)),
        lambda: _pins.check_gdn_associative_recall(fn, np.random.default_rng(73)),
        lambda: [_pins.check_gdn_sibling_independence(fn, np.random.default_rng(74 + s)) for s in range(3)],
    ]
    failed = 0
    for c in checks:
        try:
            c()
        except AssertionError:
            failed += 1
    return failed


def _gdn_mutant(step, read_before=False, leaf_first=False):
    """The oracle's per-path recurrence with the update `step` (S, k, v, beta, alpha -> S)
    and optionally the read before the node's own write or the path reversed."""
    def fn(q, k, v, beta, alpha, S0, parent, cu_nodes):
        q = np.asarray(q, np.float64)
        N, H, _ = q.shape
        out = np.zeros((N, H, np.asarray(v).shape[2]))
        for b in range(len(cu_nodes) - 1):
            n0, n1 = int(cu_nodes[b]), int(cu_nodes[b + 1])
            for i in range(n1 - n0):
                path, j = [], i
                while j >= 0:
                    path.append(n0 + j)
                    j = int(parent[n0 + j])
                path = path if leaf_first else path[::-1]
                for h in range(H):
                    S = np.array(S0[b, h], np.float64)
                    for t, node in enumerate(path):
                        if read_before and node == n0 + i:
                            break
                        S = step(S, np.asarray(k[node, h], np.float64), np.asarray(v[node, h], np.float64),
                                 beta[node, h], alpha[node, h])
                    out[n0 + i, h] = S.T @ q[n0 + i, h]
        return out
    return fn


_GDN_STEP = lambda S, k, v, b, a: a * (S - b * np.outer(k, k @ S)) + b * np.outer(k, v)  # noqa: E731


def test_real_gdn_oracle_and_faithful_mutant_frame_pass():
    from oracle import gdn_tree_outputs
    assert _gdn_pins_fail(gdn_tree_outputs) == 0
    assert _gdn_pins_fail(_gdn_mutant(_GDN_STEP)) == 0


def test_gdn_mutant_decay_on_the_write():
    assert _gdn_pins_fail(_gdn_mutant(lambda S, k, v, b, a: a * (S - b * np.outer(k, k @ S) + b * np.outer(k, v)))) > 0


def test_gdn_mutant_read_before_write():
    assert _gdn_pins_fail(_gdn_mutant(_GDN_STEP, read_before=True)) > 0


def test_gdn_mutant_erase_without_beta():
    assert _gdn_pins_fail(_gdn_mutant(lambda S, k, v, b, a: a * (S - np.outer(k, k @ S)) + b * np.outer(k, v))) > 0


def test_gdn_mutant_leaf_first_path():
    assert _gdn_pins_fail(_gdn_mutant(_GDN_STEP, leaf_first=True)) > 0


def test_gdn_mutant_decay_ignored():
    assert _gdn_pins_fail(_gdn_mutant(lambda S, k, v, b, a: S - b * np.outer(k, k @ S) + b * np.outer(k, v))) > 0
