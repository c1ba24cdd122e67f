"""Independent checks ("pins") for the CPU oracle.

Each check compares an attention or acceptance function against something that does
not reuse its code: a library routine (``torch.nn.functional.
scaled_dot_product_attention`` and ``scipy.special.logsumexp`` on CPU, float64) applied
to an independently materialised sequence, a closed form, or an exhaustive
enumeration.  The checks take the function under test as an argument so that
``test_oracle_mutations.py`` can show each one fails on a planted mistake.
"""
from __future__ import annotations

import itertools

import numpy as np
import torch
import torch.nn.functional as F
from scipy.special import logsumexp


def all_parent_arrays(m: int):
    """Every topologically ordered parent array of m nodes: parent[i] in {-1..i-1}."""
    return itertools.product(*[range(-1, i) for i in range(m)])


def random_problem(rng, P, m, Hq=4, Hkv=2, d=8, parent=None):
    """Float64 inputs of one sequence (B = 1)."""
    q = rng.standard_normal((m, Hq, d))
    kc = rng.standard_normal((P, Hkv, d))
    vc = rng.standard_normal((P, Hkv, d))
    tk = rng.standard_normal((m, Hkv, d))
    tv = rng.standard_normal((m, Hkv, d))
    if parent is None:
        parent = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, m)], dtype=np.int32)
    return dict(q=q, k_cache=kc, v_cache=vc, tree_k=tk, tree_v=tv,
                parent=np.asarray(parent, dtype=np.int32),
                cu_prefix=np.array([0, P], dtype=np.int32),
                cu_nodes=np.array([0, m], dtype=np.int32), num_kv_heads=Hkv)


def path_to(parent, i):
    """Node ids on the path root -> i (inclusive)."""
    path = []
    while i >= 0:
        path.append(i)
        i = int(parent[i])
    return path[::-1]


def causal_last_row(prob, i):
    """Causal attention at the last position of the materialised sequence
    prefix ++ path(root -> i), every query head; returns (o [Hq, d], lse [Hq]).

    The sequence is built explicitly; attention is the library's causal SDPA on it,
    with KV heads expanded in contiguous groups (head h reads KV head h // G)."""
    parent = prob["parent"]
    path = path_to(parent, i)
    Kseq = np.concatenate([prob["k_cache"], prob["tree_k"][path]], axis=0)   # [L, Hkv, d]
    Vseq = np.concatenate([prob["v_cache"], prob["tree_v"][path]], axis=0)
    L, Hkv, d = Kseq.shape
    Hq = prob["q"].shape[1]
    G = Hq // Hkv
    # queries: filler rows for earlier positions, the node's own query last
    rng = np.random.default_rng(7)
    Qseq = rng.standard_normal((L, Hq, d))
    Qseq[-1] = prob["q"][i]
    qt = torch.from_numpy(Qseq).permute(1, 0, 2)                          # [Hq, L, d]
    kt = torch.from_numpy(Kseq).permute(1, 0, 2).repeat_interleave(G, dim=0)
    vt = torch.from_numpy(Vseq).permute(1, 0, 2).repeat_interleave(G, dim=0)
    o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True)       # [Hq, L, d]
    logits = (qt[:, -1:, :] @ kt.transpose(1, 2))[:, 0, :].numpy() / np.sqrt(d)
    lse = logsumexp(logits, axis=1)
    return o[:, -1, :].numpy(), lse


def check_path_bruteforce(attn_fn, prob, rtol=1e-11, atol=1e-11):
    """Every node's output/LSE equals causal attention over prefix ++ its path."""
    out, lse = attn_fn(**prob)
    for i in range(prob["q"].shape[0]):
        o_ref, l_ref = causal_last_row(prob, i)
        np.testing.assert_allclose(out[i], o_ref, rtol=rtol, atol=atol)
        np.testing.assert_allclose(lse[i], l_ref, rtol=rtol, atol=atol)


def check_chain_is_causal(attn_fn, rng, P=13, m=7, Hq=4, Hkv=2, d=8):
    """A chain tree is ordinary causal attention over prefix ++ chain (one SDPA call)."""
    prob = random_problem(rng, P, m, Hq, Hkv, d, parent=np.arange(-1, m - 1))
    out, lse = attn_fn(**prob)
    G = Hq // Hkv
    K = np.concatenate([prob["k_cache"], prob["tree_k"]], 0)
    V = np.concatenate([prob["v_cache"], prob["tree_v"]], 0)
    Q = np.concatenate([np.zeros((P, Hq, d)), prob["q"]], 0)
    qt = torch.from_numpy(Q).permute(1, 0, 2)
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
    o = F.scaled_dot_product_attention(qt, kt, vt, is_causal=True)[:, P:, :].permute(1, 0, 2).numpy()
    np.testing.assert_allclose(out, o, rtol=1e-11, atol=1e-11)
    logits = (qt @ kt.transpose(1, 2)).numpy() / np.sqrt(d)               # [Hq, L, L]
    Ltot = P + m
    causal = np.tril(np.ones((Ltot, Ltot), dtype=bool))
    lref = logsumexp(np.where(causal[None], logits, -np.inf), axis=2)[:, P:].T
    np.testing.assert_allclose(lse, lref, rtol=1e-11, atol=1e-11)


def check_single_node_is_decode(attn_fn, rng, P=29, Hq=4, Hkv=2, d=8):
    """m = 1: plain decode attention over prefix ++ the node's own key."""
    prob = random_problem(rng, P, 1, Hq, Hkv, d, parent=[-1])
    out, lse = attn_fn(**prob)
    G = Hq // Hkv
    K = np.concatenate([prob["k_cache"], prob["tree_k"]], 0)
    V = np.concatenate([prob["v_cache"], prob["tree_v"]], 0)
    qt = torch.from_numpy(prob["q"]).permute(1, 0, 2)                    # [Hq, 1, d]
    kt = torch.from_numpy(K).permute(1, 0, 2).repeat_interleave(G, 0)
    vt = torch.from_numpy(V).permute(1, 0, 2).repeat_interleave(G, 0)
    o = F.scaled_dot_product_attention(qt, kt, vt)[:, 0, :].numpy()
    np.testing.assert_allclose(out[0], o, rtol=1e-11, atol=1e-11)


def check_uniform_closed_form(attn_fn, rng, P=9, Hq=2, Hkv=1, d=4):
    """All keys equal => softmax uniform over the visible keys:
    out = mean of the visible values and lse = z + log(#visible)."""
    m = 5
    parent = np.array([-1, 0, 1, 0, -1], dtype=np.int32)   # depths 1,2,3,2,1
    prob = random_problem(rng, P, m, Hq, Hkv, d, parent=parent)
    key = rng.standard_normal(d)
    prob["k_cache"][:] = key
    prob["tree_k"][:] = key
    out, lse = attn_fn(**prob)
    for i in range(m):
        path = path_to(parent, i)
        vis_v = np.concatenate([prob["v_cache"][:, 0], prob["tree_v"][path, 0]], 0)
        for h in range(Hq):
            z = prob["q"][i, h] @ key / np.sqrt(d)
            np.testing.assert_allclose(out[i, h], vis_v.mean(0), rtol=1e-12, atol=1e-12)
            np.testing.assert_allclose(lse[i, h], z + np.log(P + len(path)), rtol=1e-12, atol=1e-12)


def check_sibling_independence(attn_fn, rng, P=5):
    """Changing node j's key/value moves exactly the nodes that have j on their path."""
    parent = np.array([-1, 0, 0, 1, 2, -1, 5], dtype=np.int32)
    prob = random_problem(rng, P, len(parent), parent=parent)
    out0, lse0 = attn_fn(**prob)
    for j in range(len(parent)):
        p2 = {k: (v.copy() if isinstance(v, np.ndarray) else v) for k, v in prob.items()}
        p2["tree_k"][j] += 1.0
        p2["tree_v"][j] -= 1.0
        out1, lse1 = attn_fn(**p2)
        for i in range(len(parent)):
            sees = j in path_to(parent, i)
            same = np.array_equal(out0[i], out1[i]) and np.array_equal(lse0[i], lse1[i])
            assert same != sees, (i, j, sees)


def check_relabeling(attn_fn, rng, P=6):
    """Two topological orders of one tree give the same per-node results."""
    parent = np.array([-1, 0, 0, 1, 1, 2, -1], dtype=np.int32)
    prob = random_problem(rng, P, len(parent), parent=parent)
    out, lse = attn_fn(**prob)
    perm = np.array([6, 0, 2, 5, 1, 4, 3])           # new position -> old id, parents first
    inv = np.empty_like(perm)
    inv[perm] = np.arange(len(perm))
    new_parent = np.array([-1 if parent[o] < 0 else inv[parent[o]] for o in perm], dtype=np.int32)
    assert all(new_parent[i] < i for i in range(len(perm)))
    p2 = dict(prob)
    for k in ("q", "tree_k", "tree_v"):
        p2[k] = prob[k][perm]
    p2["parent"] = new_parent
    out2, lse2 = attn_fn(**p2)
    np.testing.assert_allclose(out2, out[perm], rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(lse2, lse[perm], rtol=1e-12, atol=1e-13)


# ------------------------------------------------------------------ acceptance pins

def forward_greedy_path_check(parent, draft, slot, i):
    """Is the root -> i path accepted?  Walk it forwards the way a decoder would: the
    target's greedy token at the prefix end is slot[0]; after accepting node u the next
    greedy token is slot[u + 1]."""
    expect = slot[0]
    for u in path_to(parent, i):
        if draft[u] != expect:
            return False
        expect = slot[u + 1]
    return True


def bruteforce_accept(parent, draft, slot):
    """Longest accepted path by enumerating every root -> node path; ties -> smaller id."""
    m = len(parent)
    best = None
    for i in range(m):
        if forward_greedy_path_check(parent, draft, slot, i):
            path = path_to(parent, i)
            if best is None or len(path) > len(best[1]):
                best = (i, path)
    if best is None:
        return 0, [], int(slot[0])
    return len(best[1]), best[1], int(slot[best[0] + 1])


def check_accept_bruteforce(accept_fn, rng, max_m=6, vocab=2, draws=2):
    for m in range(1, max_m + 1):
        for parent in all_parent_arrays(m):
            parent = np.asarray(parent, dtype=np.int32)
            for _ in range(draws):
                slot = rng.integers(0, vocab, m + 1).astype(np.int32)
                draft = rng.integers(0, vocab, m).astype(np.int32)
                alen, apath, nxt = accept_fn(parent, draft, slot, np.array([0, m], np.int32))
                L, path, tok = bruteforce_accept(parent, draft, slot)
                assert int(alen[0]) == L, (parent, draft, slot)
                assert list(apath[:L]) == path
                assert all(apath[L:] == -1)
                assert int(nxt[0]) == tok


def chain_expected_tokens_by_enumeration(accept_fn, conditional):
    """Sum over all 2^gamma match patterns of Pr(pattern) * (accept_len + 1) on a chain.

    Position k matches independently with probability conditional[k]; only the
    matched prefix matters to the walk, so Pr(accept_len >= k) is the running product
    of the conditional probabilities, i.e. the page's survival value s_k."""
    gamma = len(conditional)
    parent = np.arange(-1, gamma - 1, dtype=np.int32)
    slot = np.arange(100, 100 + gamma + 1, dtype=np.int32)
    total = 0.0
    for bits in itertools.product([0, 1], repeat=gamma):
        pr = 1.0
        for c, b in zip(conditional, bits):
            pr *= c if b else (1.0 - c)
        draft = np.array([slot[parent[k] + 1] if bits[k] else -5 for k in range(gamma)], np.int32)
        alen, _, _ = accept_fn(parent, draft, slot, np.array([0, gamma], np.int32))
        total += pr * (int(alen[0]) + 1)
    return total


# ----------------------------------------------------------------------------- KV commit
def commit_problem(rng, B=3, Hq=4, Hkv=2, d=8, max_m=7, room=9):
    """A batch of random trees plus a cache in which sequence b owns rows
    [base_b, base_b + P_b + room): its prefix, then reserved room filled with junk.
    One node per sequence is picked and its root->node path (from the parent array)
    is the path to commit; dst_row[b] = base_b + P_b."""
    Ps = [int(rng.integers(0, 12)) for _ in range(B)]
    ms = [int(rng.integers(1, max_m + 1)) for _ in range(B)]
    parents, paths = [], []
    for m in ms:
        par = np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, m)], dtype=np.int32)
        parents.append(par)
        paths.append(path_to(par, int(rng.integers(0, m))))
    N = sum(ms)
    cu_nodes = np.concatenate([[0], np.cumsum(ms)]).astype(np.int32)
    cu_prefix = np.concatenate([[0], np.cumsum(Ps)]).astype(np.int32)
    kc = rng.standard_normal((int(cu_prefix[-1]), Hkv, d))
    vc = rng.standard_normal((int(cu_prefix[-1]), Hkv, d))
    base = np.concatenate([[0], np.cumsum([P + room for P in Ps])]).astype(np.int64)
    k_res = rng.standard_normal((int(base[-1]), Hkv, d))     # junk in the reserved room
    v_res = rng.standard_normal((int(base[-1]), Hkv, d))
    for b in range(B):
        k_res[base[b]:base[b] + Ps[b]] = kc[cu_prefix[b]:cu_prefix[b + 1]]
        v_res[base[b]:base[b] + Ps[b]] = vc[cu_prefix[b]:cu_prefix[b + 1]]
    accept_len = np.array([len(p) for p in paths], dtype=np.int32)
    accept_path = np.full(N, -1, dtype=np.int32)
    for b, p in enumerate(paths):
        accept_path[cu_nodes[b]:cu_nodes[b] + len(p)] = p
    return dict(q=rng.standard_normal((N, Hq, d)), k_cache=kc, v_cache=vc,
                tree_k=rng.standard_normal((N, Hkv, d)), tree_v=rng.standard_normal((N, Hkv, d)),
                parent=np.concatenate(parents).astype(np.int32), cu_prefix=cu_prefix, cu_nodes=cu_nodes,
                num_kv_heads=Hkv, k_res=k_res, v_res=v_res, base=base, Ps=Ps,
                accept_len=accept_len, accept_path=accept_path,
                dst_row=(base[:-1] + np.array(Ps)).astype(np.int32))


def _commit(commit_fn, pr):
    return commit_fn(pr["k_res"], pr["v_res"], pr["tree_k"], pr["tree_v"], pr["cu_nodes"],
                     pr["accept_len"], pr["accept_path"], pr["dst_row"])


def check_commit_causal(commit_fn, attn_fn, rng, trials=6):
    """After committing the path root -> i, causal attention at every position of the
    new sequence (prefix ++ committed rows) equals tree attention for the path node
    there: tree attention lets a node see the prefix, its ancestors and itself, and the
    committed sequence is exactly that, in order."""
    for _ in range(trials):
        pr = commit_problem(rng)
        out_t, _ = attn_fn(**{k: pr[k] for k in ("q", "k_cache", "v_cache", "tree_k", "tree_v", "parent",
                                                 "cu_prefix", "cu_nodes", "num_kv_heads")})
        k_new, v_new = _commit(commit_fn, pr)
        Hq, Hkv = pr["q"].shape[1], pr["num_kv_heads"]
        G = Hq // Hkv
        for b in range(len(pr["Ps"])):
            n0, L = int(pr["cu_nodes"][b]), int(pr["accept_len"][b])
            rows = slice(int(pr["base"][b]), int(pr["dst_row"][b]) + L)
            K = torch.from_numpy(k_new[rows]).permute(1, 0, 2).repeat_interleave(G, 0)   # [Hq, S, d]
            V = torch.from_numpy(v_new[rows]).permute(1, 0, 2).repeat_interleave(G, 0)
            S = K.shape[1]
            for j in range(L):
                node = n0 + int(pr["accept_path"][n0 + j])
                pos = S - L + j                              # the node's position
                qt = torch.from_numpy(pr["q"][node])[:, None, :]
                o = F.scaled_dot_product_attention(qt, K[:, :pos + 1], V[:, :pos + 1])[:, 0].numpy()
                np.testing.assert_allclose(o, out_t[node], rtol=1e-11, atol=1e-11)


def check_commit_touches_only_the_path_rows(commit_fn, rng, trials=4):
    for _ in range(trials):
        pr = commit_problem(rng)
        k_new, v_new = _commit(commit_fn, pr)
        keep = np.ones(len(k_new), dtype=bool)
        for b in range(len(pr["Ps"])):
            keep[int(pr["dst_row"][b]):int(pr["dst_row"][b]) + int(pr["accept_len"][b])] = False
        np.testing.assert_array_equal(k_new[keep], pr["k_res"][keep])
        np.testing.assert_array_equal(v_new[keep], pr["v_res"][keep])


def check_commit_empty_path_writes_nothing(commit_fn, rng):
    pr = commit_problem(rng)
    pr["accept_len"][:] = 0
    pr["accept_path"][:] = -1
    k_new, v_new = _commit(commit_fn, pr)
    np.testing.assert_array_equal(k_new, pr["k_res"])
    np.testing.assert_array_equal(v_new, pr["v_res"])


def check_commit_full_chain(commit_fn, rng, m=6):
    """A chain accepted to its end commits the tree rows themselves, in order."""
    pr = commit_problem(rng, B=1, max_m=1)
    N = m
    pr["tree_k"] = rng.standard_normal((N, pr["num_kv_heads"], pr["k_res"].shape[2]))
    pr["tree_v"] = rng.standard_normal((N, pr["num_kv_heads"], pr["k_res"].shape[2]))
    pr["cu_nodes"] = np.array([0, m], dtype=np.int32)
    pr["accept_len"] = np.array([m], dtype=np.int32)
    pr["accept_path"] = np.arange(m, dtype=np.int32)
    k_new, v_new = _commit(commit_fn, pr)
    d0 = int(pr["dst_row"][0])
    np.testing.assert_array_equal(k_new[d0:d0 + m], pr["tree_k"])
    np.testing.assert_array_equal(v_new[d0:d0 + m], pr["tree_v"])


# ----------------------------------------------------------------- stochastic verification
def sampling_case(kind, V=6, rng=None):
    """(p, q) float32 rows of one position for the Faster decoding test list: p == q,
    partially overlapping supports, disjoint supports."""
    rng = rng or np.random.default_rng(0)
    if kind == "equal":
        p = rng.random(V) + 0.05
        q = p.copy()
    elif kind == "partial":
        p = rng.random(V) + 0.05
        q = rng.random(V) + 0.05
        p[: V // 3] = 0.0          # q has mass where p has none, and vice versa
        q[-(V // 3):] = 0.0
    elif kind == "disjoint":
        p = np.zeros(V)
        q = np.zeros(V)
        p[: V // 2] = rng.random(V // 2) + 0.05
        q[V // 2:] = rng.random(V - V // 2) + 0.05
    else:
        raise ValueError(kind)
    p = (p / p.sum()).astype(np.float32)
    q = (q / q.sum()).astype(np.float32)
    return p, q


def draw_chain(rng, ps, qs, n):
    """n independent rounds of one chain: ps [gamma+1, V], qs [gamma, V] (the same for
    every round).  Draft tokens X_i ~ q_i, uniforms in [0, 1) float32."""
    gamma, V = qs.shape
    w = qs.astype(np.float64)
    w /= w.sum(1, keepdims=True)
    draft = np.stack([rng.choice(V, size=n, p=w[i]) for i in range(gamma)], 1)
    p = np.tile(ps, (n, 1))
    q = np.tile(qs, (n, 1))
    u_acc = rng.random((n, gamma)).astype(np.float32)
    u_smp = rng.random(n).astype(np.float32)
    cu = np.arange(0, (n + 1) * gamma, gamma, dtype=np.int32)
    return p, q, draft.reshape(-1).astype(np.int32), u_acc.reshape(-1), u_smp, cu


def emitted(draft, accept_len, out_token, gamma):
    """Tokens emitted by each round: the accepted drafts, then the correction / bonus."""
    d = draft.reshape(-1, gamma)
    return [list(d[r, :accept_len[r]]) + [int(out_token[r])] for r in range(len(accept_len))]


def assert_freq(tokens, p, what):
    """Empirical frequencies within 5 standard errors of p (plus 1e-3)."""
    tokens = np.asarray(tokens)
    n = len(tokens)
    assert n > 500, (what, n)
    f = np.bincount(tokens, minlength=len(p)) / n
    se = np.sqrt(np.maximum(p * (1 - p), 1e-12) / n)
    bad = np.abs(f - p) > 5 * se + 1e-3
    assert not bad.any(), (what, f, p)


def check_sampling_marginals(verify_fn, rng, n=40000):
    """gamma = 2, three positions with different (p, q): the first emitted token ~ p_1;
    given the first draft was accepted, the second ~ p_2; given both were accepted, the
    bonus ~ p_3 - for p == q, partial overlap and disjoint supports."""
    for kind in ("equal", "partial", "disjoint"):
        rows = [sampling_case(kind, rng=np.random.default_rng(s)) for s in (1, 2)]
        ps = np.stack([rows[0][0], rows[1][0], sampling_case("equal", rng=np.random.default_rng(3))[0]])
        qs = np.stack([rows[0][1], rows[1][1]])
        p, q, draft, ua, us, cu = draw_chain(rng, ps, qs, n)
        alen, out = verify_fn(p, q, draft, ua, us, cu)
        em = emitted(draft, alen, out, 2)
        assert_freq([e[0] for e in em], ps[0].astype(np.float64), (kind, "token 1"))
        if kind != "disjoint":
            assert_freq([e[1] for e in em if len(e) > 1], ps[1].astype(np.float64), (kind, "token 2"))
        if kind == "equal":
            assert_freq([e[2] for e in em if len(e) > 2], ps[2].astype(np.float64), (kind, "bonus"))


def check_sampling_forced_cases(verify_fn, rng, n=3000):
    """Forced first rejection, late rejection and all-accept (Faster decoding, test list)."""
    V, gamma = 6, 4
    same, _ = sampling_case("equal", V, np.random.default_rng(4))
    dp, dq = sampling_case("disjoint", V, np.random.default_rng(5))
    for k in range(gamma + 1):        # positions < k have p == q, position k disjoint supports
        ps = np.stack([same] * k + [dp] * (gamma - k) + [same]).astype(np.float32)
        qs = np.stack([same] * k + [dq] * (gamma - k)).astype(np.float32)
        p, q, draft, ua, us, cu = draw_chain(rng, ps, qs, n)
        alen, out = verify_fn(p, q, draft, ua, us, cu)
        assert (alen == k).all(), (k, np.bincount(alen))
        # the correction comes from the residual, here p itself (disjoint supports)
        assert_freq(out, (dp if k < gamma else same).astype(np.float64), ("forced", k))


def check_quantised_draw_against_searchsorted(draw_fn, rng, trials=300):
    """Away from the cumulative boundaries the quantised draw is the plain inverse CDF."""
    for _ in range(trials):
        V = int(rng.integers(1, 40))
        w = rng.random(V).astype(np.float32)
        w[rng.random(V) < 0.3] = 0
        if w.sum() == 0:
            w[0] = 1
        u = np.float32(rng.random())
        c = np.cumsum(w.astype(np.float64))
        t = np.float64(u) * c[-1]
        if np.min(np.abs(c - t)) < 1e-6 * c[-1]:
            continue
        assert draw_fn(w, u) == int(np.searchsorted(c, t, side="right"))


# ----------------------------------------------------------------------------- GDN trees
def gdn_case(rng, B=2, H=2, d=6, max_m=9, beta_zero=False):
    par = [np.array([-1] + [int(rng.integers(-1, i)) for i in range(1, m)], np.int32)
           for m in [int(rng.integers(1, max_m + 1)) for _ in range(B)]]
    N = sum(len(p) for p in par)
    unit = lambda x: x / np.linalg.norm(x, axis=-1, keepdims=True)  # noqa: E731
    c = dict(q=unit(rng.standard_normal((N, H, d))), k=unit(rng.standard_normal((N, H, d))),
             v=rng.standard_normal((N, H, d)), beta=rng.random((N, H)) if not beta_zero else np.zeros((N, H)),
             alpha=0.5 + 0.5 * rng.random((N, H)), S0=rng.standard_normal((B, H, d, d)) * 0.3,
             parent=np.concatenate(par).astype(np.int32),
             cu_nodes=np.concatenate([[0], np.cumsum([len(p) for p in par])]).astype(np.int32))
    return c


def gdn_by_triangular_solve(c):
    """The page's form: per sequence and head, with gamma_i the product of alpha over
    node i's path, X_ij = beta_i (gamma_i / gamma_j) k_i . k_j for proper ancestors j,
    (I + X) W = beta (V - Gamma K S0) solved by numpy.linalg.solve, and
    o_i = gamma_i S0^T q_i + sum_{j anc-or-self of i} (gamma_i / gamma_j) (k_j . q_i) W_j."""
    q, k, v, beta, alpha, S0 = (np.asarray(c[n], np.float64) for n in ("q", "k", "v", "beta", "alpha", "S0"))
    N, H, _ = q.shape
    out = np.zeros((N, H, v.shape[2]))
    cu = c["cu_nodes"]
    for b in range(len(cu) - 1):
        n0, n1 = int(cu[b]), int(cu[b + 1])
        m = n1 - n0
        par = c["parent"][n0:n1]
        anc = np.zeros((m, m), bool)        # anc[i, j]: j is i or an ancestor of i
        for i in range(m):
            j = i
            while j >= 0:
                anc[i, j] = True
                j = int(par[j])
        proper = anc & ~np.eye(m, dtype=bool)
        for h in range(H):
            a = alpha[n0:n1, h]
            g = np.array([np.prod(a[anc[i]]) for i in range(m)])
            K, Q, V, bt = k[n0:n1, h], q[n0:n1, h], v[n0:n1, h], beta[n0:n1, h]
            ratio = g[:, None] / g[None, :]
            X = np.where(proper, bt[:, None] * ratio * (K @ K.T), 0.0)
            W = np.linalg.solve(np.eye(m) + X, bt[:, None] * (V - g[:, None] * (K @ S0[b, h])))
            Y = np.where(anc, ratio * (Q @ K.T), 0.0)
            out[n0:n1, h] = g[:, None] * (Q @ S0[b, h]) + Y @ W
    return out


def check_gdn_triangular_solve(fn, rng, trials=8):
    for _ in range(trials):
        c = gdn_case(rng)
        np.testing.assert_allclose(fn(**c), gdn_by_triangular_solve(c), rtol=1e-10, atol=1e-10)


def check_gdn_no_write(fn, rng):
    """beta = 0: the state only decays, o_i = gamma_i S0^T q_i."""
    c = gdn_case(rng, beta_zero=True)
    out = fn(**c)
    cu = c["cu_nodes"]
    for b in range(len(cu) - 1):
        n0, n1 = int(cu[b]), int(cu[b + 1])
        for i in range(n1 - n0):
            j, g = i, np.ones(c["q"].shape[1])
            while j >= 0:
                g = g * c["alpha"][n0 + j]
                j = int(c["parent"][n0 + j])
            for h in range(c["q"].shape[1]):
                np.testing.assert_allclose(out[n0 + i, h], g[h] * (c["S0"][b, h].T @ c["q"][n0 + i, h]),
                                           rtol=1e-12, atol=1e-12)


def check_gdn_associative_recall(fn, rng, d=8, m=6):
    """alpha = 1, beta = 1 and orthonormal keys: writing k_j stores v_j in place of
    whatever S0 held at k_j, so reading with q = k_j returns v_j when j is on the
    node's path (itself included) and S0^T k_j otherwise."""
    par = np.array([-1, 0, 1, 0, 3, -1], np.int32)
    Qm, _ = np.linalg.qr(rng.standard_normal((d, d)))
    K = Qm[:m]                                    # orthonormal rows
    c = dict(k=K[:, None, :], v=rng.standard_normal((m, 1, d)), beta=np.ones((m, 1)), alpha=np.ones((m, 1)),
             S0=rng.standard_normal((1, 1, d, d)), parent=par, cu_nodes=np.array([0, m], np.int32))
    for target in range(m):
        c["q"] = np.repeat(K[target][None, None, :], m, 0)
        out = fn(**c)
        for i in range(m):
            j, on_path = i, False
            while j >= 0:
                on_path |= j == target
                j = int(par[j])
            expect = c["v"][target, 0] if on_path else c["S0"][0, 0].T @ K[target]
            np.testing.assert_allclose(out[i, 0], expect, rtol=1e-10, atol=1e-10)


def check_gdn_sibling_independence(fn, rng):
    c = gdn_case(rng, B=1, max_m=9)
    m = len(c["parent"])
    if m < 3:
        return
    out = fn(**c)
    j = int(rng.integers(1, m))
    c2 = {n: np.array(x, copy=True) for n, x in c.items()}
    c2["k"][j] = -c2["k"][j]
    c2["v"][j] += 1.0
    out2 = fn(**c2)
    for i in range(m):
        a, desc = i, False
        while a >= 0:
            desc |= a == j
            a = int(c["parent"][a])
        if not desc:
            np.testing.assert_array_equal(out2[i], out[i])
        else:
            assert np.abs(out2[i] - out[i]).max() > 1e-9
