"""Tree-verification attention, written out as its plain definition in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring): never called by the library.

Definition followed
-------------------
LongSpec, "Fast Tree Attention" section (Hybrid Tree Attention, "Split key-value
pairs"): every query of a speculative tree attends to the cached key/value pairs
{K_cache, V_cache} without any mask, and to the speculative pairs {K_specs, V_specs}
under the tree mask.  "Faster decoding" (aaai.latere.ai), section "Chains and trees
consume work differently": in one target pass each tree node may only attend to its
own ancestors.  LongSpec appendix "Correctness of attention aggregation": the result
is one scaled-dot-product attention of a query q over the stacked keys
K_merge = (K_cache ; K_specs) and values V_merge, with logits q K_merge^T / sqrt(d_qk),
and LSE = log sum_j exp(Z^(j)).

This oracle computes exactly that single softmax; it never splits the keys.

Readings taken where the pages are silent
-----------------------------------------
* A node sees itself as well as its proper ancestors (a node's own key is that of its
  own token; with a chain this is ordinary causal attention).
* Grouped-query heads: query head h reads KV head h // (Hq / Hkv).
* ``parent`` holds local ids; -1 marks a child of the prefix end; ``parent[i] < i``
  (nodes in topological order).  Anything else is rejected with ``ValueError``.
* An empty prefix contributes nothing; a row is never empty because the node sees
  itself.
* LSE is the natural logarithm over the *scaled* logits.
"""
from __future__ import annotations

import numpy as np

__all__ = ["ancestor_mask", "tree_verify_attention", "tree_verify_attention_rows"]


def _check_tree(parent_local: np.ndarray) -> None:
    for i, p in enumerate(np.asarray(parent_local)):
        if not (-1 <= int(p) < i):
            raise ValueError(f"parent[{i}] = {int(p)} is not in [-1, {i})")


def ancestor_mask(parent_local: np.ndarray) -> np.ndarray:
    """vis[i, j] is True iff tree node j is node i or one of its ancestors.

    Built by walking ``parent`` from each node up to the prefix end."""
    parent_local = np.asarray(parent_local)
    _check_tree(parent_local)
    m = len(parent_local)
    vis = np.zeros((m, m), dtype=bool)
    for i in range(m):
        j = i
        while j >= 0:
            vis[i, j] = True
            j = int(parent_local[j])
    return vis


def _default_scale(d: int, softmax_scale) -> float:
    return (1.0 / np.sqrt(d)) if softmax_scale is None else float(softmax_scale)


def tree_verify_attention(q, k_cache, v_cache, cu_prefix, tree_k, tree_v, parent,
                          cu_nodes, num_kv_heads: int, softmax_scale=None):
    """out[n, h, :] and lse[n, h] for every tree node n and query head h.

    Shapes: q [N, Hq, d]; k_cache, v_cache [sum P_b, Hkv, d]; tree_k, tree_v
    [N, Hkv, d]; parent [N] (local ids); cu_prefix, cu_nodes [B + 1].
    All floating inputs are converted to float64 first.
    """
    q = np.asarray(q, dtype=np.float64)
    k_cache = np.asarray(k_cache, dtype=np.float64)
    v_cache = np.asarray(v_cache, dtype=np.float64)
    tree_k = np.asarray(tree_k, dtype=np.float64)
    tree_v = np.asarray(tree_v, dtype=np.float64)
    N, Hq, d = q.shape
    Hkv = int(num_kv_heads)
    G = Hq // Hkv
    scale = _default_scale(d, softmax_scale)
    out = np.zeros((N, Hq, d), dtype=np.float64)
    lse = np.zeros((N, Hq), dtype=np.float64)
    B = len(cu_prefix) - 1
    for b in range(B):
        p0, p1 = int(cu_prefix[b]), int(cu_prefix[b + 1])
        n0, n1 = int(cu_nodes[b]), int(cu_nodes[b + 1])
        m, P = n1 - n0, p1 - p0
        if m == 0:
            continue
        vis_tree = ancestor_mask(parent[n0:n1])                # [m, m]
        # Full visibility row over the concatenated keys: prefix always visible.
        visible = np.concatenate([np.ones((m, P), dtype=bool), vis_tree], axis=1)
        visible = np.repeat(visible, G, axis=0)                 # rows ordered (node, head-in-group)
        for g in range(Hkv):
            K = np.concatenate([k_cache[p0:p1, g, :], tree_k[n0:n1, g, :]], axis=0)
            V = np.concatenate([v_cache[p0:p1, g, :], tree_v[n0:n1, g, :]], axis=0)
            Qg = q[n0:n1, g * G:(g + 1) * G, :].reshape(m * G, d)
            Z = scale * (Qg @ K.T)                              # [m*G, P+m]
            Z = np.where(visible, Z, -np.inf)
            zmax = Z.max(axis=1, keepdims=True)
            L = zmax[:, 0] + np.log(np.exp(Z - zmax).sum(axis=1))
            O = np.exp(Z - L[:, None]) @ V
            out[n0:n1, g * G:(g + 1) * G, :] = O.reshape(m, G, d)
            lse[n0:n1, g * G:(g + 1) * G] = L.reshape(m, G)
    return out, lse


def tree_verify_attention_rows(rows, q, k_cache, v_cache, cu_prefix, tree_k, tree_v,
                               parent, cu_nodes, num_kv_heads: int, softmax_scale=None):
    """The same definition evaluated one (node n, query head h) row at a time.

    ``rows`` is a sequence of (n, h) pairs with n a global node index.  Returns
    (out [len(rows), d], lse [len(rows)]).  Used where the full problem is too large
    to materialise on the host."""
    q = np.asarray(q)
    N, Hq, d = q.shape
    Hkv = int(num_kv_heads)
    G = Hq // Hkv
    scale = _default_scale(d, softmax_scale)
    cu_nodes = np.asarray(cu_nodes)
    outs = np.zeros((len(rows), d), dtype=np.float64)
    lses = np.zeros(len(rows), dtype=np.float64)
    for r, (n, h) in enumerate(rows):
        n, h = int(n), int(h)
        b = int(np.searchsorted(cu_nodes, n, side="right") - 1)
        p0, p1 = int(cu_prefix[b]), int(cu_prefix[b + 1])
        n0, n1 = int(cu_nodes[b]), int(cu_nodes[b + 1])
        i = n - n0
        par = np.asarray(parent[n0:n1])
        _check_tree(par)
        anc = []
        j = i
        while j >= 0:
            anc.append(j)
            j = int(par[j])
        anc = sorted(anc)
        g = h // G
        K = np.concatenate([np.asarray(k_cache[p0:p1, g, :], dtype=np.float64),
                            np.asarray(tree_k[n0:n1, g, :], dtype=np.float64)[anc]], axis=0)
        V = np.concatenate([np.asarray(v_cache[p0:p1, g, :], dtype=np.float64),
                            np.asarray(tree_v[n0:n1, g, :], dtype=np.float64)[anc]], axis=0)
        z = scale * (K @ np.asarray(q[n, h, :], dtype=np.float64))
        zmax = z.max()
        L = zmax + np.log(np.exp(z - zmax).sum())
        outs[r] = np.exp(z - L) @ V
        lses[r] = L
    return outs, lses
