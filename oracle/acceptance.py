"""Greedy verification of a draft tree: the longest accepted root-to-node path.

TEST INFRASTRUCTURE ONLY (see the package docstring): never called by the library.

"Faster decoding" (aaai.latere.ai), section "Modified rejection sampling keeps the
target distribution", closing paragraph on greedy verification: the deterministic
contract accepts the longest draft prefix that agrees with the target model's greedy
tokens and then emits the target's own token at the first disagreement (or, when
everything is accepted, the bonus token after the last accepted one).  Section
"Chains and trees consume work differently": with a tree the candidates are the
root-to-node paths, each node conditioned on its ancestors only.

Readings taken where the pages are silent
-----------------------------------------
* Slots of ``target_argmax``: sequence b owns m_b + 1 slots starting at
  ``cu_nodes[b] + b``; slot 0 is the target's greedy token at the prefix end and slot
  i + 1 the token after node i.  Node i is *matched* when
  ``draft_tok[i] == slot[parent[i] + 1]``.
* Node i is *accepted* when it and all of its ancestors are matched.
* The answer is the deepest accepted node; equally deep candidates are broken towards
  the smallest node index.  No accepted node gives an empty path.
* ``next_token`` is ``slot[last + 1]`` (``slot[0]`` for an empty path), so a cycle
  emits ``accept_len + 1`` tokens.
* ``accept_path`` holds, per sequence, the accepted local node ids root first, then
  -1 up to the sequence's m_b entries.
"""
from __future__ import annotations

import numpy as np

__all__ = ["accept_longest_path"]


def accept_longest_path(parent, draft_tok, target_argmax, cu_nodes):
    """Return (accept_len [B], accept_path [N], next_token [B]), all int32."""
    parent = np.asarray(parent, dtype=np.int64)
    draft_tok = np.asarray(draft_tok, dtype=np.int64)
    target_argmax = np.asarray(target_argmax, dtype=np.int64)
    cu_nodes = np.asarray(cu_nodes, dtype=np.int64)
    B = len(cu_nodes) - 1
    N = int(cu_nodes[-1])
    accept_len = np.zeros(B, dtype=np.int32)
    accept_path = np.full(N, -1, dtype=np.int32)
    next_token = np.zeros(B, dtype=np.int32)
    for b in range(B):
        n0, n1 = int(cu_nodes[b]), int(cu_nodes[b + 1])
        m = n1 - n0
        par = parent[n0:n1]
        for i in range(m):
            if not (-1 <= par[i] < i):
                raise ValueError(f"sequence {b}: parent[{i}] = {par[i]} is not in [-1, {i})")
        slot = target_argmax[n0 + b: n1 + b + 1]
        best, best_depth = -1, 0
        for i in range(m):
            # walk node i and its ancestors; every one must be matched
            chain = []
            j = i
            while j >= 0:
                chain.append(j)
                j = int(par[j])
            if all(draft_tok[n0 + j] == slot[par[j] + 1] for j in chain):
                depth = len(chain)
                if depth > best_depth:      # strict: ties keep the smaller index
                    best, best_depth = i, depth
        if best >= 0:
            path = []
            j = best
            while j >= 0:
                path.append(j)
                j = int(par[j])
            path.reverse()
            accept_path[n0:n0 + len(path)] = path
        accept_len[b] = best_depth
        next_token[b] = slot[best + 1]
    return accept_len, accept_path, next_token
