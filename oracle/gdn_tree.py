"""Tree verification for Gated DeltaNet layers: every draft-tree node's output from the
recurrence run along its root-to-node path.

TEST INFRASTRUCTURE ONLY (see the package docstring): never called by the library.

"DFlash-TfM" (gist.science 2607.06763), Method 3, "Rollback-free tree verification for
GDN": a Gated DeltaNet layer updates its state by
    S_t = alpha_t (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T,
which does not commute across tokens, so a tree cannot be verified with an ancestor
mask alone.  The page's method (topological order, ancestor interaction matrices, a
triangular solve (I + X) U = beta V, the state update deferred until the accepted
branch is known) computes exactly what running the recurrence along each node's path
from the committed state gives; this oracle is that definition, written out.

Readings taken where the page is silent
---------------------------------------
* State S is [d_k, d_v] (keys index rows), and a node's output is o_i = S_i^T q_i,
  S_i being the state after the node's own token (the delta rule reads after writing).
* S_0 is the committed state at the prefix end, per sequence and head; every root
  (parent -1) continues from S_0.  q, k, v, beta, alpha arrive as the layer computes them
  (any key normalisation, gate activation or query scaling is already applied).
* Heads are independent (one state per head).
"""
from __future__ import annotations

import numpy as np

__all__ = ["gdn_tree_outputs", "gdn_path_state"]


def gdn_path_state(S0, k, v, beta, alpha, path):
    """State after running the recurrence over the nodes of `path` (root first) from S0.
    S0 [dk, dv]; k [n, dk]; v [n, dv]; beta, alpha [n]."""
    S = np.array(S0, dtype=np.float64, copy=True)
    for j in path:
        kj = np.asarray(k[j], dtype=np.float64)
        vj = np.asarray(v[j], dtype=np.float64)
        S = alpha[j] * (S - beta[j] * np.outer(kj, kj @ S)) + beta[j] * np.outer(kj, vj)
    return S


def gdn_tree_outputs(q, k, v, beta, alpha, S0, parent, cu_nodes):
    """o [N, H, dv] float64.

    q, k [N, H, dk]; v [N, H, dv]; beta, alpha [N, H]; S0 [B, H, dk, dv];
    parent [N] local ids (topological); cu_nodes [B+1]."""
    q = np.asarray(q, dtype=np.float64)
    N, H, _ = q.shape
    dv = np.asarray(v).shape[2]
    out = np.zeros((N, H, dv))
    cu = np.asarray(cu_nodes, dtype=np.int64)
    for b in range(len(cu) - 1):
        n0, n1 = int(cu[b]), int(cu[b + 1])
        par = np.asarray(parent[n0:n1], dtype=np.int64)
        for i in range(n1 - n0):
            if not (-1 <= par[i] < i):
                raise ValueError("parent ids must be topological: -1 <= parent[i] < i")
            path, j = [], i
            while j >= 0:
                path.append(n0 + j)
                j = int(par[j])
            path.reverse()
            for h in range(H):
                S = gdn_path_state(S0[b, h], k[:, h], v[:, h], beta[:, h], alpha[:, h], path)
                out[n0 + i, h] = S.T @ q[n0 + i, h]
    return out
