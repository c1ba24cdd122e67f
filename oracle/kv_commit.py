"""Committing the accepted path's target K/V into the cache.

TEST INFRASTRUCTURE ONLY (see the package docstring): never called by the library.

"Faster decoding" (aaai.latere.ai), section "The scheduler must plan speculative work":
the reserve / execute / commit protocol applies to speculation.  Before a round the
scheduler reserves room for every node to be scored; after verification only the
target KV of the accepted draft prefix is committed and every rejected tail or branch
is released.  The correction or bonus token gets its target KV in the next round.

Readings taken where the page is silent
---------------------------------------
* The committed rows are the accepted path's tree K/V rows, root first, written to the
  cache rows ``dst_row[b] .. dst_row[b] + accept_len[b] - 1`` (for a cache whose
  sequences own reserved room after their prefix, ``dst_row[b]`` is the prefix end).
* Releasing a rejected branch writes nothing: its rows are simply not copied.
* No other cache row changes.
"""
from __future__ import annotations

import numpy as np

__all__ = ["commit_accepted_kv"]


def commit_accepted_kv(k_cache, v_cache, tree_k, tree_v, cu_nodes, accept_len, accept_path, dst_row):
    """Return new (k_cache, v_cache) with each sequence's accepted path appended.

    k_cache / v_cache [rows, Hkv, d]; tree_k / tree_v [N, Hkv, d]; cu_nodes [B+1];
    accept_len [B]; accept_path [N] (per sequence: local ids root first, then -1);
    dst_row [B].  Any dtype: rows are copied, never converted."""
    k_out = np.array(k_cache, copy=True)
    v_out = np.array(v_cache, copy=True)
    cu_nodes = np.asarray(cu_nodes, dtype=np.int64)
    for b in range(len(cu_nodes) - 1):
        n0 = int(cu_nodes[b])
        for j in range(int(accept_len[b])):
            node = int(accept_path[n0 + j])  # the j-th node of the path, root first
            k_out[int(dst_row[b]) + j] = tree_k[n0 + node]
            v_out[int(dst_row[b]) + j] = tree_v[n0 + node]
    return k_out, v_out
