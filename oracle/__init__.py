"""CPU oracle for tree-verification attention and greedy tree acceptance.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py`` may import this package.  The library's CUDA path never
calls it and shares no code with it.

Everything here is plain float64 numpy (integers for the acceptance walk): each
function writes out the definition the method reaches exactly, in the order and
notation of the pages it cites, with no blocking, fusion or reordering beyond that
definition.

* :mod:`oracle.tree_attention` - one softmax per (node, query head) over the
  concatenation of the cached prefix keys and the tree keys, with the tree keys masked
  to the node's ancestors and itself.
* :mod:`oracle.lse_merge` - the log-sum-exp aggregation of attention partials.
* :mod:`oracle.acceptance` - the greedy longest-accepted-path walk.
* :mod:`oracle.expected_tokens` - expected tokens per verification cycle.
* :mod:`oracle.kv_commit` - committing the accepted path's K/V into the cache.
* :mod:`oracle.rejection_sampling` - stochastic verification of a draft chain.
* :mod:`oracle.gdn_tree` - tree verification for Gated DeltaNet layers.

Every function is pinned by ``tests/test_oracle_*.py`` against facts fixed by the pages
or by mathematics (closed forms, brute force, library routines on independently
constructed inputs, printed worked examples); none is "parity unpinned".
"""
from .tree_attention import ancestor_mask, tree_verify_attention, tree_verify_attention_rows
from .lse_merge import merge_partials, attention_partial
from .acceptance import accept_longest_path
from .expected_tokens import expected_tokens, survival_from_conditional, iid_expected_tokens
from .kv_commit import commit_accepted_kv
from .rejection_sampling import verify_chain_sampling, quantised_draw
from .gdn_tree import gdn_tree_outputs, gdn_path_state

__all__ = [
    "ancestor_mask",
    "tree_verify_attention",
    "tree_verify_attention_rows",
    "merge_partials",
    "attention_partial",
    "accept_longest_path",
    "expected_tokens",
    "survival_from_conditional",
    "iid_expected_tokens",
    "commit_accepted_kv",
    "verify_chain_sampling",
    "quantised_draw",
    "gdn_tree_outputs",
    "gdn_path_state",
]
