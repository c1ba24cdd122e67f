"""Log-sum-exp aggregation of attention partials, in float64.

TEST INFRASTRUCTURE ONLY (see the package docstring): never called by the library.

LongSpec, "Fast Tree Attention" section, "Aggregation", and the appendix
"Correctness of attention aggregation" (Proposition and proof): given the output and
log-sum-exp of attention over disjoint key groups,

    LSE_merge = log( exp(LSE_cache) + exp(LSE_specs) )
    O_merge   = O_cache * exp(LSE_cache - LSE_merge) + O_specs * exp(LSE_specs - LSE_merge)

equals attention over the union of the groups.  The proof rests on the numerator and
the denominator of the softmax each being a sum over the groups, so the same identity
holds for any number of groups; :func:`merge_partials` writes that S-group form.

Readings:
* the logarithm is evaluated in the mathematically identical stable form
  max + log(sum exp(LSE_s - max)) so that large logits do not overflow;
* an empty key group has LSE = -inf and output 0 and drops out of the merge with
  weight exp(-inf) = 0.
"""
from __future__ import annotations

import numpy as np

__all__ = ["attention_partial", "merge_partials"]


def attention_partial(q, K, V, softmax_scale: float):
    """Partial attention of one query over one key group.

    Returns (o, lse) with lse = log sum_j exp(Z^(j)), Z = softmax_scale * K q, and
    o = sum_j exp(Z^(j)) V^(j) / exp(lse) (the appendix's o_cache / o_specs)."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    if K.shape[0] == 0:
        return np.zeros(V.shape[1], dtype=np.float64), -np.inf
    z = softmax_scale * (K @ q)
    zmax = z.max()
    lse = zmax + np.log(np.exp(z - zmax).sum())
    o = (np.exp(z - lse)[:, None] * V).sum(axis=0)
    return o, lse


def merge_partials(o_parts, lse_parts):
    """Merge S partials: o_parts [S, ..., d], lse_parts [S, ...] -> (o [..., d], lse [...]).

    Rows whose every partial is empty (all LSE = -inf) come back as lse = -inf, o = 0."""
    o_parts = np.asarray(o_parts, dtype=np.float64)
    lse_parts = np.asarray(lse_parts, dtype=np.float64)
    mx = lse_parts.max(axis=0)
    safe = np.where(np.isfinite(mx), mx, 0.0)
    ssum = np.exp(lse_parts - safe).sum(axis=0)
    with np.errstate(divide="ignore"):
        lse = np.where(np.isfinite(mx), safe + np.log(ssum), -np.inf)
    w = np.where(np.isfinite(lse)[None], np.exp(lse_parts - np.where(np.isfinite(lse), lse, 0.0)[None]), 0.0)
    o = (o_parts * w[..., None]).sum(axis=0)
    return o, lse
