"""Stochastic verification of a draft chain by modified rejection sampling.

TEST INFRASTRUCTURE ONLY (see the package docstring): never called by the library.

"Faster decoding" (aaai.latere.ai), section "Modified rejection sampling keeps the
target distribution": with target distribution p and draft distribution q at a
position and the draft token X ~ q, accept v = X with probability
a(v) = min(1, p(v) / q(v)); on rejection sample from the residual
r(v) = [p(v) - q(v)]_+ / Z, Z = sum_u [p(u) - q(u)]_+, so that
q(v) a(v) + Z r(v) = p(v).  The rule is applied left to right: the first rejection
stops the round with one correction token and drops the remaining candidates; if all
gamma candidates are accepted, one bonus token is sampled from the target's
distribution at the next position (so p is given for gamma + 1 positions).

Readings taken where the page is silent or leaves a numerical choice open
-------------------------------------------------------------------------
* The uniforms are inputs: ``u_accept`` (one per draft position) and ``u_sample`` (one
  per sequence, for the correction or bonus draw), each in [0, 1) float32.
* Acceptance at a position with draft token x: accept when p(x) >= q(x), else when
  ``u * q(x) < p(x)`` with the product rounded to float32 (u < p/q without a division;
  the decision is taken in float32 so that it is reproducible).  q(x) must be > 0 (the
  draft token was drawn from q).
* A draw from a distribution with masses w(v) (the residual [p - q]_+ with the
  difference rounded to float32, or p itself for the bonus) is an inverse-CDF draw on
  masses quantised to 2^-40: W(v) = floor(w(v) * 2^40) as integers, T = floor(U * Z)
  with U = floor(u * 2^24) / 2^24 and Z = sum_v W(v), and the token is the smallest v
  whose running integer sum exceeds T.  Integer sums do not depend on summation order,
  so every implementation draws the same token; masses below 2^-40 are never drawn.
* If the quantised residual is empty (Z = 0: the rejection had probability ~0), the
  correction is drawn from p at that position.
* Per sequence b: draft positions cu_draft[b] .. cu_draft[b+1]-1; p rows
  cu_draft[b] + b .. cu_draft[b+1] + b (gamma_b + 1 rows), q rows as the positions.
"""
from __future__ import annotations

import numpy as np

__all__ = ["verify_chain_sampling", "quantised_draw"]

_SCALE = 2 ** 40


def quantised_draw(w, u):
    """Inverse-CDF draw from nonnegative float32 masses w with one float32 uniform u."""
    W = [int(np.floor(np.float64(x) * _SCALE)) for x in np.asarray(w, dtype=np.float32)]
    Z = sum(W)
    if Z == 0:
        return -1
    U = int(np.floor(np.float64(np.float32(u)) * 2 ** 24))
    T = (U * Z) >> 24
    run = 0
    for v, x in enumerate(W):
        run += x
        if run > T:
            return v
    raise AssertionError("unreachable: T < Z")


def verify_chain_sampling(p, q, draft_tok, u_accept, u_sample, cu_draft):
    """Return (accept_len [B], out_token [B]) int32.

    p [sum(gamma_b + 1), V] and q [sum(gamma_b), V] float32 probabilities; draft_tok,
    u_accept [sum(gamma_b)]; u_sample [B]; cu_draft [B+1]."""
    p = np.asarray(p, dtype=np.float32)
    q = np.asarray(q, dtype=np.float32)
    cu = np.asarray(cu_draft, dtype=np.int64)
    B = len(cu) - 1
    accept_len = np.zeros(B, dtype=np.int32)
    out_token = np.zeros(B, dtype=np.int32)
    for b in range(B):
        g0, gamma = int(cu[b]), int(cu[b + 1] - cu[b])
        k = 0
        while k < gamma:
            x = int(draft_tok[g0 + k])
            px, qx = p[g0 + b + k, x], q[g0 + k, x]
            if not (px >= qx or np.float32(np.float32(u_accept[g0 + k]) * qx) < px):
                break
            k += 1
        accept_len[b] = k
        prow = p[g0 + b + k]
        if k < gamma:
            resid = np.maximum(np.float32(0), prow - q[g0 + k])       # float32 difference
            tok = quantised_draw(resid, u_sample[b])
            out_token[b] = tok if tok >= 0 else quantised_draw(prow, u_sample[b])
        else:
            out_token[b] = quantised_draw(prow, u_sample[b])
    return accept_len, out_token
