"""Expected tokens emitted per verification cycle.

TEST INFRASTRUCTURE ONLY (see the package docstring): never called by the library.

"Faster decoding" (aaai.latere.ai), section "Generation is sequential, verification
can be parallel": for a linear draft of gamma tokens, with A_k the event that
positions 1..k are all accepted and s_k = Pr(A_1 and ... and A_k), s_0 = 1, a cycle
that emits the accepted prefix plus one correction or bonus token yields Y tokens with

    E[Y] = 1 + sum_{k=1..gamma} s_k .

Only when every conditional acceptance probability equals a constant alpha does
s_k = alpha^k, which gives sum_{k=0..gamma} alpha^k = (1 - alpha^(gamma+1)) / (1 - alpha)
(gamma + 1 at alpha = 1).  The same section's runnable example turns a list of
per-position conditional acceptance probabilities into survival values by running
products.
"""
from __future__ import annotations

import numpy as np

__all__ = ["survival_from_conditional", "expected_tokens", "iid_expected_tokens"]


def survival_from_conditional(conditional):
    """s_k = prod_{j<=k} c_j for k = 1..gamma."""
    s, alive = [], 1.0
    for c in conditional:
        alive *= float(c)
        s.append(alive)
    return np.asarray(s, dtype=np.float64)


def expected_tokens(survival) -> float:
    """E[Y] = 1 + sum_k s_k."""
    return 1.0 + float(np.sum(np.asarray(survival, dtype=np.float64)))


def iid_expected_tokens(alpha: float, gamma: int) -> float:
    """E[Y] under a constant conditional acceptance probability alpha."""
    alpha = float(alpha)
    if alpha == 1.0:
        return float(gamma + 1)
    return (1.0 - alpha ** (gamma + 1)) / (1.0 - alpha)
