"""Pins for oracle.rejection_sampling: frequency tests on a tiny vocabulary, as the
Faster decoding test list prescribes ("Correctness and fault tests": empirical output
frequencies against the target distribution for p = q, partial overlap and disjoint
supports; forced first rejection, late rejection and all-accept)."""
import numpy as np

from oracle import quantised_draw, verify_chain_sampling
from tests import _pins


def test_emitted_tokens_follow_the_target_distribution():
    _pins.check_sampling_marginals(verify_chain_sampling, np.random.default_rng(31))


def test_forced_first_late_and_no_rejection():
    _pins.check_sampling_forced_cases(verify_chain_sampling, np.random.default_rng(32))


def test_quantised_draw_is_the_inverse_cdf():
    _pins.check_quantised_draw_against_searchsorted(quantised_draw, np.random.default_rng(33))


def test_quantised_draw_edges():
    w = np.array([0, 0.25, 0, 0.75], np.float32)
    assert quantised_draw(w, np.float32(0.0)) == 1          # zero masses are never drawn
    assert quantised_draw(w, np.float32(0.2499)) == 1
    assert quantised_draw(w, np.float32(0.2501)) == 3
    assert quantised_draw(w, np.float32(np.nextafter(np.float32(1), np.float32(0)))) == 3
    assert quantised_draw(np.zeros(3, np.float32), np.float32(0.5)) == -1
