"""Pins for oracle.gdn_tree (DFlash-TfM, Method 3, rollback-free tree verification for
Gated DeltaNet): the per-path recurrence against the page's triangular-solve form
computed by numpy.linalg.solve, closed forms, and the tree's independence structure."""
import numpy as np

from oracle import gdn_tree_outputs
from tests import _pins


def test_recurrence_equals_the_triangular_solve_form():
    _pins.check_gdn_triangular_solve(gdn_tree_outputs, np.random.default_rng(61))


def test_no_write_only_decays():
    _pins.check_gdn_no_write(gdn_tree_outputs, np.random.default_rng(62))


def test_associative_recall_with_orthonormal_keys():
    _pins.check_gdn_associative_recall(gdn_tree_outputs, np.random.default_rng(63))


def test_a_node_sees_only_its_own_path():
    for s in range(6):
        _pins.check_gdn_sibling_independence(gdn_tree_outputs, np.random.default_rng(64 + s))
