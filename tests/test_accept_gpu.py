"""GPU acceptance walk: bit-exact against the oracle."""
import numpy as np
import pytest
import torch

import oracle
from tree_verification_attention_gb300 import api, workloads
from tests import _gpu, _pins

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _run(parent, draft, slots, cu):
    i32 = lambda a: torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()  # noqa: E731
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = api.accept_longest_path(i32(cu), i32(parent), i32(draft), i32(slots), dev_status=st)
    torch.cuda.synchronize()
    return [x.cpu().numpy() for x in a], int(st.item())


def _check(parent, draft, slots, cu):
    (alen, path, nxt), st = _run(parent, draft, slots, cu)
    assert st == 0
    r = oracle.accept_longest_path(parent, draft, slots, cu)
    np.testing.assert_array_equal(alen, r[0])
    np.testing.assert_array_equal(path, r[1])
    np.testing.assert_array_equal(nxt, r[2])


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_workload_trees(cfg):
    w = workloads.make_workload(cfg, prefix=16 if cfg != 4 else (16, 32))
    _check(w.parent, w.draft_tok, w.target_argmax, w.cu_nodes)


def test_every_tree_up_to_six_nodes_in_one_batch():
    rng = np.random.default_rng(0)
    parents, drafts, slots, sizes = [], [], [], []
    for m in range(1, 7):
        for par in _pins.all_parent_arrays(m):
            for _ in range(2):
                parents.append(np.array(par, np.int32))
                drafts.append(rng.integers(0, 2, m).astype(np.int32))
                slots.append(rng.integers(0, 2, m + 1).astype(np.int32))
                sizes.append(m)
    cu = np.cumsum([0] + sizes).astype(np.int32)
    _check(np.concatenate(parents), np.concatenate(drafts), np.concatenate(slots), cu)


def test_max_size_and_empty_trees_and_all_accept():
    m = 128
    parent_chain = np.arange(-1, m - 1, dtype=np.int32)
    slots_chain = np.arange(1, m + 2, dtype=np.int32)
    draft_chain = slots_chain[parent_chain + 1]            # every node matches: all accepted
    parent_wide = np.full(m, -1, np.int32)
    slots_wide = np.full(m + 1, 5, np.int32)
    draft_wide = np.arange(m, dtype=np.int32) + 100         # nothing matches
    cu = np.array([0, m, m, 2 * m], np.int32)                # middle sequence is empty
    parent = np.concatenate([parent_chain, parent_wide])
    draft = np.concatenate([draft_chain, draft_wide])
    slots = np.concatenate([slots_chain, np.array([42], np.int32), slots_wide])
    (alen, path, nxt), st = _run(parent, draft, slots, cu)
    assert st == 0
    assert list(alen) == [128, 0, 0] and list(nxt) == [129, 42, 5]
    assert list(path[:m]) == list(range(m)) and np.all(path[m:] == -1)
    _check(parent, draft, slots, cu)


def test_random_deep_trees():
    rng = np.random.default_rng(1)
    B = 300
    sizes = rng.integers(1, 129, B)
    parents, drafts, slots = [], [], []
    for m in sizes:
        par = workloads.random_tree(rng, int(m)) if rng.random() < 0.5 else workloads.chain_tree(int(m))
        sl = rng.integers(0, 3, m + 1).astype(np.int32)
        dr = np.where(rng.random(m) < 0.8, sl[par + 1], rng.integers(0, 3, m)).astype(np.int32)
        parents.append(par), drafts.append(dr), slots.append(sl)
    cu = np.cumsum([0] + list(sizes)).astype(np.int32)
    _check(np.concatenate(parents), np.concatenate(drafts), np.concatenate(slots), cu)


def test_bad_parent_and_oversized_tree_flag_status():
    parent = np.array([-1, 0, 2], np.int32)
    (alen, path, nxt), st = _run(parent, np.zeros(3, np.int32), np.arange(4, dtype=np.int32), np.array([0, 3], np.int32))
    assert st == 3 and alen[0] == 0 and nxt[0] == 0 and np.all(path == -1)
    m = 129
    (alen, _, nxt), st = _run(np.arange(-1, m - 1, dtype=np.int32), np.zeros(m, np.int32),
                             np.zeros(m + 1, np.int32), np.array([0, m], np.int32))
    assert st == 1 and alen[0] == 0 and nxt[0] == -1
