"""GPU commit of the accepted path's K/V: bit-exact against the oracle (it is a copy)."""
import numpy as np
import pytest
import torch

import oracle
from tree_verification_attention_gb300 import api, workloads
from tests import _pins

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    import __graft_entry__
    __graft_entry__.build()


def _to_dev(a, dtype):
    t = torch.from_numpy(np.ascontiguousarray(a))
    if dtype == "bf16":
        t = t.view(torch.int16).view(torch.bfloat16)
    return t.cuda()


def _to_host(t, dtype):
    t = t.cpu()
    return t.view(torch.int16).numpy().view(np.uint16) if dtype == "bf16" else t.numpy()


def _i32(a):
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).cuda()


def _reserved_cache(w, room, rng):
    """Sequence b owns cache rows [base_b, base_b + P_b + room): its prefix, then junk."""
    P = [int(x) for x in w.prefix_lens]
    base = np.concatenate([[0], np.cumsum([p + room for p in P])]).astype(np.int64)
    shape = (int(base[-1]),) + tuple(w.k_cache.shape[1:])
    junk = lambda: (rng.integers(0, 1 << 16, shape, dtype=np.uint16) if w.dtype == "bf16"  # noqa: E731
                    else rng.standard_normal(shape).astype(np.float32))
    kc, vc = junk(), junk()
    for b in range(w.batch):
        src = slice(int(w.cu_prefix[b]), int(w.cu_prefix[b + 1]))
        kc[base[b]:base[b] + P[b]] = w.k_cache[src]
        vc[base[b]:base[b] + P[b]] = w.v_cache[src]
    return kc, vc, (base[:-1] + np.array(P)).astype(np.int32)


def _commit_gpu(w, kc, vc, alen, apath, dst, max_nodes=None):
    k_t, v_t = _to_dev(kc, w.dtype), _to_dev(vc, w.dtype)
    st = api.commit_accepted_kv(_i32(w.cu_nodes), _i32(alen), _i32(apath), _to_dev(w.tree_k, w.dtype),
                                _to_dev(w.tree_v, w.dtype), _i32(dst), k_t, v_t,
                                max_nodes=max_nodes or int(w.tree_sizes.max()))
    torch.cuda.synchronize()
    return _to_host(k_t, w.dtype), _to_host(v_t, w.dtype), int(st.item())


def _check(w, alen, apath, room=None, seed=0):
    rng = np.random.default_rng(seed)
    kc, vc, dst = _reserved_cache(w, room or int(w.tree_sizes.max()), rng)
    k_exp, v_exp = oracle.commit_accepted_kv(kc, vc, w.tree_k, w.tree_v, w.cu_nodes, alen, apath, dst)
    k_got, v_got, st = _commit_gpu(w, kc, vc, alen, apath, dst)
    assert st == 0
    np.testing.assert_array_equal(k_got, k_exp)
    np.testing.assert_array_equal(v_got, v_exp)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4, 5])
def test_workload_acceptance_committed(cfg):
    w = workloads.make_workload(cfg, prefix=16 if cfg != 4 else (16, 40))
    alen, apath, _ = oracle.accept_longest_path(w.parent, w.draft_tok, w.target_argmax, w.cu_nodes)
    _check(w, alen, apath, seed=cfg)


def test_paths_to_every_node():
    """A batch of 128 trees of 128 nodes, d = 64: sequence b commits the path to node b."""
    B = m = 128
    w = workloads.make_workload(1, seed=9, m=m, batch=B, prefix=3, Hq=8, Hkv=2, dtype="bf16")
    assert (w.tree_sizes == m).all()
    alen = np.zeros(B, np.int32)
    apath = np.full(B * m, -1, np.int32)
    for b in range(B):
        p = _pins.path_to(w.parent[b * m:(b + 1) * m], b)
        alen[b] = len(p)
        apath[b * m:b * m + len(p)] = p
    _check(w, alen, apath, seed=5)


def test_gpu_walk_then_gpu_commit_equals_oracle_walk_then_oracle_commit():
    w = workloads.make_workload(4, batch=6, prefix=(8, 60), m=32)
    t_par, t_tok, t_tgt, t_cu = _i32(w.parent), _i32(w.draft_tok), _i32(w.target_argmax), _i32(w.cu_nodes)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    alen_t, apath_t, _ = api.accept_longest_path(t_cu, t_par, t_tok, t_tgt, dev_status=st)
    rng = np.random.default_rng(3)
    kc, vc, dst = _reserved_cache(w, 32, rng)
    k_t, v_t = _to_dev(kc, w.dtype), _to_dev(vc, w.dtype)
    api.commit_accepted_kv(t_cu, alen_t, apath_t, _to_dev(w.tree_k, w.dtype), _to_dev(w.tree_v, w.dtype),
                           _i32(dst), k_t, v_t, max_nodes=32, dev_status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    alen, apath, _ = oracle.accept_longest_path(w.parent, w.draft_tok, w.target_argmax, w.cu_nodes)
    k_exp, v_exp = oracle.commit_accepted_kv(kc, vc, w.tree_k, w.tree_v, w.cu_nodes, alen, apath, dst)
    np.testing.assert_array_equal(_to_host(k_t, w.dtype), k_exp)
    np.testing.assert_array_equal(_to_host(v_t, w.dtype), v_exp)


def test_empty_paths_write_nothing():
    w = workloads.make_workload(4, batch=3, prefix=(8, 30), m=20)
    _check(w, np.zeros(3, np.int32), np.full(w.num_nodes, -1, np.int32))


def _bad_case(mutate):
    w = workloads.make_workload(4, batch=3, prefix=(8, 30), m=20)
    alen, apath, _ = oracle.accept_longest_path(w.parent, w.draft_tok, w.target_argmax, w.cu_nodes)
    alen = alen.copy(); apath = apath.copy()
    alen[1] = 3
    apath[w.cu_nodes[1]:w.cu_nodes[1] + 3] = [0, 1, 2]
    rng = np.random.default_rng(4)
    kc, vc, dst = _reserved_cache(w, 20, rng)
    mutate(w, alen, apath, dst)
    k_got, v_got, st = _commit_gpu(w, kc, vc, alen, apath, dst)
    assert st == 1  # TVA_ERR_INVALID_ARG
    # sequence 1 untouched, the others committed
    ok = np.array([1, 0, 1], bool)
    alen_ok = np.where(ok, alen, 0).astype(np.int32)
    k_exp, v_exp = oracle.commit_accepted_kv(kc, vc, w.tree_k, w.tree_v, w.cu_nodes, alen_ok, apath, dst)
    np.testing.assert_array_equal(k_got, k_exp)
    np.testing.assert_array_equal(v_got, v_exp)


def test_path_id_out_of_range_leaves_the_sequence_untouched():
    def m(w, alen, apath, dst):
        apath[w.cu_nodes[1] + 2] = int(w.tree_sizes[1])   # one past the sequence's nodes
    _bad_case(m)


def test_length_above_tree_size_leaves_the_sequence_untouched():
    def m(w, alen, apath, dst):
        alen[1] = int(w.tree_sizes[1]) + 1
    _bad_case(m)


def test_destination_past_the_cache_leaves_the_sequence_untouched():
    def m(w, alen, apath, dst):
        dst[1] = int(w.cu_prefix[-1]) + 3 * 20 - 2                      # 2 rows short of room
    _bad_case(m)


def test_host_rejects_overlap_of_source_and_cache():
    w = workloads.make_workload(2, prefix=16)
    kc = _to_dev(np.zeros((64,) + w.k_cache.shape[1:], np.uint16), "bf16")
    tk = kc[:w.num_nodes]                                   # the tree rows live inside the cache
    vc = _to_dev(np.zeros((64,) + w.k_cache.shape[1:], np.uint16), "bf16")
    with pytest.raises(api.TvaError):
        api.commit_accepted_kv(_i32(w.cu_nodes), _i32([1]), _i32(np.zeros(w.num_nodes)), tk, tk, _i32([40]),
                               kc, vc, max_nodes=8)


def test_full_size_cache_commit():
    """Config 3's shapes: a 64-node tree appended after a 65536-row prefix."""
    w = workloads.make_workload(3)
    alen, apath, _ = oracle.accept_longest_path(w.parent, w.draft_tok, w.target_argmax, w.cu_nodes)
    room = 64
    rows = int(w.cu_prefix[-1]) + room
    kc = np.zeros((rows,) + w.k_cache.shape[1:], np.uint16)
    kc[:-room] = w.k_cache
    vc = kc.copy()
    dst = np.array([rows - room], np.int32)
    k_got, v_got, st = _commit_gpu(w, kc, vc, alen, apath, dst)
    assert st == 0
    k_exp, v_exp = oracle.commit_accepted_kv(kc, vc, w.tree_k, w.tree_v, w.cu_nodes, alen, apath, dst)
    np.testing.assert_array_equal(k_got[-room:], k_exp[-room:])
    np.testing.assert_array_equal(v_got[-room:], v_exp[-room:])
    idx = np.random.default_rng(0).integers(0, rows - room, 4096)
    np.testing.assert_array_equal(k_got[idx], kc[idx])
