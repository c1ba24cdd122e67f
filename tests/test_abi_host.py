"""The C-ABI library loads and exports every entry point include/tva.h declares, and
its host-side argument checks reject bad calls before touching a GPU."""
import ctypes
import os
import re

import pytest

import __graft_entry__
from tree_verification_attention_gb300 import api, build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    __graft_entry__.build()
    return api.load_library()


def _declared_functions():
    names = []
    for h in sorted(os.listdir(os.path.join(ROOT, "include"))):
        if not h.endswith(".h"):
            continue
        text = open(os.path.join(ROOT, "include", h)).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names += re.findall(r"^\s*(?:const\s+)?[A-Za-z_][A-Za-z0-9_]*\s*\*?\s+\*?([a-z_][a-z0-9_]*)\s*\(",
                            text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_expected_entry_points():
    names = _declared_functions()
    for n in ("tree_verify_attn_varlen", "tree_verify_attn", "accept_longest_path",
              "tva_workspace_size", "tree_verify_attn_partials", "tree_verify_attn_combine",
              "tva_status_string", "tva_release", "tva_read_device_status", "tva_num_workers",
              "commit_accepted_kv", "verify_chain_sampling", "gdn_tree_verify", "tva_diag_set_wait_limit", "tva_diag_use_cta_pair"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in _declared_functions() if not hasattr(lib, n)]
    assert not missing, missing
    assert os.path.dirname(build.LIB_PATH).endswith("tree_verification_attention_gb300")


def test_checked_build_exports_the_same_entry_points(lib):
    """libtva_checked.so (device-side index checks) is a drop-in for libtva.so."""
    checked = ctypes.CDLL(build.build(checked=True))
    missing = [n for n in _declared_functions() if not hasattr(checked, n)]
    assert not missing, missing


def test_status_strings(lib):
    assert api.status_string(0) == "TVA_OK"
    assert api.status_string(3) == "TVA_ERR_BAD_TREE"
    assert api.status_string(99) == "TVA_ERR_UNKNOWN"


def _params(**kw):
    base = dict(batch=1, num_q_heads=4, num_kv_heads=1, head_dim=64, dtype=1, softmax_scale=0.0,
                cu_prefix=8, cu_nodes=8, max_prefix_len=256, max_nodes=8, kv_capacity=256,
                node_capacity=8)
    base.update(kw)
    return api.Params(**base)


@pytest.mark.parametrize("kw,code", [
    (dict(head_dim=96), 2), (dict(num_q_heads=6, num_kv_heads=4), 1), (dict(max_nodes=129), 2),
    (dict(batch=0), 1), (dict(dtype=7), 2), (dict(max_prefix_len=-1), 1),
])
def test_host_checks_reject_bad_shapes(lib, kw, code):
    p = _params(**kw)
    assert lib.tva_workspace_size(ctypes.byref(p)) == 0
    assert lib.tva_num_workers(ctypes.byref(p)) == -1
    fake = ctypes.c_void_p(4096)
    r = lib.tree_verify_attn_partials(ctypes.byref(p), fake, fake, fake, fake, fake, fake, fake, 1 << 30, fake, None)
    assert r == code


def test_host_checks_reject_null_and_misaligned_pointers(lib):
    p = _params()
    a = ctypes.c_void_p(4096)
    mis = ctypes.c_void_p(4098)
    assert lib.tree_verify_attn_partials(None, a, a, a, a, a, a, a, 1 << 20, a, None) == 1
    assert lib.tree_verify_attn_partials(ctypes.byref(p), None, a, a, a, a, a, a, 1 << 20, a, None) == 1
    assert lib.tree_verify_attn_partials(ctypes.byref(p), mis, a, a, a, a, a, a, 1 << 20, a, None) == 1
    assert lib.tree_verify_attn_partials(ctypes.byref(p), a, a, a, a, a, a, a, 1 << 20, None, None) == 1
    assert lib.tree_verify_attn_varlen(ctypes.byref(p), a, a, a, a, a, a, mis, a, a, 1 << 20, a, None) == 1
    assert lib.tree_verify_attn(a, a, a, 16, a, a, a, 0, 4, 1, 64, 1, a, a, None) == 1
    assert lib.tree_verify_attn(a, a, a, -1, a, a, a, 4, 4, 1, 64, 1, a, a, None) == 1
    assert lib.accept_longest_path(0, 8, a, a, a, a, a, a, a, a, None) == 1
    assert lib.accept_longest_path(2, 8, a, None, a, a, a, a, a, a, None) == 1
    assert lib.accept_longest_path(2, -1, a, a, a, a, a, a, a, a, None) == 1


def test_commit_rejects_bad_arguments_on_the_host(lib):
    """Host-side checks return TVA_ERR_INVALID_ARG before anything is launched (the
    pointers below are never dereferenced)."""
    P = ctypes.c_void_p
    a = 1 << 20          # fake, 16-byte aligned device addresses
    row = 8 * 128 * 2    # Hkv=8, d=128, bf16

    def call(batch=1, hkv=8, d=128, dtype=0, ncap=16, maxn=16, kvcap=64, tk=a, tv=a + 16 * row,
             kc=a + 64 * row, vc=a + 256 * row):
        return lib.commit_accepted_kv(batch, hkv, d, dtype, ncap, maxn, kvcap, P(8), P(8), P(8), P(tk), P(tv),
                                      P(8), P(kc), P(vc), P(8), None)
    assert call(batch=0) == 1
    assert call(d=96) == 1
    assert call(dtype=7) == 1
    assert call(maxn=0) == 1 and call(maxn=129) == 1
    assert call(tk=a + 8) == 1                       # misaligned
    assert call(kc=a + 8 * row) == 1                 # k_cache overlaps tree_k
    assert call(vc=a + 64 * row + 10 * row) == 1     # v_cache overlaps k_cache
