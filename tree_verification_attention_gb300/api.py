"""ctypes binding over ``libtva.so`` (include/tva.h), with the C entry points' names.

Argument marshalling only: torch tensors provide device memory and the current CUDA
stream; every step of the computation runs in the library's kernels.  There is no
CPU path: if the library is missing or a tensor is not on a CUDA device, the call
raises.
"""
from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build

__all__ = [
    "TvaError", "Params", "load_library", "workspace_size", "num_workers",
    "tree_verify_attn_varlen", "tree_verify_attn_partials", "tree_verify_attn_combine",
    "tree_verify_attn", "read_device_status", "release", "diag_set_wait_limit", "diag_use_cta_pair", "accept_longest_path",
    "status_string", "STATUS",
]

STATUS = {0: "TVA_OK", 1: "TVA_ERR_INVALID_ARG", 2: "TVA_ERR_UNSUPPORTED", 3: "TVA_ERR_BAD_TREE",
          4: "TVA_ERR_WORKSPACE", 5: "TVA_ERR_CUDA", 6: "TVA_ERR_TIMEOUT"}
DTYPES = {torch.bfloat16: 0, torch.float32: 1, torch.float16: 2}


class TvaError(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {STATUS.get(code, code)}")
        self.code = code


class Params(ctypes.Structure):
    _fields_ = [
        ("batch", ctypes.c_int), ("num_q_heads", ctypes.c_int), ("num_kv_heads", ctypes.c_int),
        ("head_dim", ctypes.c_int), ("dtype", ctypes.c_int), ("softmax_scale", ctypes.c_float),
        ("cu_prefix", ctypes.c_void_p), ("cu_nodes", ctypes.c_void_p),
        ("max_prefix_len", ctypes.c_int), ("max_nodes", ctypes.c_int),
        ("kv_capacity", ctypes.c_int), ("node_capacity", ctypes.c_int),
    ]


_lib = None
_P = ctypes.c_void_p
_I = ctypes.c_int
_SZ = ctypes.c_size_t


def load_library(path: str | None = None):
    """Load libtva.so (built by ``build.build()``); raises if it is absent.  The
    environment variable TVA_LIBRARY selects another build of the same library (for
    example libtva_checked.so, the index-checked variant)."""
    global _lib
    if _lib is not None:
        return _lib
    path = path or os.environ.get("TVA_LIBRARY") or _build.LIB_PATH
    if not os.path.exists(path):
        raise RuntimeError(f"{path} is missing: run tree_verification_attention_gb300.build.build() "
                           "(or __graft_entry__.build()) first; there is no fallback path")
    lib = ctypes.CDLL(path)
    PP = ctypes.POINTER(Params)
    sig = {
        "tva_workspace_size": (_SZ, [PP]),
        "tva_num_workers": (_I, [PP]),
        "tree_verify_attn_varlen": (_I, [PP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
        "tree_verify_attn_partials": (_I, [PP, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P]),
        "tree_verify_attn_combine": (_I, [PP, _P, _SZ, _P, _P, _P, _P]),
        "tree_verify_attn": (_I, [_P, _P, _P, _I, _P, _P, _P, _I, _I, _I, _I, _I, _P, _P, _P]),
        "tva_read_device_status": (_I, [ctypes.POINTER(ctypes.c_int32), _P]),
        "tva_release": (None, []),
        "tva_diag_set_wait_limit": (None, [ctypes.c_ulonglong, _I]),
        "tva_diag_use_cta_pair": (None, [_I]),
        "accept_longest_path": (_I, [_I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
        "commit_accepted_kv": (_I, [_I, _I, _I, _I, _I, _I, ctypes.c_longlong, _P, _P, _P, _P, _P, _P, _P, _P,
                                    _P, _P]),
        "verify_chain_sampling": (_I, [_I, _I, _I, ctypes.c_longlong, ctypes.c_longlong, _P, _P, _P, _P, _P, _P,
                                       _P, _P, _P, _P]),
        "gdn_tree_verify": (_I, [_I, _I, _I, _I, _I, _I, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]),
        "tva_status_string": (ctypes.c_char_p, [_I]),
        "tva_last_error": (ctypes.c_char_p, []),
    }
    for name, (res, args) in sig.items():
        fn = getattr(lib, name)
        fn.restype = res
        fn.argtypes = args
    _lib = lib
    return lib


def status_string(code: int) -> str:
    return load_library().tva_status_string(code).decode()


def _check(code: int, where: str):
    if code != 0:
        detail = load_library().tva_last_error().decode() if code == 5 else ""
        raise TvaError(code, where + (f" [{detail}]" if detail else ""))


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _dev(t: torch.Tensor, name: str, dtype=None):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor (there is no CPU path)")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dtype is not None and t.dtype != dtype:
        raise ValueError(f"{name} must be {dtype}, got {t.dtype}")
    return t


def make_params(q, k_cache, cu_prefix, cu_nodes, num_kv_heads, max_prefix_len, max_nodes,
                softmax_scale=0.0) -> Params:
    if q.dtype not in DTYPES:
        raise ValueError(f"unsupported dtype {q.dtype}")
    N, Hq, d = q.shape
    return Params(batch=cu_prefix.numel() - 1, num_q_heads=Hq, num_kv_heads=num_kv_heads, head_dim=d,
                  dtype=DTYPES[q.dtype], softmax_scale=float(softmax_scale),
                  cu_prefix=cu_prefix.data_ptr(), cu_nodes=cu_nodes.data_ptr(),
                  max_prefix_len=int(max_prefix_len), max_nodes=int(max_nodes),
                  kv_capacity=k_cache.shape[0], node_capacity=N)


def workspace_size(params: Params) -> int:
    return int(load_library().tva_workspace_size(ctypes.byref(params)))


def num_workers(params: Params) -> int:
    return int(load_library().tva_num_workers(ctypes.byref(params)))


def alloc_workspace(params: Params, device) -> torch.Tensor:
    n = workspace_size(params)
    if n == 0:
        raise TvaError(1, "tva_workspace_size")
    return torch.empty(n, dtype=torch.uint8, device=device)


def _attn_inputs(q, k_cache, v_cache, tree_k, tree_v, parent, cu_prefix, cu_nodes):
    _dev(q, "q")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("tree_k", tree_k), ("tree_v", tree_v)):
        _dev(t, name, q.dtype)
    for name, t in (("parent", parent), ("cu_prefix", cu_prefix), ("cu_nodes", cu_nodes)):
        _dev(t, name, torch.int32)
    if k_cache.shape != v_cache.shape or tree_k.shape != tree_v.shape:
        raise ValueError("k/v shapes differ")
    if tree_k.shape[0] != q.shape[0] or parent.shape[0] != q.shape[0]:
        raise ValueError("q, tree_k and parent must have one row per tree node")


def tree_verify_attn_partials(q, k_cache, v_cache, tree_k, tree_v, parent, cu_prefix, cu_nodes,
                              max_prefix_len, max_nodes, workspace, dev_status,
                              softmax_scale=0.0, stream=None, params=None):
    _attn_inputs(q, k_cache, v_cache, tree_k, tree_v, parent, cu_prefix, cu_nodes)
    p = params or make_params(q, k_cache, cu_prefix, cu_nodes, tree_k.shape[1], max_prefix_len,
                              max_nodes, softmax_scale)
    code = load_library().tree_verify_attn_partials(
        ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(tree_k), _ptr(tree_v),
        _ptr(parent), _ptr(workspace), workspace.numel(), _ptr(dev_status), _stream(stream))
    _check(code, "tree_verify_attn_partials")


def tree_verify_attn_combine(params: Params, workspace, out, lse, dev_status, stream=None):
    code = load_library().tree_verify_attn_combine(
        ctypes.byref(params), _ptr(workspace), workspace.numel(), _ptr(out), _ptr(lse),
        _ptr(dev_status), _stream(stream))
    _check(code, "tree_verify_attn_combine")


def tree_verify_attn_varlen(q, k_cache, v_cache, tree_k, tree_v, parent, cu_prefix, cu_nodes,
                            max_prefix_len, max_nodes, out=None, lse=None, workspace=None,
                            dev_status=None, softmax_scale=0.0, stream=None, params=None):
    """Returns (out [N, Hq, d], lse [N, Hq] float32).  Raises TvaError on a host-side
    error; device-side errors land in ``dev_status`` (allocated and zeroed here when
    not given; check it after synchronising)."""
    _attn_inputs(q, k_cache, v_cache, tree_k, tree_v, parent, cu_prefix, cu_nodes)
    p = params or make_params(q, k_cache, cu_prefix, cu_nodes, tree_k.shape[1], max_prefix_len,
                              max_nodes, softmax_scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    if workspace is None:
        workspace = alloc_workspace(p, q.device)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=q.device)
    code = load_library().tree_verify_attn_varlen(
        ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(tree_k), _ptr(tree_v),
        _ptr(parent), _ptr(out), _ptr(lse), _ptr(workspace), workspace.numel(), _ptr(dev_status),
        _stream(stream))
    _check(code, "tree_verify_attn_varlen")
    return out, lse


def tree_verify_attn(q, k_cache, v_cache, tree_k, tree_v, parent, out=None, lse=None, stream=None):
    """Single-sequence form: q [m, Hq, d], k_cache/v_cache [P, Hkv, d], tree_k/tree_v
    [m, Hkv, d], parent [m] int32.  Uses the library-owned workspace."""
    _dev(q, "q")
    for name, t in (("k_cache", k_cache), ("v_cache", v_cache), ("tree_k", tree_k), ("tree_v", tree_v)):
        _dev(t, name, q.dtype)
    _dev(parent, "parent", torch.int32)
    m, Hq, d = q.shape
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty((m, Hq), dtype=torch.float32, device=q.device)
    code = load_library().tree_verify_attn(
        _ptr(q), _ptr(k_cache), _ptr(v_cache), k_cache.shape[0], _ptr(tree_k), _ptr(tree_v),
        _ptr(parent), m, Hq, tree_k.shape[1], d, DTYPES[q.dtype], _ptr(out), _ptr(lse),
        _stream(stream))
    _check(code, "tree_verify_attn")
    return out, lse


def read_device_status(stream=None) -> int:
    v = ctypes.c_int32(0)
    _check(load_library().tva_read_device_status(ctypes.byref(v), _stream(stream)), "tva_read_device_status")
    return int(v.value)


def release():
    load_library().tva_release()


def diag_set_wait_limit(wait_limit_ns: int = 0, force_stall: bool = False):
    """Diagnostics for the device timeout path (tva_diag_set_wait_limit): the main-loop
    wait limit of the tensor-core partials kernel in ns (0 = default 2 s) and, with
    ``force_stall``, a wait that nothing completes.  Call with no arguments to reset."""
    load_library().tva_diag_set_wait_limit(int(wait_limit_ns), 1 if force_stall else 0)


def diag_use_cta_pair(enable: bool = False):
    """Diagnostics (tva_diag_use_cta_pair): select the CTA-pair partials kernel
    (cta_group::2, M = 256) for later calls where it applies; call with no argument to
    return to the default one-SM-per-worker kernel."""
    load_library().tva_diag_use_cta_pair(1 if enable else 0)


def accept_longest_path(cu_nodes, parent, draft_tok, target_argmax, accept_len=None,
                        accept_path=None, next_token=None, dev_status=None, stream=None):
    """Returns (accept_len [B], accept_path [N], next_token [B]) as int32 CUDA tensors."""
    for name, t in (("cu_nodes", cu_nodes), ("parent", parent), ("draft_tok", draft_tok),
                    ("target_argmax", target_argmax)):
        _dev(t, name, torch.int32)
    B = cu_nodes.numel() - 1
    N = parent.numel()
    if target_argmax.numel() != N + B or draft_tok.numel() != N:
        raise ValueError("target_argmax must hold N + B slots and draft_tok N tokens")
    dev = parent.device
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if accept_path is None:
        accept_path = torch.empty(N, dtype=torch.int32, device=dev)
    if next_token is None:
        next_token = torch.empty(B, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    code = load_library().accept_longest_path(
        B, N, _ptr(cu_nodes), _ptr(parent), _ptr(draft_tok), _ptr(target_argmax), _ptr(accept_len),
        _ptr(accept_path), _ptr(next_token), _ptr(dev_status), _stream(stream))
    _check(code, "accept_longest_path")
    return accept_len, accept_path, next_token


def commit_accepted_kv(cu_nodes, accept_len, accept_path, tree_k, tree_v, dst_row, k_cache, v_cache,
                       max_nodes=None, dev_status=None, stream=None):
    """Copies each sequence's accepted path (root first) of tree_k / tree_v [N, Hkv, d]
    into k_cache / v_cache [rows, Hkv, d] at rows dst_row[b] .. dst_row[b] +
    accept_len[b] - 1, in place.  Returns dev_status (int32 [1], 0 = ok)."""
    for name, t in (("cu_nodes", cu_nodes), ("accept_len", accept_len), ("accept_path", accept_path),
                    ("dst_row", dst_row)):
        _dev(t, name, torch.int32)
    _dev(tree_k, "tree_k")
    for name, t in (("tree_v", tree_v), ("k_cache", k_cache), ("v_cache", v_cache)):
        _dev(t, name, tree_k.dtype)
    if tree_k.dtype not in DTYPES:
        raise TypeError(f"unsupported dtype {tree_k.dtype}")
    B = cu_nodes.numel() - 1
    N, Hkv, d = tree_k.shape
    if max_nodes is None:
        max_nodes = int((cu_nodes[1:] - cu_nodes[:-1]).max().item()) if B > 0 else 1
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=tree_k.device)
    code = load_library().commit_accepted_kv(
        B, Hkv, d, DTYPES[tree_k.dtype], N, max(1, int(max_nodes)), k_cache.shape[0], _ptr(cu_nodes),
        _ptr(accept_len), _ptr(accept_path), _ptr(tree_k), _ptr(tree_v), _ptr(dst_row), _ptr(k_cache),
        _ptr(v_cache), _ptr(dev_status), _stream(stream))
    _check(code, "commit_accepted_kv")
    return dev_status


def verify_chain_sampling(cu_draft, p, q, draft_tok, u_accept, u_sample, max_draft=None, accept_len=None,
                          out_token=None, dev_status=None, stream=None):
    """Modified rejection sampling over draft chains.  p [sum(gamma+1), V], q [sum gamma, V]
    float32; draft_tok, u_accept [sum gamma]; u_sample [B]; cu_draft [B+1].
    Returns (accept_len [B], out_token [B]) int32 CUDA tensors."""
    for name, t in (("cu_draft", cu_draft), ("draft_tok", draft_tok)):
        _dev(t, name, torch.int32)
    for name, t in (("p", p), ("q", q), ("u_accept", u_accept), ("u_sample", u_sample)):
        _dev(t, name, torch.float32)
    B = cu_draft.numel() - 1
    V = p.shape[1]
    if q.shape[1] != V and q.numel() > 0:
        raise ValueError("p and q must share the vocabulary")
    if max_draft is None:
        max_draft = int((cu_draft[1:] - cu_draft[:-1]).max().item()) if B > 0 else 0
    dev = p.device
    if accept_len is None:
        accept_len = torch.empty(B, dtype=torch.int32, device=dev)
    if out_token is None:
        out_token = torch.empty(B, dtype=torch.int32, device=dev)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=dev)
    # with no draft position at all, q / draft_tok / u_accept are never read: any
    # valid address stands in for the empty tensors
    some = lambda t: _ptr(t) if t.numel() > 0 else _ptr(p)  # noqa: E731
    code = load_library().verify_chain_sampling(
        B, V, int(max_draft), p.shape[0], q.shape[0] if q.numel() > 0 else 0, _ptr(cu_draft), _ptr(p), some(q),
        some(draft_tok), some(u_accept), _ptr(u_sample), _ptr(accept_len), _ptr(out_token), _ptr(dev_status),
        _stream(stream))
    _check(code, "verify_chain_sampling")
    return accept_len, out_token


def gdn_tree_verify(cu_nodes, parent, q, k, v, beta, alpha, S0, out=None, max_nodes=None, dev_status=None,
                    stream=None):
    """Gated DeltaNet tree verification.  q, k, v [N, H, d] float32 or bfloat16 (all three
    alike); beta, alpha [N, H] and S0 [B, H, d, d] float32; CUDA tensors.  Returns out
    [N, H, d] in q's dtype."""
    for name, t in (("cu_nodes", cu_nodes), ("parent", parent)):
        _dev(t, name, torch.int32)
    if q.dtype not in (torch.float32, torch.bfloat16):
        raise ValueError(f"unsupported dtype {q.dtype}")
    for name, t in (("q", q), ("k", k), ("v", v)):
        _dev(t, name, q.dtype)
    for name, t in (("beta", beta), ("alpha", alpha), ("S0", S0)):
        _dev(t, name, torch.float32)
    B = cu_nodes.numel() - 1
    N, H, d = q.shape
    if max_nodes is None:
        max_nodes = int((cu_nodes[1:] - cu_nodes[:-1]).max().item()) if B > 0 else 1
    if out is None:
        out = torch.empty_like(v)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=q.device)
    code = load_library().gdn_tree_verify(B, H, d, DTYPES[q.dtype], N, max(1, int(max_nodes)), _ptr(cu_nodes),
                                          _ptr(parent), _ptr(q), _ptr(k), _ptr(v), _ptr(beta), _ptr(alpha),
                                          _ptr(S0), _ptr(out), _ptr(dev_status), _stream(stream))
    _check(code, "gdn_tree_verify")
    return out


def tree_verify_attn_varlen_noalloc(q, k_cache, v_cache, tree_k, tree_v, parent, cu_prefix, cu_nodes,
                                    max_prefix_len, max_nodes, out=None, lse=None, dev_status=None,
                                    softmax_scale=0.0, stream=None, params=None):
    """tree_verify_attn_varlen without a workspace argument, for callers that may not
    allocate device memory: the library's fixed 32 MiB per-GPU scratch holds the
    partials.  Larger problems raise TvaError (TVA_ERR_WORKSPACE).  Calls share that
    scratch, so calls that overlap on the GPU must be serialised by the caller.
    ``out``, ``lse`` and ``dev_status`` are allocated here only when not given."""
    _attn_inputs(q, k_cache, v_cache, tree_k, tree_v, parent, cu_prefix, cu_nodes)
    lib = load_library()
    fn = lib.tree_verify_attn_varlen_noalloc
    fn.restype = _I
    fn.argtypes = [ctypes.POINTER(Params), _P, _P, _P, _P, _P, _P, _P, _P, _P, _P]
    p = params or make_params(q, k_cache, cu_prefix, cu_nodes, tree_k.shape[1], max_prefix_len,
                              max_nodes, softmax_scale)
    if out is None:
        out = torch.empty_like(q)
    if lse is None:
        lse = torch.empty(q.shape[:2], dtype=torch.float32, device=q.device)
    if dev_status is None:
        dev_status = torch.zeros(1, dtype=torch.int32, device=q.device)
    code = fn(ctypes.byref(p), _ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(tree_k), _ptr(tree_v),
              _ptr(parent), _ptr(out), _ptr(lse), _ptr(dev_status), _stream(stream))
    if code != 0:
        detail = lib.tva_last_error().decode()
        raise TvaError(code, "tree_verify_attn_varlen_noalloc" + (f" [{detail}]" if detail else ""))
    return out, lse
