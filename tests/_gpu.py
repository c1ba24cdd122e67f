"""Helpers for the GPU parity tests: move a workload to cuda:0, run the library, and
compare with the oracle at the tolerances stated for each dtype."""
from __future__ import annotations

import numpy as np
import torch

import oracle
from tree_verification_attention_gb300 import api

# bf16: max-abs(out) <= 2e-2 and relative LSE error <= 1e-3; fp32: 1e-4 and 1e-5.  The LSE
# error is taken relative to max(|LSE|, 1): a row's LSE is 0 when its softmax denominator
# is 1 (a root with a zero logit, say), where an error relative to |LSE| has no meaning.
# fp16 (10 mantissa bits against bf16's 7): P and out rounded to fp16 give relative
# errors of a few 2^-11 on |out| <= ~4, so max-abs 5e-3; the LSE comes from fp32 sums.
TOL = {"bf16": (2e-2, 1e-3), "fp32": (1e-4, 1e-5), "fp16": (5e-3, 5e-4)}


def to_device(w):
    dev = torch.device("cuda:0")

    def f(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if w.dtype == "bf16":
            t = t.view(torch.int16).view(torch.bfloat16)
        elif w.dtype == "fp16":
            t = t.view(torch.int16).view(torch.float16)
        return t.to(dev)

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32)).to(dev)

    return dict(q=f(w.q), k_cache=f(w.k_cache), v_cache=f(w.v_cache), tree_k=f(w.tree_k),
                tree_v=f(w.tree_v), parent=i32(w.parent), cu_prefix=i32(w.cu_prefix),
                cu_nodes=i32(w.cu_nodes), draft_tok=i32(w.draft_tok),
                target_argmax=i32(w.target_argmax))


def run_attention(w, t=None, max_prefix=None, max_nodes=None):
    t = t or to_device(w)
    st = torch.zeros(1, dtype=torch.int32, device="cuda:0")
    out, lse = api.tree_verify_attn_varlen(
        t["q"], t["k_cache"], t["v_cache"], t["tree_k"], t["tree_v"], t["parent"], t["cu_prefix"],
        t["cu_nodes"], max_prefix if max_prefix is not None else max(1, int(w.prefix_lens.max())),
        max_nodes if max_nodes is not None else int(w.tree_sizes.max()), dev_status=st)
    torch.cuda.synchronize()
    return out.double().cpu().numpy(), lse.double().cpu().numpy(), int(st.item())


def oracle_attention(w):
    return oracle.tree_verify_attention(w.f64("q"), w.f64("k_cache"), w.f64("v_cache"), w.cu_prefix,
                                        w.f64("tree_k"), w.f64("tree_v"), w.parent, w.cu_nodes,
                                        w.num_kv_heads, w.softmax_scale)


def assert_close(w, out, lse, o_ref, l_ref, where=""):
    ta, tl = TOL[w.dtype]
    err = np.abs(out - o_ref)
    lerr = np.abs(lse - l_ref) / np.maximum(np.abs(l_ref), 1.0)
    assert np.all(np.isfinite(out)) and np.all(np.isfinite(lse)), where
    assert err.max() <= ta, f"{where}: max-abs(out) {err.max():.3e} > {ta} at {np.unravel_index(err.argmax(), err.shape)}"
    assert lerr.max() <= tl, f"{where}: rel(lse) {lerr.max():.3e} > {tl} at {np.unravel_index(lerr.argmax(), lerr.shape)}"
    return float(err.max()), float(lerr.max())


def sample_rows(w, k, seed=0):
    """k (node, head) rows spread over every sequence, including first/last nodes/heads."""
    rng = np.random.default_rng(seed)
    rows = set()
    for b in range(w.batch):
        n0, n1 = int(w.cu_nodes[b]), int(w.cu_nodes[b + 1])
        if n1 > n0:
            rows.add((n0, 0))
            rows.add((n1 - 1, w.num_q_heads - 1))
    while len(rows) < k:
        rows.add((int(rng.integers(0, w.num_nodes)), int(rng.integers(0, w.num_q_heads))))
    return sorted(rows)
