"""Seeded synthetic inputs for tree-verification attention and greedy acceptance.

This module only *draws* inputs: tree shapes, token ids and Gaussian Q/K/V values,
rounded once to the storage precision.  It holds none of the attention, merge or
acceptance arithmetic, so both the CPU oracle (through the tests and the bench's CPU
baseline) and the CUDA path consume exactly the same bytes.

Shapes follow the five workloads this library is measured on (all sizes are the
defaults of :func:`make_workload`):

1. tiny fp32 case: B=1, Hq=4, Hkv=1, d=64, prefix 256, 8-node random tree;
2. Llama-3-8B-shaped chain: B=1, Hq=32, Hkv=8, d=128, prefix 16384, chain of 8,
   keys of the first half of the KV heads scaled x3 (peaked softmax);
3. long prefix with a best-first tree: prefix 65536, 64 nodes, width 4, depth <= 8;
4. ragged batch: B=8, prefix lengths uniform in [4096, 32768], 32-node random
   trees of depth <= 6;
5. large case: Hq=64, Hkv=8, prefix 131072, 128-node best-first tree of width 8 and
   depth <= 10, 1% of prefix keys scaled x4 (attention sinks).

The best-first tree follows the w-parallel variant of DySpec-style construction
described in the DFlash-TfM summary (gist.science 2607.06763, Method, "Tree
construction"): the top-w candidates of a score heap are expanded together.  Node ids
are given in creation order, so every parent precedes its children (the topological
order the same summary's verification section relies on).

Draw order from one ``numpy.random.Generator(PCG64(seed))``: prefix lengths, trees,
tokens, Q, K_cache, V_cache, tree K, tree V, then the scaling draws.  Values are drawn
as float32 and rounded to bfloat16 (round-to-nearest-even) exactly once.
"""
from __future__ import annotations

import heapq
import math
from dataclasses import dataclass, field

import numpy as np

__all__ = [
    "Workload",
    "make_workload",
    "bf16_round_bits",
    "bits_to_f64",
    "random_tree",
    "chain_tree",
    "depth_limited_tree",
    "best_first_tree",
    "beam_tree",
    "f16_round_bits",
    "f16_bits_to_f64",
    "tree_depths",
    "WORKLOAD_NAMES",
]

WORKLOAD_NAMES = {
    1: "tiny-fp32-P256-m8",
    2: "chain-bf16-P16384-m8-Hq32-Hkv8",
    3: "bestfirst-bf16-P65536-m64-Hq32-Hkv8",
    4: "ragged-bf16-B8-P4096..32768-m32-Hq32-Hkv8",
    5: "sinks-bf16-P131072-m128-Hq64-Hkv8",
    6: "beam-fp16-P32768-m68-Hq32-Hkv8",
}


# --------------------------------------------------------------------------- storage

def bf16_round_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to bfloat16 (nearest, ties to even); return the uint16 bits.

    Inputs are finite Gaussian draws, so NaN handling is not needed."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    u = x.view(np.uint32)
    # finite inputs stay below 0xFF800000 after the increment, so uint32 cannot wrap
    rounded = (u + np.uint32(0x7FFF) + ((u >> np.uint32(16)) & np.uint32(1))) >> np.uint32(16)
    return rounded.astype(np.uint16)


def bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of bfloat16 values given as uint16 bits."""
    return (bits.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def f16_round_bits(x: np.ndarray) -> np.ndarray:
    """Round float32 values to IEEE float16 (nearest, ties to even); return the uint16 bits."""
    return np.ascontiguousarray(x, dtype=np.float32).astype(np.float16).view(np.uint16)


def f16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact float64 value of float16 values given as uint16 bits."""
    return np.ascontiguousarray(bits).view(np.float16).astype(np.float64)


# --------------------------------------------------------------------------- trees

def random_tree(rng: np.random.Generator, m: int) -> np.ndarray:
    """parent[0] = -1 and parent[i] uniform over {-1, 0, ..., i-1}."""
    parent = np.empty(m, dtype=np.int32)
    for i in range(m):
        parent[i] = -1 if i == 0 else int(rng.integers(-1, i))
    return parent


def chain_tree(m: int) -> np.ndarray:
    """A linear draft of gamma = m tokens: parent[i] = i - 1."""
    return np.arange(-1, m - 1, dtype=np.int32)


def beam_tree(rng: np.random.Generator, widths) -> np.ndarray:
    """LongSpec's tree decoding shape ("Experiment details": dynamic beam search with
    beam widths [4, 16, 16, 16, 16] per speculative step; low-likelihood branches stay in
    the tree but are not expanded further).

    Step 1 keeps the widths[0] best children of the prefix end.  Step s keeps the
    widths[s] best of the candidates proposed by the previous step's nodes (each
    proposes widths[s] children), scored by cumulative log-likelihood, a candidate
    scoring its parent's score + log u, u ~ U(0, 1).  Nodes are numbered step by step
    (topological).  A node none of whose candidates survives is a leaf.  Returns parent
    ids (-1 for step-1 nodes), sum(widths) of them."""
    widths = [int(w) for w in widths]
    parent = [-1] * widths[0]
    score = list(np.sort(np.log(rng.random(widths[0])))[::-1])
    level = list(range(widths[0]))
    for w in widths[1:]:
        cand = []
        for node in level:
            for lu in np.log(rng.random(w)):
                cand.append((score[node] + float(lu), node))
        cand.sort(key=lambda c: -c[0])
        new_level = []
        for sc, par in cand[:w]:
            parent.append(par)
            score.append(sc)
            new_level.append(len(parent) - 1)
        level = new_level
    return np.asarray(parent, dtype=np.int32)


def tree_depths(parent: np.ndarray) -> np.ndarray:
    """Depth of every node (a child of the prefix end has depth 1); needs parent[i] < i."""
    depth = np.zeros(len(parent), dtype=np.int32)
    for i, p in enumerate(parent):
        depth[i] = 1 if p < 0 else depth[p] + 1
    return depth


def depth_limited_tree(rng: np.random.Generator, m: int, max_depth: int) -> np.ndarray:
    """parent[i] uniform over {-1} and the earlier nodes whose depth is below max_depth."""
    parent = np.empty(m, dtype=np.int32)
    depth = np.empty(m, dtype=np.int32)
    for i in range(m):
        cands = [-1] + [j for j in range(i) if depth[j] < max_depth]
        p = cands[int(rng.integers(0, len(cands)))]
        parent[i] = p
        depth[i] = 1 if p < 0 else depth[p] + 1
    return parent


def best_first_tree(rng: np.random.Generator, m: int, width: int, max_depth: int,
                    max_branch: int = 4) -> np.ndarray:
    """w-parallel best-first tree (DySpec-style construction as summarised for DFlash-TfM).

    Every node's score is its parent's score plus log(u), u ~ U(0, 1].  A max-heap holds
    the expandable nodes and starts with a virtual root at the prefix end (score 0,
    depth 0).  Each round pops the top ``width`` entries; a popped node whose depth is
    below ``max_depth`` receives U{1..max_branch} children.  Construction stops at m
    nodes, cutting the last round short in pop order.
    """
    parent: list[int] = []
    heap = [(-0.0, -1, 0)]  # (-score, node id, depth); ties broken by smaller id
    while len(parent) < m:
        if not heap:
            raise ValueError("best-first tree ran out of expandable nodes")
        popped = [heapq.heappop(heap) for _ in range(min(width, len(heap)))]
        for neg_score, node, depth in popped:
            if depth >= max_depth:
                continue
            nchild = int(rng.integers(1, max_branch + 1))
            for _ in range(nchild):
                if len(parent) == m:
                    break
                score = -neg_score + math.log(1.0 - float(rng.random()))
                child = len(parent)
                parent.append(node)
                heapq.heappush(heap, (-score, child, depth + 1))
            if len(parent) == m:
                break
    return np.asarray(parent, dtype=np.int32)


# --------------------------------------------------------------------------- workload

@dataclass
class Workload:
    """One batch of synthetic inputs.

    Layouts (row-major, contiguous):
      q          [N, Hq, d]        N = sum of tree sizes
      k_cache    [sum P_b, Hkv, d] sequence b occupies rows cu_prefix[b] .. cu_prefix[b+1]-1
      v_cache    [sum P_b, Hkv, d]
      tree_k     [N, Hkv, d]       node i of sequence b is row cu_nodes[b] + i
      tree_v     [N, Hkv, d]
      parent     [N] int32         local ids, -1 = child of the prefix end, parent[i] < i
      draft_tok  [N] int32
      target_argmax [N + B] int32  sequence b owns slots cu_nodes[b]+b .. cu_nodes[b+1]+b;
                                   its slot 0 is the target's greedy token at the prefix
                                   end and slot i+1 the one after node i
    Floating-point arrays hold uint16 bfloat16 bits when ``dtype == "bf16"`` and float32
    values when ``dtype == "fp32"``.
    """
    name: str
    dtype: str
    num_q_heads: int
    num_kv_heads: int
    head_dim: int
    cu_prefix: np.ndarray
    cu_nodes: np.ndarray
    parent: np.ndarray
    draft_tok: np.ndarray
    target_argmax: np.ndarray
    q: np.ndarray
    k_cache: np.ndarray
    v_cache: np.ndarray
    tree_k: np.ndarray
    tree_v: np.ndarray
    softmax_scale: float
    seed: int
    meta: dict = field(default_factory=dict)

    @property
    def batch(self) -> int:
        return len(self.cu_prefix) - 1

    @property
    def num_nodes(self) -> int:
        return int(self.cu_nodes[-1])

    @property
    def prefix_lens(self) -> np.ndarray:
        return np.diff(self.cu_prefix)

    @property
    def tree_sizes(self) -> np.ndarray:
        return np.diff(self.cu_nodes)

    def f64(self, name: str) -> np.ndarray:
        """The exact float64 value of a floating-point input, as the kernels see it."""
        a = getattr(self, name)
        if self.dtype == "bf16":
            return bits_to_f64(a)
        if self.dtype == "fp16":
            return f16_bits_to_f64(a)
        return a.astype(np.float64)


_DEFAULTS = {
    1: dict(batch=1, Hq=4, Hkv=1, d=64, prefix=256, m=8, tree="random", dtype="fp32",
            vocab=32),
    6: dict(batch=1, Hq=32, Hkv=8, d=128, prefix=32768, m=68, tree="beam", widths=(4, 16, 16, 16, 16),
            dtype="fp16", vocab=32000),
    2: dict(batch=1, Hq=32, Hkv=8, d=128, prefix=16384, m=8, tree="chain", dtype="bf16",
            vocab=32000, k_scale_half_heads=3.0),
    3: dict(batch=1, Hq=32, Hkv=8, d=128, prefix=65536, m=64, tree="best_first", width=4,
            max_depth=8, dtype="bf16", vocab=32000),
    4: dict(batch=8, Hq=32, Hkv=8, d=128, prefix=(4096, 32768), m=32, tree="depth_limited",
            max_depth=6, dtype="bf16", vocab=32000),
    5: dict(batch=1, Hq=64, Hkv=8, d=128, prefix=131072, m=128, tree="best_first", width=8,
            max_depth=10, dtype="bf16", vocab=32000, sink_frac=0.01, sink_scale=4.0),
}


def workload_defaults(config: int) -> dict:
    return dict(_DEFAULTS[config])


def make_workload(config: int, seed: int | None = None, **overrides) -> Workload:
    """Draw the inputs of workload ``config`` (1..5); keyword overrides change sizes.

    ``prefix`` is an int (every sequence) or an inclusive (lo, hi) range drawn per
    sequence; ``m`` is the tree size of every sequence.  ``p_match`` (default 0.7) is
    the probability that a draft token equals the target's greedy token at its parent.
    """
    spec = workload_defaults(config)
    spec.update(overrides)
    if seed is None:
        seed = 1000 + config
    rng = np.random.Generator(np.random.PCG64(seed))
    B, Hq, Hkv, d, m = spec["batch"], spec["Hq"], spec["Hkv"], spec["d"], spec["m"]
    if Hq % Hkv:
        raise ValueError("Hq must be a multiple of Hkv")

    # 1. prefix lengths
    pre = spec["prefix"]
    if isinstance(pre, (tuple, list)):
        plens = rng.integers(pre[0], pre[1], endpoint=True, size=B).astype(np.int64)
    else:
        plens = np.full(B, int(pre), dtype=np.int64)
    ms = np.full(B, int(m), dtype=np.int64)
    cu_prefix = np.concatenate([[0], np.cumsum(plens)]).astype(np.int32)
    cu_nodes = np.concatenate([[0], np.cumsum(ms)]).astype(np.int32)

    # 2. trees
    parents = []
    for b in range(B):
        kind = spec["tree"]
        if kind == "random":
            parents.append(random_tree(rng, int(ms[b])))
        elif kind == "chain":
            parents.append(chain_tree(int(ms[b])))
        elif kind == "depth_limited":
            parents.append(depth_limited_tree(rng, int(ms[b]), spec["max_depth"]))
        elif kind == "best_first":
            parents.append(best_first_tree(rng, int(ms[b]), spec["width"], spec["max_depth"]))
        elif kind == "beam":
            par = beam_tree(rng, spec["widths"])
            if len(par) != int(ms[b]):
                raise ValueError("a beam tree has sum(widths) nodes")
            parents.append(par)
        elif kind == "given":
            parents.append(np.asarray(spec["parent"][b], dtype=np.int32))
        else:
            raise ValueError(kind)
    parent = np.concatenate(parents).astype(np.int32) if parents else np.zeros(0, np.int32)

    # 3. tokens: target greedy tokens per slot, then draft tokens matching w.p. p_match
    vocab = spec["vocab"]
    p_match = spec.get("p_match", 0.7)
    tgts, drafts = [], []
    for b in range(B):
        mb = int(ms[b])
        tgt = rng.integers(0, vocab, size=mb + 1).astype(np.int32)
        par = parents[b]
        want = tgt[par + 1]
        u = rng.random(mb)
        alt = rng.integers(0, vocab - 1, size=mb).astype(np.int32)
        alt = alt + (alt >= want)  # uniform over the other vocab-1 tokens
        drafts.append(np.where(u < p_match, want, alt).astype(np.int32))
        tgts.append(tgt)
    target_argmax = np.concatenate(tgts).astype(np.int32)
    draft_tok = np.concatenate(drafts).astype(np.int32) if drafts else np.zeros(0, np.int32)

    # 4. Gaussian values, float32
    N = int(cu_nodes[-1])
    T = int(cu_prefix[-1])
    q = rng.standard_normal((N, Hq, d), dtype=np.float32)
    k_cache = rng.standard_normal((T, Hkv, d), dtype=np.float32)
    v_cache = rng.standard_normal((T, Hkv, d), dtype=np.float32)
    tree_k = rng.standard_normal((N, Hkv, d), dtype=np.float32)
    tree_v = rng.standard_normal((N, Hkv, d), dtype=np.float32)

    # 5. scalings (applied in float32 before the single rounding)
    if "k_scale_half_heads" in spec:
        s = np.float32(spec["k_scale_half_heads"])
        k_cache[:, : Hkv // 2, :] *= s
        tree_k[:, : Hkv // 2, :] *= s
    if "sink_frac" in spec:
        s = np.float32(spec["sink_scale"])
        for b in range(B):
            P = int(plens[b])
            nsink = int(round(spec["sink_frac"] * P))
            if nsink:
                pos = rng.choice(P, size=nsink, replace=False) + int(cu_prefix[b])
                k_cache[pos, :, :] *= s

    dtype = spec["dtype"]
    if dtype == "bf16":
        conv = bf16_round_bits
    elif dtype == "fp32":
        conv = lambda a: np.ascontiguousarray(a, dtype=np.float32)  # noqa: E731
    elif dtype == "fp16":
        conv = f16_round_bits
    else:
        raise ValueError(dtype)
    meta = {k: v for k, v in spec.items() if k not in ("parent",)}
    return Workload(
        name=spec.get("name", WORKLOAD_NAMES.get(config, f"config{config}")),
        dtype=dtype, num_q_heads=Hq, num_kv_heads=Hkv, head_dim=d,
        cu_prefix=cu_prefix, cu_nodes=cu_nodes, parent=parent, draft_tok=draft_tok,
        target_argmax=target_argmax,
        q=conv(q), k_cache=conv(k_cache), v_cache=conv(v_cache),
        tree_k=conv(tree_k), tree_v=conv(tree_v),
        softmax_scale=1.0 / math.sqrt(d), seed=seed, meta=meta)


def make_chain_sampling_case(batch: int = 8, gamma: int = 8, vocab: int = 128256, seed: int = 2002,
                             temperature: float = 3.0, overlap: float = 0.7):
    """Synthetic inputs for stochastic chain verification: per sequence gamma draft
    positions and gamma + 1 target positions over `vocab` tokens.

    q rows are softmax(z * temperature) of N(0, 1) logits (peaked, like a drafter at
    low temperature); the target rows at draft positions mix the draft row with an
    independent one (``overlap`` of the mass shared), the bonus row is independent.
    Draft tokens are drawn from their q rows; the uniforms are float32 in [0, 1).
    Returns (p [B*(gamma+1), V], q [B*gamma, V], draft [B*gamma], u_accept [B*gamma],
    u_sample [B], cu_draft [B+1]) as numpy arrays."""
    rng = np.random.default_rng(seed)

    def rows(n):
        z = rng.standard_normal((n, vocab)).astype(np.float32) * temperature
        z -= z.max(1, keepdims=True)
        e = np.exp(z, dtype=np.float32)
        return e / e.sum(1, keepdims=True, dtype=np.float32)

    q = rows(batch * gamma)
    p = rows(batch * (gamma + 1))
    for b in range(batch):
        for k in range(gamma):
            r = b * (gamma + 1) + k
            p[r] = overlap * q[b * gamma + k] + (1 - overlap) * p[r]
    cdf = np.cumsum(q.astype(np.float64), 1)
    cdf /= cdf[:, -1:]
    draft = np.array([np.searchsorted(cdf[i], rng.random(), side="right") for i in range(batch * gamma)],
                     dtype=np.int32)
    draft = np.minimum(draft, vocab - 1)
    u_accept = rng.random(batch * gamma).astype(np.float32)
    u_sample = rng.random(batch).astype(np.float32)
    cu_draft = np.arange(0, batch * gamma + 1, gamma, dtype=np.int32)
    return p.astype(np.float32), q.astype(np.float32), draft, u_accept, u_sample, cu_draft


def make_gdn_case(batch: int = 1, heads: int = 32, d: int = 128, m: int = 64, tree: str = "best_first",
                  seed: int = 3003, parents=None, dtype: str = "fp32"):
    """Synthetic inputs for Gated DeltaNet tree verification (fp32, or with dtype="bf16"
    q, k and v rounded once to bfloat16 - returned as float32 arrays holding exactly the
    bfloat16 values, so the same arrays feed the oracle and a bf16 device copy).

    q and k are L2-normalised per (node, head) as Gated DeltaNet layers normalise them;
    v ~ N(0, 1); beta = sigmoid(z) in (0, 1); alpha = exp(-0.1 softplus(z)) (decays
    near 1); the committed state S0 [B, H, d, d] is a sum of 32 random outer products
    k v^T scaled by 1/4 (a state that has absorbed some context).  Trees: best-first
    (width 4, depth <= 8), beam (LongSpec's widths), chain, or `parents` (a list of
    parent arrays).  Returns a dict of numpy arrays."""
    rng = np.random.default_rng(seed)
    if parents is None:
        parents = []
        for _ in range(batch):
            if tree == "best_first":
                parents.append(best_first_tree(rng, m, 4, 8))
            elif tree == "beam":
                parents.append(beam_tree(rng, (4, 16, 16, 16, 16))[:m])
            elif tree == "chain":
                parents.append(chain_tree(m))
            elif tree == "random":
                parents.append(random_tree(rng, m))
            else:
                raise ValueError(tree)
    sizes = [len(p) for p in parents]
    cu_nodes = np.concatenate([[0], np.cumsum(sizes)]).astype(np.int32)
    N = int(cu_nodes[-1])

    def unit(x):
        return (x / np.linalg.norm(x, axis=-1, keepdims=True)).astype(np.float32)

    q = unit(rng.standard_normal((N, heads, d)))
    k = unit(rng.standard_normal((N, heads, d)))
    v = rng.standard_normal((N, heads, d)).astype(np.float32)
    beta = (1 / (1 + np.exp(-rng.standard_normal((N, heads))))).astype(np.float32)
    alpha = np.exp(-0.1 * np.log1p(np.exp(rng.standard_normal((N, heads))))).astype(np.float32)
    ks = unit(rng.standard_normal((batch, heads, 32, d)))
    vs = rng.standard_normal((batch, heads, 32, d)).astype(np.float32)
    S0 = (0.25 * np.einsum("bhtk,bhtv->bhkv", ks, vs)).astype(np.float32)
    parent = np.concatenate(parents).astype(np.int32) if parents else np.zeros(0, np.int32)
    if dtype == "bf16":
        q, k, v = (bits_to_f64(bf16_round_bits(x)).astype(np.float32) for x in (q, k, v))
    elif dtype != "fp32":
        raise ValueError(dtype)
    return dict(q=q, k=k, v=v, beta=beta, alpha=alpha, S0=S0, parent=parent, cu_nodes=cu_nodes)
