"""Throughput of the tree-verification hot path on GB300.

One step = one pass of the whole path over one batch of synthetic inputs:
attention partials (prefix split-KV + masked tree tile), the log-sum-exp combine, and
the greedy acceptance walk.  Default workload: B=1, Hq=32, Hkv=8, d=128, bf16,
prefix 65536, 64-node best-first tree (width 4, depth <= 8).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--config C] [--impl ours|reference]

Prints one JSON line (rank 0).  `value` is tree nodes verified per second over all
ranks (each rank runs its own copy of the workload: weak scaling).  When a step's
inputs are more than 1.5 times the L2 size, the K timed steps run back to back between
one pair of CUDA events: each step streams inputs the L2 cannot hold (the previous
step's leave it long before they are read again).  The same steps are also timed one
at a time (each between its own events, after a GPU sleep of random length) and
reported under "isolated".  Smaller workloads are timed one step at a time with the L2
flushed (256 MiB write, outside the timed interval) before each.
`--impl reference` times the CPU oracle on the host cores instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "tree-verify attn nodes/s & prefix-KV GB/s (1×GB300), fraction of roofline"


def algorithmic_bytes(w):
    """Bytes the method must move (16-bit or fp32 storage): prefix K+V, tree K+V, Q, parent
    (read by the partials kernel) and out + lse (written by the combine)."""
    es = 4 if w.dtype == "fp32" else 2
    d, Hq, Hkv, N = w.head_dim, w.num_q_heads, w.num_kv_heads, w.num_nodes
    prefix_kv = int(w.cu_prefix[-1]) * Hkv * d * es * 2
    k1 = prefix_kv + N * Hkv * d * es * 2 + N * Hq * d * es + 4 * N
    total = k1 + N * Hq * d * es + N * Hq * 4
    return prefix_kv, k1, total


def algorithmic_flops(w):
    d, Hq = w.head_dim, w.num_q_heads
    from tree_verification_attention_gb300.workloads import tree_depths
    f = 0
    for b in range(w.batch):
        n0, n1 = int(w.cu_nodes[b]), int(w.cu_nodes[b + 1])
        P = int(w.cu_prefix[b + 1] - w.cu_prefix[b])
        depths = tree_depths(w.parent[n0:n1])
        f += 4 * d * Hq * ((n1 - n0) * P + int(depths.sum()))
    return f


def l2_streams(mode, input_bytes, l2_bytes):
    """Whether timed steps run without an L2 flush between them: forced by `mode`
    ("stream" / "flush"), or ("auto") when a step's inputs exceed 1.5x the L2, so that
    none of them can still be cached when the next step reads them."""
    if mode in ("stream", "flush"):
        return mode == "stream"
    return input_bytes > 3 * l2_bytes // 2


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return float(p["hbm_gbs"]), float(p["bf16_tflops"]), "measured"
    return 6800.0, 1900.0, "fallback"


PARTIALS_SOURCES = ("k_partials_tc.cu", "tc_pipeline.cuh", "tc_ptx.cuh", "tva_common.cuh", "tva_internal.h")


def kernel_source_hash():
    """Hash of the partials kernel's sources (the kernel whose DRAM traffic is recorded)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tree_verification_attention_gb300", "csrc")
    for f in PARTIALS_SOURCES:
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(workload_name):
    """DRAM bytes per launch of the partials kernel from the committed ncu summary, if it
    was taken on the current kernel sources (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    if not os.path.exists(path):
        return None
    src = kernel_source_hash()
    with open(path) as f:
        for line in f:
            parts = line.split()
            if len(parts) >= 3 and not line.startswith("#") and parts[0] == workload_name and parts[2] == src:
                return int(parts[1])
    return None


class ClockSampler:
    """nvidia-smi clock / throttle samples while the timed region runs."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
              "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
              "clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id):
        self.gpu_id = gpu_id
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu_id}", f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [x.strip() for x in ln.split(",")]
            if len(parts) != 7:
                continue
            try:
                sm.append(float(parts[0]))
                mx.append(float(parts[1]))
            except ValueError:
                continue
            for name, v in zip(names, parts[3:]):
                if v.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx), "reasons": sorted(reasons),
                "samples": len(sm)}


def max_over_ranks(values, device):
    """Element-wise maximum of `values` over the ranks of the default process group (the
    slowest rank sets each timing)."""
    import torch
    import torch.distributed as dist
    t = torch.tensor(values, dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t]


def dist_setup(n_gpus):
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world != n_gpus and world > 1:
        raise SystemExit(f"--gpus {n_gpus} but WORLD_SIZE={world}")
    return rank, world, local


def cpu_oracle_sample(w, kv_heads, repeats):
    """Oracle on the rows of the first `kv_heads` KV heads (all nodes), `repeats` times;
    returns (seconds per repeat, node-equivalents per repeat)."""
    import oracle
    G = w.num_q_heads // w.num_kv_heads
    k = kv_heads
    q = w.f64("q")[:, : G * k]
    kc = w.f64("k_cache")[:, :k]
    vc = w.f64("v_cache")[:, :k]
    tk = w.f64("tree_k")[:, :k]
    tv = w.f64("tree_v")[:, :k]
    t0 = time.perf_counter()
    for _ in range(repeats):
        oracle.tree_verify_attention(q, kc, vc, w.cu_prefix, tk, tv, w.parent, w.cu_nodes, k, w.softmax_scale)
        oracle.accept_longest_path(w.parent, w.draft_tok, w.target_argmax, w.cu_nodes)
    dt = (time.perf_counter() - t0) / repeats
    return dt, w.num_nodes * k / w.num_kv_heads


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def cpu_model():
    """The host CPU's model name (lscpu), or the machine type when lscpu has none."""
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for line in out.splitlines():
            if line.split(":")[0].strip() == "Model name":
                return line.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    import platform
    return platform.machine()


SINGLE_THREAD_ENV = ("OMP_NUM_THREADS", "OPENBLAS_NUM_THREADS", "MKL_NUM_THREADS", "BLIS_NUM_THREADS")


def single_thread_oracle(config):
    """The oracle's nodes/s on the same bounded sample with its BLAS limited to one
    thread (a child process, since BLAS reads the thread count when it loads)."""
    env = dict(os.environ, **{k: "1" for k in SINGLE_THREAD_ENV})
    code = ("import sys, json; sys.path.insert(0, %r); import bench; "
            "from tree_verification_attention_gb300 import workloads; "
            "w = workloads.make_workload(%d); bench.cpu_oracle_sample(w, 1, 1); "
            "dt, n = bench.cpu_oracle_sample(w, 1, 1); print(json.dumps([dt, n]))") % (ROOT, int(config))
    try:
        r = subprocess.run([sys.executable, "-c", code], env=env, capture_output=True, text=True, timeout=600)
        dt, n = json.loads(r.stdout.strip().splitlines()[-1])
    except (OSError, subprocess.SubprocessError, ValueError, IndexError):
        return None
    return {"value": n / dt, "unit": "nodes/s", "cores": 1, "seconds_per_sample": dt}


def run_reference(args, w, rank):
    if rank != 0:
        return
    # bounded sample: one KV head's rows (all nodes) per step; the node count is scaled by
    # the fraction of query heads covered so the unit stays nodes/s of the full problem
    for _ in range(args.warmup):
        cpu_oracle_sample(w, 1, 1)
    times = []
    for _ in range(args.steps):
        dt, nodes = cpu_oracle_sample(w, 1, 1)
        times.append(dt)
    sec = float(np.mean(times))
    value = nodes / sec
    sample = (f"oracle (float64 numpy) on all {w.num_nodes} nodes x the {w.num_q_heads // w.num_kv_heads} "
              f"query heads of 1 of {w.num_kv_heads} KV heads per step, + acceptance walk")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "nodes/s", "n_gpus": args.gpus,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": sec * 1e3, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "batch": w.batch, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "prefix_len": [int(x) for x in w.prefix_lens][:8], "tree_nodes": int(w.tree_sizes.max())},
        "cpu_baseline": {"value": value, "unit": "nodes/s", "cores": cpu_cores(), "kind": "oracle",
                         "cpu_model": cpu_model(), "sample": sample},
        "e2e": {"value": value, "unit": "nodes/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--l2", default="auto", choices=["auto", "flush", "stream"],
                    help="between timed steps: flush the L2, or not (inputs larger than it); "
                         "auto streams when the inputs exceed 1.5x the L2 size")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="rough budget of host-core seconds for the cpu_baseline sample")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank, world, local = dist_setup(args.gpus)
    from tree_verification_attention_gb300 import workloads
    w = workloads.make_workload(args.config)

    if args.impl == "reference":
        if world > 1:
            import torch.distributed as dist
            dist.init_process_group("gloo")
            if rank == 0:
                run_reference(args, w, rank)
            dist.barrier()
            dist.destroy_process_group()
        else:
            run_reference(args, w, rank)
        return

    import torch
    import __graft_entry__
    __graft_entry__.build()
    from tree_verification_attention_gb300 import api

    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)

    # ---- device-resident inputs
    def f(a):
        t = torch.from_numpy(np.ascontiguousarray(a))
        if w.dtype == "bf16":
            t = t.view(torch.int16).view(torch.bfloat16)
        elif w.dtype == "fp16":
            t = t.view(torch.int16).view(torch.float16)
        return t

    def i32(a):
        return torch.from_numpy(np.ascontiguousarray(a, dtype=np.int32))

    host = dict(q=f(w.q), k_cache=f(w.k_cache), v_cache=f(w.v_cache), tree_k=f(w.tree_k),
                tree_v=f(w.tree_v), parent=i32(w.parent), cu_prefix=i32(w.cu_prefix),
                cu_nodes=i32(w.cu_nodes), draft_tok=i32(w.draft_tok), target_argmax=i32(w.target_argmax))
    d = {k: v.to(dev) for k, v in host.items()}
    max_prefix = int(w.prefix_lens.max())
    max_nodes = int(w.tree_sizes.max())
    params = api.make_params(d["q"], d["k_cache"], d["cu_prefix"], d["cu_nodes"], w.num_kv_heads,
                             max_prefix, max_nodes)
    ws = api.alloc_workspace(params, dev)
    status = torch.zeros(1, dtype=torch.int32, device=dev)
    out = torch.empty_like(d["q"])
    lse = torch.empty(d["q"].shape[:2], dtype=torch.float32, device=dev)
    B, N = w.batch, w.num_nodes
    alen = torch.empty(B, dtype=torch.int32, device=dev)
    apath = torch.empty(N, dtype=torch.int32, device=dev)
    nxt = torch.empty(B, dtype=torch.int32, device=dev)
    flush = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
    l2_bytes = int(getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0) or (126 << 20))
    input_bytes = algorithmic_bytes(w)[1]
    stream_l2 = l2_streams(args.l2, input_bytes, l2_bytes)
    dither = np.random.default_rng(12345)

    def between_steps(i):
        """Untimed: flush the L2 (unless the inputs are larger than it) and a short
        random sleep."""
        if not stream_l2:
            flush.fill_(i & 0xFF)
        torch.cuda._sleep(int(dither.integers(0, 8192)))
    stream = torch.cuda.current_stream()

    def step(src):
        """The partials kernel alone (for the roofline figure)."""
        api.tree_verify_attn_partials(src["q"], src["k_cache"], src["v_cache"], src["tree_k"], src["tree_v"],
                                      src["parent"], src["cu_prefix"], src["cu_nodes"], max_prefix, max_nodes,
                                      ws, status, params=params)

    # A single sequence goes through the single-sequence entry point (prefix length and
    # node count passed by value, library-owned workspace); a batch through the varlen one.
    single = B == 1

    def attn(src):
        if single:
            api.tree_verify_attn(src["q"], src["k_cache"], src["v_cache"], src["tree_k"], src["tree_v"],
                                 src["parent"], out=out, lse=lse)
        else:
            step(src)
            api.tree_verify_attn_combine(params, ws, out, lse, status)

    def accept(src):
        api.accept_longest_path(src["cu_nodes"], src["parent"], src["draft_tok"], src["target_argmax"],
                                alen, apath, nxt, status)

    def device_status():
        st = int(status.item())
        return st if st != 0 or not single else api.read_device_status()

    for _ in range(args.warmup):
        attn(d)
        accept(d)
    torch.cuda.synchronize()
    if device_status() != 0:
        raise SystemExit(f"device status {device_status()} during warm-up")

    K = args.steps
    gpu_id = "GPU-" + str(torch.cuda.get_device_properties(dev).uuid) if hasattr(
        torch.cuda.get_device_properties(dev), "uuid") else str(local)
    sampler = ClockSampler(gpu_id)

    def timed(fn, offset):
        """Mean milliseconds per call of `fn` over K calls.  When the inputs exceed 1.5x
        the L2 the K calls run back to back between one pair of CUDA events (nothing of
        one call's inputs is still cached when the next reads them); otherwise each
        call has its own event pair, preceded by an untimed L2 flush.  Returns (mean ms,
        per-call isolated ms or None)."""
        torch.cuda._sleep(int(20e6))   # the host enqueues ahead of the GPU: no launch gaps
        if stream_l2:
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(K):
                fn()
            e1.record(stream)
            # the same calls one at a time, each between its own events after a random
            # GPU sleep (so each pays its own launch latency): reported beside the mean
            evi = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
            for i in range(K):
                between_steps(i + offset)
                evi[i][0].record(stream)
                fn()
                evi[i][1].record(stream)
            torch.cuda.synchronize()
            return e0.elapsed_time(e1) / K, float(np.mean([a.elapsed_time(b) for a, b in evi]))
        evi = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
        for i in range(K):
            between_steps(i + offset)
            evi[i][0].record(stream)
            fn()
            evi[i][1].record(stream)
        torch.cuda.synchronize()
        return float(np.mean([a.elapsed_time(b) for a, b in evi])), None

    if world > 1:
        dist.barrier()
    torch.cuda.synchronize()
    sampler.start()
    time.sleep(0.3)
    # Whole steps (partials, combine, acceptance); nothing separates the kernels of a step.
    ms, ms_iso = timed(lambda: (attn(d), accept(d)), 0)
    # The attention alone (partials + combine), and the dominant kernel alone (partials).
    att_ms, att_iso = timed(lambda: attn(d), 3)
    k1, k1_iso = timed(lambda: step(d), 7)
    # The CTA-pair partials kernel (a diagnostic selection of the library: cta_group::2,
    # M = 256, each SM loading half of every K/V tile), timed the same way for comparison
    # where the library applies it (two-M-tile row groups at head_dim 128, 16-bit types).
    workers_default = api.num_workers(params)
    api.diag_use_cta_pair(True)
    pair_applies = api.num_workers(params) != workers_default   # the pair runs one worker per two SMs
    api.diag_use_cta_pair(False)
    pair_ms = pair_iso = None
    if pair_applies:
        api.diag_use_cta_pair(True)
        try:
            for _ in range(args.warmup):
                step(d)
            pair_ms, pair_iso = timed(lambda: step(d), 11)
        finally:
            api.diag_use_cta_pair(False)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    clocks = sampler.stop()
    if world > 1:
        ms, att_ms, k1 = max_over_ranks([ms, att_ms, k1], dev)

    # ---- KV commit of the accepted path (a "next" row, measured on its own, outside the
    # step): the step's own acceptance result, appended to a reserved cache region.
    room = int(w.tree_sizes.max())
    k_dst = torch.zeros((B * room,) + tuple(d["k_cache"].shape[1:]), dtype=d["k_cache"].dtype, device=dev)
    v_dst = torch.zeros_like(k_dst)
    dst_row = torch.arange(0, B * room, room, dtype=torch.int32, device=dev)

    def commit():
        api.commit_accepted_kv(d["cu_nodes"], alen, apath, d["tree_k"], d["tree_v"], dst_row, k_dst, v_dst,
                               max_nodes=max_nodes, dev_status=status)

    accept(d)
    for _ in range(args.warmup):
        commit()
    torch.cuda.synchronize()
    evc = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda._sleep(int(20e6))
    for i in range(K):
        flush.fill_((i + 3) & 0xFF)
        torch.cuda._sleep(int(dither.integers(0, 8192)))
        evc[i][0].record(stream)
        commit()
        evc[i][1].record(stream)
    torch.cuda.synchronize()
    commit_ms = float(np.mean([evc[i][0].elapsed_time(evc[i][1]) for i in range(K)]))
    committed_rows = int(alen.sum().item())
    commit_bytes = 2 * 2 * committed_rows * w.num_kv_heads * w.head_dim * (4 if w.dtype == "fp32" else 2)

    # ---- stochastic chain verification (a "next" row, measured on its own): 8 chains of
    # 8 drafts over a 128256-token vocabulary.
    sp = [torch.from_numpy(x).to(dev) for x in workloads.make_chain_sampling_case(8, 8, 128256)]

    def sample():
        return api.verify_chain_sampling(sp[5], sp[0], sp[1], sp[2], sp[3], sp[4], max_draft=8, dev_status=status)

    for _ in range(args.warmup):
        sample()
    torch.cuda.synchronize()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda._sleep(int(20e6))
    for i in range(K):
        flush.fill_((i + 5) & 0xFF)
        torch.cuda._sleep(int(dither.integers(0, 8192)))
        evs[i][0].record(stream)
        s_alen, _ = sample()
        evs[i][1].record(stream)
    torch.cuda.synchronize()
    sample_ms = float(np.mean([evs[i][0].elapsed_time(evs[i][1]) for i in range(K)]))
    rows_read = int((2 - (s_alen == 8).int()).sum().item())   # residual: p and q rows; bonus: p row
    sample_bytes = rows_read * 128256 * 4 + 8 * 8 * 16

    # ---- Gated DeltaNet tree verification (a "next" row, measured on its own): the same
    # tree shape family, 32 heads of d = 128, fp32 state.
    gc = workloads.make_gdn_case(batch=1, heads=32, d=128, m=64, tree="best_first")
    gt = {n: torch.from_numpy(x).to(dev) for n, x in gc.items()}
    g_out = torch.empty_like(gt["v"])

    def gdn():
        api.gdn_tree_verify(gt["cu_nodes"], gt["parent"], gt["q"], gt["k"], gt["v"], gt["beta"], gt["alpha"],
                            gt["S0"], out=g_out, max_nodes=64, dev_status=status)

    for _ in range(args.warmup):
        gdn()
    torch.cuda.synchronize()
    evg = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(K)]
    torch.cuda._sleep(int(20e6))
    for i in range(K):
        flush.fill_((i + 11) & 0xFF)
        torch.cuda._sleep(int(dither.integers(0, 8192)))
        evg[i][0].record(stream)
        gdn()
        evg[i][1].record(stream)
    torch.cuda.synchronize()
    gdn_ms = float(np.mean([evg[i][0].elapsed_time(evg[i][1]) for i in range(K)]))
    gdn_bytes = sum(x.nbytes for n, x in gc.items() if n not in ("parent", "cu_nodes")) + g_out.numel() * 4
    # the same shape with bf16 q / k / v / out (fp32 state, gates and arithmetic)
    gb = {n: (torch.from_numpy(x).to(dev).to(torch.bfloat16) if n in ("q", "k", "v") else torch.from_numpy(x).to(dev))
          for n, x in workloads.make_gdn_case(batch=1, heads=32, d=128, m=64, tree="best_first", dtype="bf16").items()}
    gb_out = torch.empty_like(gb["v"])

    def gdn_bf16():
        api.gdn_tree_verify(gb["cu_nodes"], gb["parent"], gb["q"], gb["k"], gb["v"], gb["beta"], gb["alpha"],
                            gb["S0"], out=gb_out, max_nodes=64, dev_status=status)

    for _ in range(args.warmup):
        gdn_bf16()
    torch.cuda.synchronize()
    torch.cuda._sleep(int(20e6))
    for i in range(K):
        flush.fill_((i + 13) & 0xFF)
        torch.cuda._sleep(int(dither.integers(0, 8192)))
        evg[i][0].record(stream)
        gdn_bf16()
        evg[i][1].record(stream)
    torch.cuda.synchronize()
    gdn16_ms = float(np.mean([evg[i][0].elapsed_time(evg[i][1]) for i in range(K)]))
    gdn16_bytes = sum(x.numel() * x.element_size() for n, x in gb.items() if n not in ("parent", "cu_nodes")) + \
        gb_out.numel() * 2

    # ---- end to end through the public API from pinned host buffers.  A step's inputs
    # are staged back to back in one pinned buffer and copied up in one transfer, and its
    # results are written into one device buffer and read back in one transfer, as a
    # serving loop stages them (a dozen separate small copies cost ~30 us of fixed
    # per-copy latency on their own).
    def packed(shapes, device):
        """One buffer holding tensors of the given shapes and dtypes back to back (256-byte
        aligned); returns the buffer, views of it by name, and the payload bytes."""
        offs, total = {}, 0
        for k, (shape, dt) in shapes.items():
            nb = int(np.prod(shape)) * torch.empty(0, dtype=dt).element_size()
            offs[k] = (total, nb)
            total += (nb + 255) // 256 * 256
        buf = torch.empty(max(total, 256), dtype=torch.uint8, device=device)
        if device == "cpu":
            buf = buf.pin_memory()
        views = {k: buf[o:o + nb].view(shapes[k][1]).view(shapes[k][0]) for k, (o, nb) in offs.items()}
        return buf, views, sum(nb for _, nb in offs.values())

    in_shapes = {k: (tuple(v.shape), v.dtype) for k, v in host.items()}
    h_in, h_in_v, h2d = packed(in_shapes, "cpu")
    for k, v in host.items():
        h_in_v[k].copy_(v)
    d_in, d_in_v, _ = packed(in_shapes, dev)
    res_shapes = {"out": (tuple(out.shape), out.dtype), "lse": (tuple(lse.shape), torch.float32),
                  "alen": ((B,), torch.int32), "apath": ((N,), torch.int32), "nxt": ((B,), torch.int32)}
    d_res, d_res_v, d2h = packed(res_shapes, dev)
    h_res, _, _ = packed(res_shapes, "cpu")

    def e2e_params(src):
        return api.make_params(src["q"], src["k_cache"], src["cu_prefix"], src["cu_nodes"], w.num_kv_heads,
                               max_prefix, max_nodes)

    def e2e_step(d_buf, h_buf, src, prm):
        d_buf.copy_(h_buf, non_blocking=True)
        if single:
            api.tree_verify_attn(src["q"], src["k_cache"], src["v_cache"], src["tree_k"], src["tree_v"],
                                 src["parent"], out=d_res_v["out"], lse=d_res_v["lse"])
        else:
            api.tree_verify_attn_partials(src["q"], src["k_cache"], src["v_cache"], src["tree_k"], src["tree_v"],
                                          src["parent"], src["cu_prefix"], src["cu_nodes"], max_prefix, max_nodes,
                                          ws, status, params=prm)
            api.tree_verify_attn_combine(prm, ws, d_res_v["out"], d_res_v["lse"], status)
        api.accept_longest_path(src["cu_nodes"], src["parent"], src["draft_tok"], src["target_argmax"],
                                d_res_v["alen"], d_res_v["apath"], d_res_v["nxt"], status)
        h_res.copy_(d_res, non_blocking=True)

    def e2e_time(d_buf, h_buf, src):
        prm = e2e_params(src)
        for _ in range(args.warmup):
            e2e_step(d_buf, h_buf, src, prm)
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        torch.cuda._sleep(int(20e6))
        e0.record(stream)
        for _ in range(Ke):
            e2e_step(d_buf, h_buf, src, prm)
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / Ke

    Ke = max(3, K // 2)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e2e_ms = e2e_time(d_in, h_in, d_in_v)
    # The same step with the prefix K/V cache resident in HBM (as it is across the steps
    # of a serving loop: the cache holds what earlier steps committed), copying up only
    # the draft tree's inputs - q, the tree's K/V, parent ids, draft and target tokens,
    # the cu arrays - and reading back the same results.  Reported beside e2e, which
    # copies the cache too.
    resident = ("k_cache", "v_cache")
    tree_shapes = {k: v for k, v in in_shapes.items() if k not in resident}
    h_tr, h_tr_v, h2d_tree = packed(tree_shapes, "cpu")
    for k in tree_shapes:
        h_tr_v[k].copy_(host[k])
    d_tr, d_tr_v, _ = packed(tree_shapes, dev)
    e2e_tree_ms = e2e_time(d_tr, h_tr, dict(d_tr_v, k_cache=d_in_v["k_cache"], v_cache=d_in_v["v_cache"]))
    if not torch.equal(h_res, d_res.cpu()):
        raise SystemExit("end-to-end results read back differ from the device copy")
    # What the host link itself gives: the step's two large inputs copied from pinned
    # memory in one transfer of the same total size, on the same stream.
    big = torch.empty(h2d, dtype=torch.uint8).pin_memory()
    big_d = torch.empty(h2d, dtype=torch.uint8, device=dev)
    big_d.copy_(big, non_blocking=True)
    torch.cuda.synchronize()
    e0.record(stream)
    for _ in range(Ke):
        big_d.copy_(big, non_blocking=True)
    e1.record(stream)
    torch.cuda.synchronize()
    h2d_one_copy_gbs = h2d / (e0.elapsed_time(e1) / Ke * 1e-3) / 1e9
    del big, big_d
    if world > 1:
        (e2e_ms, e2e_tree_ms) = max_over_ranks([e2e_ms, e2e_tree_ms], dev)
    if device_status() != 0:
        raise SystemExit(f"device status {device_status()}")

    # ---- CPU oracle baseline (rank 0 only), bounded sample
    cpu = None
    if rank == 0:
        dt1, nodes1 = cpu_oracle_sample(w, 1, 1)
        reps = max(1, min(20, int(args.cpu_seconds / max(dt1, 1e-3))))
        dt, nodes = cpu_oracle_sample(w, 1, reps)
        cpu = {"value": nodes / dt, "unit": "nodes/s", "cores": cpu_cores(), "kind": "oracle",
               "cpu_model": cpu_model(),
               "sample": f"{reps}x: all {w.num_nodes} nodes x the {w.num_q_heads // w.num_kv_heads} query heads "
                         f"of 1 of {w.num_kv_heads} KV heads (node count scaled by 1/{w.num_kv_heads}), "
                         f"float64 numpy, + acceptance walk"}
        if args.cpu_seconds > 0.5:
            cpu["single_thread"] = single_thread_oracle(args.config)

    if world > 1:
        dist.barrier()
        dist.destroy_process_group()
    if rank != 0:
        return

    hbm_peak, tc_peak, peak_kind = load_peaks()
    prefix_kv, k1_bytes, total_bytes = algorithmic_bytes(w)
    flops = algorithmic_flops(w)
    k1_gbs = k1_bytes / (k1 * 1e-3) / 1e9
    roof_s = max(total_bytes / (hbm_peak * 1e9), flops / (tc_peak * 1e12))
    l2_note = (f"not flushed: the {input_bytes / 1e6:.0f} MB of inputs each step streams exceed 1.5x the "
               f"{l2_bytes / 1e6:.0f} MB L2, so the K steps run back to back between one event pair" if stream_l2 else
               "flushed before every timed step (256 MiB write, untimed); one event pair per step")
    traffic = recorded_traffic(w.name)
    # The partials kernel's own bound: the slower of its bytes at the HBM peak and its
    # FLOPs at the bf16 tensor peak (the burst figure: the kernel is timed alone).
    tensor_bound = flops / (tc_peak * 1e12) > k1_bytes / (hbm_peak * 1e9)
    roofline_obj = {"bound": "tensor" if tensor_bound else "hbm",
                    "kernel": "partials (prefix split-KV + tree tile)",
                    "traffic": traffic, "algorithmic_bytes": k1_bytes, "algorithmic_flops": flops,
                    "us_per_launch": k1 * 1e3,
                    "us_per_launch_isolated": None if k1_iso is None else k1_iso * 1e3,
                    "timed": f"{K} launches of the partials kernel alone, " + l2_note}
    if tensor_bound:
        k1_tf = flops / (k1 * 1e-3) / 1e12
        roofline_obj.update({"achieved": k1_tf, "peak": tc_peak, "unit": "TFLOP/s", "frac": k1_tf / tc_peak,
                             "peak_kind": f"{peak_kind} bf16_tflops (burst)"})
    else:
        roofline_obj.update({"achieved": k1_gbs, "peak": hbm_peak, "unit": "GB/s", "frac": k1_gbs / hbm_peak,
                             "peak_kind": f"{peak_kind} hbm_gbs"})
    line = {
        "metric": METRIC,
        "value": world * N / (ms * 1e-3),
        "unit": "nodes/s",
        "n_gpus": world,
        "steps": K,
        "warmup": args.warmup,
        "ms_per_step": ms,
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {"workload": w.name, "batch": B, "num_q_heads": w.num_q_heads,
                   "num_kv_heads": w.num_kv_heads, "head_dim": w.head_dim,
                   "prefix_len": [int(x) for x in w.prefix_lens][:8], "tree_nodes": int(w.tree_sizes.max()),
                   "seed": w.seed, "parallelism": f"replicas x{world}",
                   "api": "tree_verify_attn + accept_longest_path" if single
                          else "tree_verify_attn_partials + _combine + accept_longest_path",
                   "l2": l2_note},
        "prefix_kv_gbs": prefix_kv / (ms * 1e-3) / 1e9,
        "step_roofline_frac": roof_s / (ms * 1e-3),
        "attention_us": att_ms * 1e3,
        "attention_roofline_frac": roof_s / (att_ms * 1e-3),
        "isolated": None if ms_iso is None else {
            "step_us": ms_iso * 1e3, "attention_us": att_iso * 1e3, "partials_us": k1_iso * 1e3,
            "step_roofline_frac": roof_s / (ms_iso * 1e-3), "attention_roofline_frac": roof_s / (att_iso * 1e-3),
            "timed": f"{K} calls one at a time, each between its own events after a random GPU sleep"},
        "roofline": roofline_obj,
        "cta_pair_partials": None if pair_ms is None else {
            "kernel": "partials on CTA pairs (cta_group::2, M = 256; tva_diag_use_cta_pair), not the default",
            "us_per_launch": pair_ms * 1e3,
            "us_per_launch_isolated": None if pair_iso is None else pair_iso * 1e3,
            "frac": ((flops / (pair_ms * 1e-3) / 1e12) / tc_peak if tensor_bound
                     else (k1_bytes / (pair_ms * 1e-3) / 1e9) / hbm_peak),
            "timed": "as roofline"},
        "cpu_baseline": cpu,
        "e2e": {"value": world * N / (e2e_ms * 1e-3), "unit": "nodes/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": e2e_ms,
                "h2d_gbs_in_step": h2d / (e2e_ms * 1e-3) / 1e9,
                "h2d_gbs_one_pinned_copy": h2d_one_copy_gbs},
        "e2e_resident_cache": {"value": world * N / (e2e_tree_ms * 1e-3), "unit": "nodes/s",
                               "h2d_bytes_per_step": h2d_tree, "d2h_bytes_per_step": d2h,
                               "ms_per_step": e2e_tree_ms,
                               "note": "prefix K/V cache resident in HBM; each step copies up the draft "
                                       "tree's inputs only"},
        "kv_commit": {"us_per_launch": commit_ms * 1e3, "rows": committed_rows, "bytes": commit_bytes,
                      "gbs": commit_bytes / (commit_ms * 1e-3) / 1e9,
                      "timed": f"{K} launches alone (not in the step), L2 flushed before each"},
        "chain_sampling": {"workload": "B=8 chains, gamma=8, V=128256, fp32 p/q", "us_per_launch": sample_ms * 1e3,
                           "bytes": sample_bytes, "gbs": sample_bytes / (sample_ms * 1e-3) / 1e9,
                           "timed": f"{K} launches alone (not in the step), L2 flushed before each"},
        "gdn_tree_bf16": {"workload": "B=1, H=32, d=128, 64-node best-first tree, bf16 q/k/v/out, fp32 state",
                          "us_per_launch": gdn16_ms * 1e3, "bytes": gdn16_bytes,
                          "gbs": gdn16_bytes / (gdn16_ms * 1e-3) / 1e9,
                          "timed": f"{K} launches alone (not in the step), L2 flushed before each"},
        "gdn_tree": {"workload": "B=1, H=32, d=128, 64-node best-first tree, fp32", "us_per_launch": gdn_ms * 1e3,
                     "bytes": gdn_bytes, "gbs": gdn_bytes / (gdn_ms * 1e-3) / 1e9,
                     "timed": f"{K} launches alone (not in the step), L2 flushed before each"},
        # this library's kernels in the timed region: steps (3 each), attention (2), partials (1);
        # with streamed inputs each is timed back to back and once more one call at a time
        "gpu_launches": ((12 if stream_l2 else 6) + (0 if pair_ms is None else (2 if stream_l2 else 1))) * K,
        "clocks": clocks,
    }
    print(json.dumps(line), flush=True)


if __name__ == "__main__":
    main()
