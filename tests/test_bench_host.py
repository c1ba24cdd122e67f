"""bench.py's host-side accounting, checked without a GPU: the algorithmic bytes and
FLOPs of the roofline (the per-unit figures written out from their definition), the
choice of L2 handling between timed steps, the traffic record lookup and the JSON line
of the reference arm (the oracle on the host cores)."""
import json
import os
import subprocess
import sys

import numpy as np
import pytest

import bench
from tree_verification_attention_gb300 import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_algorithmic_bytes_of_the_64k_workload():
    w = workloads.make_workload(3)
    prefix_kv, k1, total = bench.algorithmic_bytes(w)
    # prefix K and V: 65536 keys x 8 KV heads x 128 x 2 bytes, twice
    assert prefix_kv == 65536 * 8 * 128 * 2 * 2
    # + tree K/V (64 nodes x 8 heads), Q (64 x 32 heads), parent ids
    assert k1 == prefix_kv + 64 * 8 * 128 * 2 * 2 + 64 * 32 * 128 * 2 + 4 * 64
    # + out (bf16) and lse (fp32)
    assert total == k1 + 64 * 32 * 128 * 2 + 64 * 32 * 4


def _anc_or_self_counts(parent):
    counts = []
    for i in range(len(parent)):
        c, j = 1, int(parent[i])
        while j >= 0:
            c += 1
            j = int(parent[j])
        counts.append(c)
    return np.array(counts)


@pytest.mark.parametrize("cfg", [2, 3, 4])
def test_algorithmic_flops_count_prefix_and_visible_tree_pairs(cfg):
    """4 d Hq per (row, visible key) pair: every node sees the whole prefix and its
    ancestors-and-self among the tree keys."""
    w = workloads.make_workload(cfg)
    d, Hq = w.head_dim, w.num_q_heads
    expect = 0
    for b in range(w.batch):
        n0, n1 = int(w.cu_nodes[b]), int(w.cu_nodes[b + 1])
        P = int(w.cu_prefix[b + 1] - w.cu_prefix[b])
        expect += 4 * d * Hq * ((n1 - n0) * P + int(_anc_or_self_counts(w.parent[n0:n1]).sum()))
    assert bench.algorithmic_flops(w) == expect
    if cfg == 2:  # an 8-node chain: node i sees i + 1 tree keys
        assert int(_anc_or_self_counts(w.parent).sum()) == 36


def test_l2_handling_choice():
    l2 = 136 << 20
    assert bench.l2_streams("auto", 269_222_144, l2)       # 64k prefix: 1.9x the L2
    assert not bench.l2_streams("auto", 67_400_000, l2)    # 16k prefix: flushed
    assert not bench.l2_streams("auto", 3 * l2 // 2, l2)   # exactly 1.5x: flushed
    assert bench.l2_streams("stream", 1, l2)
    assert not bench.l2_streams("flush", 10 * l2, l2)


def test_traffic_record_is_tied_to_the_kernel_sources():
    h = bench.kernel_source_hash()
    assert len(h) == 16 and h == bench.kernel_source_hash()
    assert bench.recorded_traffic("no-such-workload") is None
    path = os.path.join(ROOT, "profiles", "traffic.txt")
    for line in open(path):
        parts = line.split()
        if line.startswith("#") or len(parts) < 3:
            continue
        got = bench.recorded_traffic(parts[0])
        assert got == (int(parts[1]) if parts[2] == h else None)


def test_reference_arm_prints_the_contract_line():
    out = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--steps", "1", "--warmup", "3",
                          "--cpu-seconds", "0.2", "--config", "2"], cwd=ROOT, capture_output=True, text=True,
                         timeout=600)
    assert out.returncode == 0, out.stderr[-2000:]
    line = json.loads([l for l in out.stdout.splitlines() if l.startswith("{")][-1])
    assert line["impl"] == "reference" and line["unit"] == "nodes/s" and line["value"] > 0
    assert line["higher_is_better"] is True and line["config"]["workload"].startswith("chain")
    assert line["cpu_baseline"]["kind"] == "oracle" and line["cpu_baseline"]["cores"] >= 1
    assert line["cpu_baseline"]["value"] == line["value"] and line["cpu_baseline"]["sample"]
    assert line["e2e"] == {"value": line["value"], "unit": "nodes/s", "h2d_bytes_per_step": 0,
                           "d2h_bytes_per_step": 0}


def test_cpu_baseline_records_the_host_model_and_a_single_thread_figure():
    assert isinstance(bench.cpu_model(), str) and bench.cpu_model()
    one = bench.single_thread_oracle(2)
    assert one is not None and one["cores"] == 1 and one["value"] > 0 and one["unit"] == "nodes/s"
