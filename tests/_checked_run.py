"""Runs the scaled-down parity cases, the acceptance walk and the KV commit through the
library named by TVA_LIBRARY (the index-checked build, libtva_checked.so) and compares them
with the oracle.  Executed as a child process by tests/test_checked_gpu.py, so that the
checked library is the one this process loads; prints one line per case and exits 1 on
any mismatch or non-zero device status."""
import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402
import torch  # noqa: E402

import oracle  # noqa: E402
from tree_verification_attention_gb300 import api, workloads  # noqa: E402
from tests import _gpu  # noqa: E402

CASES = [
    (1, {}),
    (2, dict(prefix=1100)),
    (3, dict(prefix=1500)),
    (4, dict(prefix=(200, 1300))),
    (5, dict(prefix=900)),
    (6, dict(prefix=700, batch=3)),
    (1, dict(batch=40, Hq=32, Hkv=8, d=128, prefix=(50, 300), m=8, tree="random", dtype="bf16", vocab=8)),
    (1, dict(batch=3, Hq=16, Hkv=2, d=64, prefix=(0, 300), m=17, tree="random", dtype="bf16", vocab=8)),
    (1, dict(batch=2, Hq=12, Hkv=4, d=128, prefix=(77, 200), m=50, tree="random", dtype="bf16", vocab=8)),
]


def main():
    lib = api.load_library()
    assert os.path.basename(lib._name) == "libtva_checked.so", lib._name
    bad = 0
    for cfg, over in CASES:
        w = workloads.make_workload(cfg, seed=None if cfg != 1 or not over else 77, **over)
        out, lse, st = _gpu.run_attention(w)
        o_ref, l_ref = _gpu.oracle_attention(w)
        try:
            _gpu.assert_close(w, out, lse, o_ref, l_ref, w.name)
            ok = st == 0
        except AssertionError as e:
            print("mismatch", w.name, str(e)[:200])
            ok = False
        t = _gpu.to_device(w)
        ast = torch.zeros(1, dtype=torch.int32, device="cuda:0")
        alen, apath, nxt = api.accept_longest_path(t["cu_nodes"], t["parent"], t["draft_tok"], t["target_argmax"],
                                                   dev_status=ast)
        torch.cuda.synchronize()
        a_ref = oracle.accept_longest_path(w.parent, w.draft_tok, w.target_argmax, w.cu_nodes)
        ok = ok and int(ast.item()) == 0 and np.array_equal(alen.cpu().numpy(), a_ref[0]) and \
            np.array_equal(apath.cpu().numpy(), a_ref[1]) and np.array_equal(nxt.cpu().numpy(), a_ref[2])
        print(("ok  " if ok else "FAIL"), w.name, over, "status", st, int(ast.item()), flush=True)
        bad += 0 if ok else 1
    print("checked build:", "PASS" if bad == 0 else f"{bad} FAILED")
    sys.exit(1 if bad else 0)


if __name__ == "__main__":
    main()
