"""The work decomposition that the attention kernels share (tva_common.cuh: stream-K unit
ranges, ranges aligned to row groups, teams of workers sharing K/V tiles, and the partial
slots), compiled for the host with a plain C++ compiler and walked on a sweep of
problems, one sequence and ragged batches, exactly as the partials kernels walk it.
Every (row group, key tile) unit must be covered once, each segment must stay inside
one row group, and each (worker, segment) must own a distinct partial slot inside the
workspace the host reserves (tests/schedule_host.cpp)."""
import os
import shutil
import subprocess

import pytest

from tree_verification_attention_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))


def _cuda_include():
    try:
        nvcc = build._nvcc()
    except RuntimeError:
        return None
    inc = os.path.join(os.path.dirname(os.path.dirname(nvcc)), "include")
    return inc if os.path.exists(os.path.join(inc, "cuda_runtime.h")) else None


def test_work_decomposition_covers_every_unit_once_with_distinct_slots(tmp_path):
    cxx = shutil.which("g++") or shutil.which("c++")
    inc = _cuda_include()
    if cxx is None or inc is None:
        pytest.skip("needs a C++ compiler and the CUDA headers")
    exe = str(tmp_path / "schedule_host")
    subprocess.run([cxx, "-std=c++17", "-O1", "-I" + inc, "-I" + build.CSRC, "-I" + build.INCLUDE,
                    os.path.join(HERE, "schedule_host.cpp"), "-o", exe], check=True, capture_output=True)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
    assert int(r.stdout.split()[1]) > 500
