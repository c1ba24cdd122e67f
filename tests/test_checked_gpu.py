"""The index-checked build (libtva_checked.so, compiled with -DTVA_CHECKED).

compute-sanitizer is closed on the GPU pool this library is developed on, so the
checked build stands in for it: every index the kernels compute themselves - TMA tile
coordinates, partial slots, merged output rows, positions on an accepted path - is
checked on the device, and a failed check records TVA_ERR_INVALID_ARG instead of
touching memory out of bounds (no trap).  The scaled-down parity cases and the
acceptance walk run through that build in a child process and must match the oracle
with the device status still zero, i.e. no check fired on a consistent schedule.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_checked_build_matches_the_oracle_with_no_check_firing():
    import __graft_entry__
    __graft_entry__.build()
    from tree_verification_attention_gb300 import build
    env = dict(os.environ, TVA_LIBRARY=build.CHECKED_LIB_PATH)
    r = subprocess.run([sys.executable, os.path.join(ROOT, "tests", "_checked_run.py")], env=env,
                       capture_output=True, text=True, timeout=900)
    print(r.stdout)
    assert r.returncode == 0, r.stdout[-3000:] + r.stderr[-3000:]
    assert "checked build: PASS" in r.stdout
