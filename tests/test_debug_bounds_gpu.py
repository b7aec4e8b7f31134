"""The range-checked build (-DSGEMM_DEBUG_BOUNDS) run over every path.

compute-sanitizer is closed on this machine, so the library carries its own
memory checker: a build in which every kernel checks the indices of its
shared-memory, global-memory, tensor-memory and TMA accesses, skips an access
out of range and reports it as SGEMM_ERR_BOUNDS.  The guarded, zero-padded
tiles of the exercise page ("3.3 Shared memory and tiling - exercises",
exercise 1) are what it checks at run time.  This test builds that library
and runs tests/_debug_bounds_cases.py against it in a subprocess: every entry
point, kernel variant and edge case there must stay in range and match the
oracle.
"""
import os
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

HERE = os.path.dirname(os.path.abspath(__file__))


def test_range_checked_build_keeps_every_index_in_range(cuda_device):
    from dense_fp32_gemm_02_gb300 import build
    build.build(debug_bounds=True)
    env = dict(os.environ, SGEMM_LIBRARY="debug_bounds")
    r = subprocess.run([sys.executable, os.path.join(HERE, "_debug_bounds_cases.py")], env=env,
                       capture_output=True, text=True, timeout=1200)
    assert r.returncode == 0, (r.stdout[-4000:] + "\n" + r.stderr[-4000:])
    assert "all cases in range" in r.stdout
