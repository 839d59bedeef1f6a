"""The small-shape GPU parity suites again, against the bounds-checked debug build of the library.

compute-sanitizer is not available here, so the library has its own debug build (-DTPMLP_DEBUG_BOUNDS): the
row kernels and the GEMM epilogues check every hand-computed global index against the extent of its buffer,
count the ones outside and skip those accesses.  This test builds that library beside the release one and
runs the parity tests of the row kernels, the blocks, the SP region and FP8 in a child pytest that loads it
(TPMLP_LIBRARY); there, after every test, an autouse fixture asserts that the build checks and counted no
violation, and every test still compares its results with the oracle.
"""
import os
import subprocess
import sys

import pytest

from tensor_transformer_mlp_tp_gb300 import build

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SUITES = ["tests/test_gpu_parity.py", "tests/test_gpu_sp_region.py", "tests/test_gpu_fp8.py"]


def test_parity_suites_under_bounds_checks():
    lib = build.build(debug_bounds=True)
    env = dict(os.environ, TPMLP_LIBRARY=lib, TPMLP_EXPECT_BOUNDS_CHECKED="1")
    r = subprocess.run([sys.executable, "-m", "pytest", *SUITES, "-m", "gpu", "-q", "-x", "-p", "no:cacheprovider"],
                       cwd=ROOT, env=env, capture_output=True, text=True, timeout=1800)
    tail = "\n".join((r.stdout + r.stderr).strip().splitlines()[-25:])
    assert r.returncode == 0, tail
    assert " passed" in tail and "failed" not in tail, tail
