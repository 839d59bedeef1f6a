import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden(name):
    """Rows of a whitespace-separated golden file, comments stripped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(autouse=True)
def _debug_bounds_clean(request):
    """In a run against the bounds-checked debug build (TPMLP_EXPECT_BOUNDS_CHECKED set, as
    test_gpu_debug_bounds.py sets it for its child pytest), every GPU test must leave the library with no
    out-of-range global index counted."""
    yield
    if os.environ.get("TPMLP_EXPECT_BOUNDS_CHECKED") and request.node.get_closest_marker("gpu") is not None:
        from tensor_transformer_mlp_tp_gb300 import binding

        checked, violations, site = binding.tpmlp_debug_bounds_status()
        assert checked, "the loaded library is not the bounds-checked build"
        assert violations == 0, f"{violations} global indices out of range (first at site {site})"
