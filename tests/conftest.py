import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running check")
    config.addinivalue_line("markers", "fused_pipeline: runs with the library's default "
                                       "(small problems take the fused single-launch pipeline)")


@pytest.fixture(autouse=True)
def _multi_kernel_path_by_default(request):
    """GPU tests exercise the multi-kernel path (tensor-core and CUDA-core
    sweeps) even on the small sets the fused single-launch pipeline would
    otherwise take; tests marked fused_pipeline keep the library default."""
    if request.node.get_closest_marker("gpu") is None or \
            request.node.get_closest_marker("fused_pipeline") is not None:
        yield
        return
    from all_pairs_distance_gb300 import binding
    with binding.options(fused=0):
        yield


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def load_golden(name):
    """Parse a tests/golden/*.txt fixture: header keys, points, expected arrays."""
    import numpy as np

    path = os.path.join(GOLDEN, name)
    meta, pts, exp = {}, [], {}
    mode = "meta"
    with open(path) as f:
        for raw in f:
            line = raw.strip()
            if not line or line.startswith("#"):
                continue
            head, *rest = line.split()
            if mode == "meta" and head == "points":
                mode = "points"
                continue
            if mode == "points" and head in ("cnt", "core", "label"):
                mode = "expect"
            if mode == "meta":
                meta[head] = rest[0]
            elif mode == "points":
                pts.append([float(v) for v in line.split()])
            else:
                exp[head] = np.array([int(v) for v in rest])
    d = int(meta["d"])
    P = np.array(pts, dtype=np.float32).reshape(-1, d)
    return P, float(meta["eps"]), int(meta["min_pts"]), exp


GOLDEN_FILES = sorted(f for f in os.listdir(GOLDEN) if f.endswith(".txt"))
