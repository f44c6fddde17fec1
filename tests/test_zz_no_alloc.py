"""dbscan_fit_noalloc: the DBSCAN entry point for callers that cannot
allocate device memory (a host framework's allocator owns the device memory,
or a serving path must not allocate after start-up).  Its workspace is a
static device array inside the library; its results must equal the oracle's
and those of dbscan_fit_ex, call after call, since every call reuses that
array -- on the legacy default stream and on a stream of the caller's, where
the entry point launches directly instead of capturing a graph."""
import ctypes

import numpy as np
import pytest
import torch

import oracle
from all_pairs_distance_gb300 import binding, synth
from gpu_util import assert_same

pytestmark = pytest.mark.gpu


def _entry():
    lib = binding.load()
    f = lib.dbscan_fit_noalloc
    P = ctypes.c_void_p
    f.argtypes = [P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                  ctypes.c_int32, P, P, P]
    f.restype = ctypes.c_int
    return f


def _noalloc(f, x, eps, min_pts):
    n, d = x.shape
    labels = torch.full((n,), -7, dtype=torch.int32, device=x.device)
    core = torch.full((n,), 9, dtype=torch.uint8, device=x.device)
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    st = f(x.data_ptr(), binding.DTYPES[x.dtype], n, d, float(eps), int(min_pts),
           labels.data_ptr(), core.data_ptr(), stream)
    assert st == 0, binding.dbscan_strerror(st)
    return labels, core


CASES = [
    (lambda: synth.scaled("blobs_1m_d3", 50_000, seed=21), 10.0, 8, torch.float32),
    (lambda: synth.scaled("blobs_100k_d2", 30_000, seed=22), 20.0, 10, torch.float32),
    (lambda: synth.scaled("blobs_500k_d64", 6_000, seed=23), 100.0, 16, torch.bfloat16),
]


@pytest.mark.parametrize("stream_kind", ["legacy", "own"])
def test_noalloc_matches_oracle_and_dbscan_fit_ex_on_consecutive_calls(stream_kind):
    f = _entry()
    stream = torch.cuda.current_stream() if stream_kind == "legacy" else torch.cuda.Stream()
    for make, eps, min_pts, dtype in CASES:
        P = make()
        _, core_ref, label_ref = oracle.dbscan(P, eps, min_pts)
        x = torch.from_numpy(P).cuda().to(dtype)
        ref_labels, ref_core = binding.dbscan_fit_ex(x, eps, min_pts)
        torch.cuda.synchronize()
        with torch.cuda.stream(stream):
            for _ in range(2):   # two calls in a row on the shared static workspace
                labels, core = _noalloc(f, x, eps, min_pts)
                stream.synchronize()
                assert torch.equal(labels, ref_labels)
                assert torch.equal(core, ref_core)
                assert_same(labels.cpu().numpy(), label_ref, "noalloc labels vs oracle")
                assert_same(core.cpu().numpy(), core_ref, "noalloc core flags vs oracle")


def test_noalloc_rejects_problems_beyond_its_scratch():
    f = _entry()
    assert f(None, 0, 10_000_000, 3, 1.0, 2, None, None, None) == binding.Status.UNSUPPORTED
    assert f(None, 0, -1, 3, 1.0, 2, None, None, None) == binding.Status.INVALID_ARG
    assert binding.dbscan_workspace_size(10_000_000, 3) > (64 << 20)
