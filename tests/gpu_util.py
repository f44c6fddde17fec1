"""Helpers shared by the GPU tests: run the CUDA path through the C ABI and
check DBSCAN invariants against the oracle's per-row functions."""
import numpy as np
import torch

import oracle
from all_pairs_distance_gb300 import binding


def gpu_run(P, eps, min_pts, dtype=torch.float32, counts=True):
    """(cnt, core, label) from the CUDA library for host array P."""
    x = torch.from_numpy(np.ascontiguousarray(P)).to("cuda").to(dtype)
    ws = binding.workspace_for(x)
    labels, core = binding.dbscan_fit_ex(x, eps, min_pts, workspace=ws)
    st = binding.dbscan_workspace_status(ws)
    assert st == 0, binding.dbscan_strerror(st)
    cnt = None
    if counts:
        cnt = binding.dbscan_neighbor_counts(x, eps, workspace=ws)
        st = binding.dbscan_workspace_status(ws)
        assert st == 0, binding.dbscan_strerror(st)
        cnt = cnt.cpu().numpy()
    return cnt, core.cpu().numpy(), labels.cpu().numpy()


def assert_same(got, exp, what):
    got = np.asarray(got)
    exp = np.asarray(exp)
    if not np.array_equal(got, exp):
        bad = np.flatnonzero(got != exp)
        raise AssertionError(f"{what}: {len(bad)} mismatches, first at {bad[:8].tolist()}: "
                             f"got {got[bad[:8]].tolist()} expected {exp[bad[:8]].tolist()}")


def check_sampled(P64, eps, min_pts, cnt, core, label, rows):
    """Check a full-size result on sampled rows with the oracle's per-row
    functions, plus the invariants that hold at any size."""
    n = len(label)
    # core labels: a core point's label is a core point of the same cluster
    # with a smaller or equal index, and is its own label
    ci = np.flatnonzero(core == 1)
    lab_c = label[ci]
    assert np.all(lab_c >= 0) and np.all(lab_c <= ci)
    assert np.all(core[lab_c] == 1)
    assert np.all(label[lab_c] == lab_c)
    # non-core points are labelled -1 or with an existing cluster name
    nc = np.flatnonzero(core == 0)
    lab_n = label[nc]
    assert np.all((lab_n == -1) | ((lab_n >= 0) & (core[np.maximum(lab_n, 0)] == 1)))
    # sampled rows against the oracle
    if cnt is not None:
        assert_same(cnt[rows], oracle.row_counts(P64, eps, rows), "sampled counts")
        assert_same(core[rows], (cnt[rows] >= min_pts).astype(np.uint8), "core from counts")
    else:
        rc = oracle.row_counts(P64, eps, rows)
        assert_same(core[rows], (rc >= min_pts).astype(np.uint8), "sampled core flags")
    for i in rows:
        nb = oracle.row_neighbours(P64, eps, int(i))
        cn = nb[core[nb] == 1]
        if core[i]:
            # every core neighbour is in the same cluster
            assert np.all(label[cn] == label[i]), f"core {i}: neighbour in another cluster"
        elif len(cn):
            assert label[i] == label[cn].min(), f"border {i}: not the smallest neighbouring label"
        else:
            assert label[i] == -1, f"noise {i} labelled {label[i]}"
