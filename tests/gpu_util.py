"""Helpers shared by the GPU tests: run the CUDA path through the C ABI and
check DBSCAN invariants against the oracle's per-row functions."""
import numpy as np
import torch

import oracle
from all_pairs_distance_gb300 import binding


def gpu_run(P, eps, min_pts, dtype=torch.float32, counts=True, info=None):
    """(cnt, core, label) from the CUDA library for host array P.  When
    ``info`` is a dict it receives dbscan_workspace_info of the fit."""
    x = torch.from_numpy(np.ascontiguousarray(P)).to("cuda").to(dtype)
    ws = binding.workspace_for(x)
    labels, core = binding.dbscan_fit_ex(x, eps, min_pts, workspace=ws)
    st = binding.dbscan_workspace_status(ws)
    assert st == 0, binding.dbscan_strerror(st)
    if info is not None:
        info.update(binding.dbscan_workspace_info(ws))
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


def kdtree_dbscan(P, eps, min_pts):
    """Exact DBSCAN for integer coordinates, independent of the oracle: k-d tree
    pairs within eps + 0.5, an exact integer filter d^2 <= eps^2, scipy's
    connected components over core-core pairs, smallest-index names, border
    points to the smallest neighbouring core label."""
    from scipy.sparse import coo_matrix
    from scipy.sparse.csgraph import connected_components
    from scipy.spatial import cKDTree

    X = P.astype(np.int64)
    n = len(X)
    thr = int(np.float32(eps) * np.float32(eps))
    # integer squared distances <= thr imply distance <= sqrt(thr) < eps + 0.5
    pairs = cKDTree(P.astype(np.float64)).query_pairs(r=float(eps) + 0.5, output_type="ndarray")
    d2 = ((X[pairs[:, 0]] - X[pairs[:, 1]]) ** 2).sum(1)
    pairs = pairs[d2 <= thr]
    a, b = pairs[:, 0], pairs[:, 1]
    cnt = 1 + np.bincount(a, minlength=n) + np.bincount(b, minlength=n)
    core = cnt >= min_pts
    label = np.full(n, -1, np.int64)
    cc = core[a] & core[b]
    g = coo_matrix((np.ones(int(cc.sum()), np.int8), (a[cc], b[cc])), shape=(n, n)).tocsr()
    _, comp = connected_components(g, directed=False)
    ci = np.flatnonzero(core)
    name = np.full(comp.max() + 1, np.iinfo(np.int64).max)
    np.minimum.at(name, comp[ci], ci)
    label[ci] = name[comp[ci]]
    big = np.iinfo(np.int64).max
    border = np.full(n, big)
    m1 = core[a] & ~core[b]
    np.minimum.at(border, b[m1], label[a[m1]])
    m2 = core[b] & ~core[a]
    np.minimum.at(border, a[m2], label[b[m2]])
    nc = ~core & (border != big)
    label[nc] = border[nc]
    return cnt.astype(np.int32), core.astype(np.uint8), label.astype(np.int32)
