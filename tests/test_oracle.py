"""Pins for the CPU oracle (no GPU).

The oracle is checked against things other than itself: hand-derived
fixtures from the definitions of "Design and optimization of DBSCAN Algorithm
based on CUDA" §II (tests/golden), closed forms, a brute-force restatement
built on a library connected-components routine, scikit-learn's DBSCAN where
it is installed, symmetries, and planted mistakes that must break a pin.
"""
import os
import subprocess
import tempfile

import numpy as np
import pytest

import oracle
from all_pairs_distance_gb300 import synth
from conftest import GOLDEN_FILES, load_golden


# --------------------------------------------------------------------------
# helpers (independent of the oracle)
# --------------------------------------------------------------------------

def brute_force_dbscan(P, eps, min_pts):
    """Tiny-input DBSCAN through a dense neighbour matrix and scipy's
    connected components -- a different algorithm from the oracle's BFS."""
    from scipy.sparse import csr_matrix
    from scipy.sparse.csgraph import connected_components

    X = np.asarray(P, dtype=np.float64)
    thr = float(np.float32(eps) * np.float32(eps))
    D2 = ((X[:, None, :] - X[None, :, :]) ** 2).sum(-1)
    A = D2 <= thr
    cnt = A.sum(1).astype(np.int32)
    core = cnt >= min_pts
    n = len(X)
    label = np.full(n, -1, np.int64)
    ci = np.flatnonzero(core)
    if len(ci):
        sub = csr_matrix(A[np.ix_(ci, ci)])
        ncomp, comp = connected_components(sub, directed=False)
        name = np.full(ncomp, np.iinfo(np.int64).max)
        np.minimum.at(name, comp, ci)
        label[ci] = name[comp]
        for i in np.flatnonzero(~core):
            nb = ci[A[i, ci]]
            if len(nb):
                label[i] = label[nb].min()
    return cnt, core.astype(np.uint8), label.astype(np.int32)


def canonical(label, core):
    """Relabel clusters by their smallest core index (noise stays -1)."""
    out = np.full(len(label), -1, np.int64)
    for lab in np.unique(label[label >= 0]):
        members = np.flatnonzero(label == lab)
        cores = members[core[members] == 1]
        out[members] = cores.min() if len(cores) else members.min()
    return out


# --------------------------------------------------------------------------
# hand-derived fixtures
# --------------------------------------------------------------------------

@pytest.mark.parametrize("name", GOLDEN_FILES)
def test_golden_fixture(name):
    P, eps, min_pts, exp = load_golden(name)
    cnt, core, label = oracle.dbscan(P, eps, min_pts)
    np.testing.assert_array_equal(cnt, exp["cnt"])
    np.testing.assert_array_equal(core, exp["core"])
    np.testing.assert_array_equal(label, exp["label"])


# --------------------------------------------------------------------------
# closed forms
# --------------------------------------------------------------------------

@pytest.mark.parametrize("n,s", [(2, 1), (7, 3), (50, 5), (129, 2)])
def test_collinear_counts(n, s):
    # Points at spacing s along an axis with eps = s: each point sees its two
    # neighbours and itself, the ends one neighbour and themselves.
    P = np.zeros((n, 2), np.float32)
    P[:, 0] = np.arange(n) * s
    cnt, core, label = oracle.dbscan(P, float(s), 3)
    expect = np.full(n, 3)
    expect[0] = expect[-1] = 2
    if n == 2:
        expect[:] = 2
    np.testing.assert_array_equal(cnt, expect)
    if n >= 3:
        # all interior points are core and chained: one cluster named 1
        np.testing.assert_array_equal(label, np.ones(n))


@pytest.mark.parametrize("d,L", [(1, 9), (2, 6), (3, 4), (4, 3)])
def test_lattice_counts(d, L):
    # Unit lattice with eps = 1: cnt = 1 + number of axis neighbours inside
    # the lattice (1 + 2d in the interior).
    grid = np.stack(np.meshgrid(*[np.arange(L)] * d, indexing="ij"), -1).reshape(-1, d)
    P = grid.astype(np.float32)
    cnt = oracle.counts(P, 1.0)
    expect = 1 + ((grid > 0).astype(int) + (grid < L - 1).astype(int)).sum(1)
    np.testing.assert_array_equal(cnt, expect)


def test_isolated_points_are_noise():
    P = np.arange(40, dtype=np.float32).reshape(20, 2) * 50.0
    cnt, core, label = oracle.dbscan(P, 10.0, 2)
    np.testing.assert_array_equal(cnt, np.ones(20))
    np.testing.assert_array_equal(core, np.zeros(20))
    np.testing.assert_array_equal(label, -np.ones(20))
    # MinPts = 1: every point is core and its own cluster
    cnt, core, label = oracle.dbscan(P, 10.0, 1)
    np.testing.assert_array_equal(core, np.ones(20))
    np.testing.assert_array_equal(label, np.arange(20))


@pytest.mark.parametrize("seed", range(6))
def test_minpts1_is_runs_in_1d(seed):
    # MinPts = 1 makes every point core, so clusters are the connected
    # components of the eps-graph; in 1-D those are the runs of sorted points
    # whose gaps are <= eps, each named by its smallest index.
    rng = np.random.default_rng(seed)
    n, eps = 300, 4.0
    x = rng.integers(0, 600, n).astype(np.float32)
    order = np.argsort(x, kind="stable")
    run = np.zeros(n, np.int64)
    r = 0
    for a, b in zip(order[:-1], order[1:]):
        if x[b] - x[a] > eps:
            r += 1
        run[b] = r
    run[order[0]] = 0
    expect = np.empty(n, np.int64)
    for k in np.unique(run):
        m = np.flatnonzero(run == k)
        expect[m] = m.min()
    cnt, core, label = oracle.dbscan(x[:, None], eps, 1)
    assert core.all()
    np.testing.assert_array_equal(label, expect)


def test_eps_zero_counts_duplicates_only():
    P = np.array([[1, 1], [2, 2], [1, 1], [3, 3], [1, 1], [2, 2]], np.float32)
    cnt, core, label = oracle.dbscan(P, 0.0, 2)
    np.testing.assert_array_equal(cnt, [3, 2, 3, 1, 3, 2])
    np.testing.assert_array_equal(label, [0, 1, 0, -1, 0, 1])


# --------------------------------------------------------------------------
# brute force / library cross-checks on small random inputs
# --------------------------------------------------------------------------

@pytest.mark.parametrize("seed", range(12))
def test_matches_brute_force(seed):
    rng = np.random.default_rng(100 + seed)
    n = int(rng.integers(1, 160))
    d = int(rng.choice([1, 2, 3, 5, 16]))
    hi = int(rng.choice([8, 30, 255]))
    P = synth.uniform_ints(n, d, hi, seed=seed)
    eps = float(rng.choice([1.0, 2.5, 4.0, 9.0, 30.0]))
    min_pts = int(rng.integers(1, 6))
    exp = brute_force_dbscan(P, eps, min_pts)
    got = oracle.dbscan(P, eps, min_pts)
    for g, e in zip(got, exp):
        np.testing.assert_array_equal(g, e)


@pytest.mark.parametrize("name", ["blobs_2k_d2", "blobs_100k_d2", "blobs_1m_d3"])
def test_matches_sklearn_on_blobs(name):
    skl = pytest.importorskip("sklearn.cluster")
    w = synth.WORKLOADS[name]
    P = synth.generate(name) if name == "blobs_2k_d2" else synth.scaled(name, 3000)
    cnt, core, label = oracle.dbscan(P, w.eps, w.min_pts)
    db = skl.DBSCAN(eps=w.eps, min_samples=w.min_pts, algorithm="brute").fit(P.astype(np.float64))
    sk_core = np.zeros(len(P), np.uint8)
    sk_core[db.core_sample_indices_] = 1
    np.testing.assert_array_equal(core, sk_core)
    # same partition of the core points; scikit-learn hands border points to
    # whichever cluster reaches them first, so only their noise status is compared
    c = core == 1
    np.testing.assert_array_equal(canonical(label, core)[c], canonical(db.labels_, sk_core)[c])
    np.testing.assert_array_equal(label == -1, db.labels_ == -1)


@pytest.mark.parametrize("name,n", [("blobs_1m_d3", 8000), ("blobs_100k_d2", 6000),
                                    ("blobs_200k_d16", 2000)])
def test_matches_kdtree_restatement(name, n):
    # an exact DBSCAN built from a k-d tree neighbour search and scipy's
    # connected components (used at full size by the GPU tests)
    from gpu_util import kdtree_dbscan
    w = synth.WORKLOADS[name]
    P = synth.scaled(name, n)
    for g, e in zip(kdtree_dbscan(P, w.eps, w.min_pts), oracle.dbscan(P, w.eps, w.min_pts)):
        np.testing.assert_array_equal(g, e)


# --------------------------------------------------------------------------
# symmetries
# --------------------------------------------------------------------------

def test_permutation_and_translation_invariance():
    P = synth.scaled("blobs_2k_d2", 1500, seed=11)
    cnt, core, label = oracle.dbscan(P, 30.0, 5)
    rng = np.random.default_rng(5)
    perm = rng.permutation(len(P))
    cnt2, core2, label2 = oracle.dbscan(P[perm], 30.0, 5)
    np.testing.assert_array_equal(cnt2, cnt[perm])
    np.testing.assert_array_equal(core2, core[perm])
    # same partition: relabelling by smallest (new) core index must agree
    np.testing.assert_array_equal(label2 == -1, label[perm] == -1)
    same = label[perm][:, None] == label[perm][None, :]
    same2 = label2[:, None] == label2[None, :]
    cmask = core2 == 1
    np.testing.assert_array_equal(same[np.ix_(cmask, cmask)], same2[np.ix_(cmask, cmask)])
    # integer translation and axis swap change nothing
    Q = P[:, ::-1] + np.float32(517.0)
    for g, e in zip(oracle.dbscan(Q, 30.0, 5), (cnt, core, label)):
        np.testing.assert_array_equal(g, e)


def test_row_helpers_agree_with_counts():
    P = synth.scaled("blobs_1m_d3", 2000, seed=3)
    cnt = oracle.counts(P, 10.0)
    rows = np.array([0, 5, 17, 1999, 1000])
    np.testing.assert_array_equal(oracle.row_counts(P, 10.0, rows), cnt[rows])
    for i in rows:
        nb = oracle.row_neighbours(P, 10.0, int(i))
        assert len(nb) == cnt[i] and i in nb
        assert np.all(np.diff(nb) > 0)


# --------------------------------------------------------------------------
# planted mistakes: each must break at least one pin
# --------------------------------------------------------------------------

MUTANTS = {
    "strict_threshold": [("sq_dist(pts, d, i, j) <= thr", "sq_dist(pts, d, i, j) < thr")],
    "core_greater_than": [("cnt[i] >= min_pts", "cnt[i] > min_pts")],
    "self_excluded": [("if (sq_dist(pts, d, i, j) <= thr)\n            ++c;",
                       "if (j != i && sq_dist(pts, d, i, j) <= thr)\n            ++c;")],
    "border_expands": [("if (core[j])\n                    queue", "if (1)\n                    queue")],
    "border_last_claim": [("if (label[j] != -1)\n                    continue;",
                           "if (label[j] != -1 && core[j])\n                    continue;")],
    "sign_error": [("double t = a[k] - b[k];", "double t = a[k] + b[k];")],
    "index_error": [("double t = a[k] - b[k];", "double t = a[k] - b[0];")],
    "eps_not_squared": [("volatile float e2 = eps * eps;", "volatile float e2 = eps;")],
}


def _run_fixture_with(lib_path, P, eps, min_pts):
    import ctypes
    lib = ctypes.CDLL(lib_path)
    p = np.ascontiguousarray(P, np.float64)
    n, d = p.shape
    cnt = np.zeros(n, np.int32)
    core = np.zeros(n, np.uint8)
    label = np.zeros(n, np.int32)
    f = lib.oracle_dbscan
    f.argtypes = [ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                  ctypes.c_int32, ctypes.c_void_p, ctypes.c_void_p, ctypes.c_void_p]
    vp = lambda a: a.ctypes.data_as(ctypes.c_void_p)
    f(vp(p), n, d, eps, min_pts, vp(cnt), vp(core), vp(label))
    return cnt, core, label


@pytest.mark.parametrize("mutant", sorted(MUTANTS))
def test_planted_mistake_is_caught(mutant):
    src = open(os.path.join(os.path.dirname(oracle.__file__), "dbscan_oracle.c")).read()
    for old, new in MUTANTS[mutant]:
        assert old in src, f"mutation anchor missing: {old!r}"
        src = src.replace(old, new)
    with tempfile.TemporaryDirectory() as tmp:
        c = os.path.join(tmp, "m.c")
        so = os.path.join(tmp, "m.so")
        open(c, "w").write(src)
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-o", so, c])
        caught = False
        for name in GOLDEN_FILES:
            P, eps, min_pts, exp = load_golden(name)
            got = _run_fixture_with(so, P, eps, min_pts)
            if any(not np.array_equal(g, exp[k]) for g, k in zip(got, ("cnt", "core", "label"))):
                caught = True
                break
        assert caught, f"no golden fixture detects mutant {mutant}"


def test_compact_labels_worked_examples():
    # hand-worked: distinct labels in increasing order become 0, 1, ...
    out, k = oracle.compact_labels([5, -1, 5, 2, 2, -1, 9])
    assert k == 3
    assert out.tolist() == [1, -1, 1, 0, 0, -1, 2]
    out, k = oracle.compact_labels([-1, -1])
    assert k == 0 and out.tolist() == [-1, -1]
    out, k = oracle.compact_labels([])
    assert k == 0 and out.size == 0
    out, k = oracle.compact_labels([0, 1, 2, 3])
    assert k == 4 and out.tolist() == [0, 1, 2, 3]


def test_compact_labels_of_a_clustering_keeps_the_partition():
    # on a real clustering: same partition, noise kept, ids contiguous and in
    # the order of each cluster's smallest core index (its first point)
    P = np.array([[0.0], [1.0], [2.0], [10.0], [11.0], [12.0], [30.0], [20.0], [21.0], [22.0]])
    cnt, core, lab = oracle.dbscan(P, 1.0, 2)
    out, k = oracle.compact_labels(lab)
    assert k == 3
    assert out.tolist() == [0, 0, 0, 1, 1, 1, -1, 2, 2, 2]
    for i in range(len(lab)):
        for j in range(len(lab)):
            assert (lab[i] == lab[j]) == (out[i] == out[j])


def test_openmp_build_gives_identical_results():
    # the separately timed OpenMP build of the same source (count loop on all
    # host cores) must return exactly what the single-threaded build does
    if oracle.parallel_threads() == 0:
        pytest.skip("no OpenMP-capable compiler")
    for P, eps, mp in ((synth.scaled("blobs_1m_d3", 3_000, seed=81), 10.0, 8),
                       (synth.scaled("blobs_200k_d16", 1_500, seed=82), 120.0, 20)):
        a = oracle.dbscan(P, eps, mp)
        b = oracle.dbscan_parallel(P, eps, mp)
        for x, y in zip(a, b):
            assert np.array_equal(x, y)
