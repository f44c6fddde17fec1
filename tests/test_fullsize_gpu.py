"""Full-size workloads through the same entry point and launch configuration
the benchmark times.

* blobs_100k_d2: element-by-element against the full oracle (tens of seconds).
* blobs_200k_d16, blobs_1m_d3, blobs_500k_d64: every count, core flag and
  label against the oracle's, through SHA-256 digests of the oracle's arrays
  (written by tests/golden/make_fullsize.py, which calls the oracle alone: an
  hour of host time at 500k x 64, too long to repeat per test run).
* 70,000-point sets at d = 16 (f16 and tf32) and d = 64 (bf16): past one
  512-tile column chunk of the tensor-core schedule, element by element
  against the oracle's OpenMP build, for one and two row blocks per unit.
* every workload: sampled rows -- counts from the oracle's per-row count, and
  for each sampled core / border / noise point the DBSCAN conditions checked
  against the oracle's per-row neighbour list -- plus the invariants that hold
  at any size (core labels are core indices, no larger than the point's own
  index, fixed points of the labelling).
* blobs_1m_d3: additionally a complete exact DBSCAN built independently from a
  k-d tree neighbour search (radius slack, then an exact integer filter) and
  scipy's connected components.
"""
import hashlib
import json
import os

import numpy as np
import pytest
import torch

import oracle
from all_pairs_distance_gb300 import binding, synth
from gpu_util import assert_same, check_sampled, gpu_run, kdtree_dbscan

pytestmark = pytest.mark.gpu

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def _digest(a, dtype):
    return hashlib.sha256(np.ascontiguousarray(a, dtype=dtype).tobytes()).hexdigest()


@pytest.mark.parametrize("name", ["blobs_200k_d16", "blobs_1m_d3", "blobs_500k_d64"])
def test_full_size_every_value_matches_the_oracle(name):
    with open(os.path.join(GOLDEN, f"fullsize_{name}.json")) as f:
        exp = json.load(f)
    w = synth.WORKLOADS[name]
    P = synth.generate(name)
    assert _digest(P, "<f4") == exp["input_sha256"], \
        "the generator drew a different input than the one the oracle ran on"
    dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    info = {}
    cnt, core, label = gpu_run(P, w.eps, w.min_pts, dtype, info=info)
    summary = (f"path {info.get('path')}: n_core {int(core.sum())} (oracle {exp['n_core']}), "
               f"noise {int((label == -1).sum())} (oracle {exp['n_noise']}), clusters "
               f"{np.unique(label[label >= 0]).size} (oracle {exp['n_clusters']}), count sum "
               f"{int(cnt.astype(np.int64).sum())} (oracle {exp['cnt_sum']})")
    assert _digest(cnt, "<i4") == exp["cnt_sha256"], "neighbour counts differ; " + summary
    assert _digest(core, "<u1") == exp["core_sha256"], "core flags differ; " + summary
    assert _digest(label, "<i4") == exp["label_sha256"], "labels differ; " + summary


CHUNK_CASES = {
    # name: (points, eps, min_pts, dtype, paths to force)
    "d16_70k": (lambda: synth.scaled("blobs_200k_d16", 70_001, seed=61), 120.0, 20, torch.float32,
                ("f16", "tf32")),
    "d64_70k_bf16": (lambda: synth.scaled("blobs_500k_d64", 70_003, seed=62), 100.0, 16,
                     torch.bfloat16, ("bf16",)),
}


@pytest.mark.parametrize("name", sorted(CHUNK_CASES))
def test_past_one_column_chunk_every_value(name):
    make, eps, min_pts, dtype, paths = CHUNK_CASES[name]
    P = make()
    assert len(P) > 512 * 128
    threads = oracle.parallel_threads()
    ref = oracle.dbscan_parallel(P, eps, min_pts) if threads else oracle.dbscan(P, eps, min_pts)
    for path in paths:
        for rows in (1, 2):
            info = {}
            with binding.options(paths=[path], rows=rows):
                got = gpu_run(P, eps, min_pts, dtype, info=info)
            assert info["path"] == path, info
            for g, e, what in zip(got, ref, ("cnt", "core", "label")):
                assert_same(g, e, f"{name} [{path}, rows {rows}] {what}")


def _sample_rows(core, label, seed, per_kind=40):
    rng = np.random.default_rng(seed)
    kinds = [np.flatnonzero(core == 1),
             np.flatnonzero((core == 0) & (label >= 0)),
             np.flatnonzero(label == -1)]
    rows = [rng.choice(k, size=min(per_kind, len(k)), replace=False) for k in kinds if len(k)]
    rows.append(rng.choice(len(core), size=per_kind, replace=False))
    return np.unique(np.concatenate(rows))


@pytest.mark.parametrize("name", ["blobs_2k_d2", "blobs_100k_d2", "blobs_200k_d16",
                                  "blobs_1m_d3", "blobs_500k_d64"])
def test_full_size_sampled(name):
    w = synth.WORKLOADS[name]
    P = synth.generate(name)
    dtype = torch.bfloat16 if w.dtype == "bf16" else torch.float32
    cnt, core, label = gpu_run(P, w.eps, w.min_pts, dtype)
    assert_same(core, (cnt >= w.min_pts).astype(np.uint8), "core flags vs counts")
    P64 = np.ascontiguousarray(P, dtype=np.float64)
    rows = _sample_rows(core, label, seed=w.seed)
    check_sampled(P64, w.eps, w.min_pts, cnt, core, label, rows)
    # the workload has clusters and noise
    assert core.sum() > 0 and (label == -1).sum() > 0


def test_full_oracle_parity_100k_d2():
    w = synth.WORKLOADS["blobs_100k_d2"]
    P = synth.generate(w.name)
    cnt_ref, core_ref, label_ref = oracle.dbscan(P, w.eps, w.min_pts)
    cnt, core, label = gpu_run(P, w.eps, w.min_pts)
    assert_same(cnt, cnt_ref, "counts")
    assert_same(core, core_ref, "core")
    assert_same(label, label_ref, "labels")


def test_full_exact_1m_d3_against_kdtree_dbscan():
    pytest.importorskip("scipy.spatial")
    w = synth.WORKLOADS["blobs_1m_d3"]
    P = synth.generate(w.name)
    cnt_ref, core_ref, label_ref = kdtree_dbscan(P, w.eps, w.min_pts)
    cnt, core, label = gpu_run(P, w.eps, w.min_pts)
    assert_same(cnt, cnt_ref, "counts")
    assert_same(core, core_ref, "core")
    assert_same(label, label_ref, "labels")


def test_culled_equals_all_pairs_at_1m_d3():
    # the bench workload: tile culling must not change a single label or flag
    P = synth.generate("blobs_1m_d3")
    x = torch.from_numpy(P).cuda()
    ws = binding.workspace_for(x)
    lab_a, core_a = binding.dbscan_fit_ex(x, 10.0, 8, workspace=ws)
    assert binding.dbscan_workspace_status(ws) == 0
    lab_c, core_c = binding.dbscan_fit_culled(x, 10.0, 8, workspace=ws)
    assert binding.dbscan_workspace_status(ws) == 0
    assert torch.equal(lab_a, lab_c) and torch.equal(core_a, core_c)
