"""Full-size workloads through the same entry point and launch configuration
the benchmark times.

* blobs_100k_d2: element-by-element against the full oracle (tens of seconds).
* every workload: sampled rows -- counts from the oracle's per-row count, and
  for each sampled core / border / noise point the DBSCAN conditions checked
  against the oracle's per-row neighbour list -- plus the invariants that hold
  at any size (core labels are core indices, no larger than the point's own
  index, fixed points of the labelling).
* blobs_1m_d3: additionally a complete exact DBSCAN built independently from a
  k-d tree neighbour search (radius slack, then an exact integer filter) and
  scipy's connected components.
"""
import numpy as np
import pytest
import torch

import oracle
from all_pairs_distance_gb300 import binding, synth
from gpu_util import assert_same, check_sampled, gpu_run, kdtree_dbscan

pytestmark = pytest.mark.gpu


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
