"""Label compaction on the GPU (dbscan_compact_labels) against the oracle's."""
import numpy as np
import pytest
import torch

import oracle
from all_pairs_distance_gb300 import binding, synth
from gpu_util import assert_same, gpu_run

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["c4_like_20k_d3", "c5_like_3k_d64", "noise_only"])
def test_compact_labels_of_clusterings(case):
    if case == "c4_like_20k_d3":
        P, eps, mp, dt = synth.scaled("blobs_1m_d3", 20_011), 10.0, 8, torch.float32
    elif case == "c5_like_3k_d64":
        P, eps, mp, dt = synth.scaled("blobs_500k_d64", 3_001, seed=61), 100.0, 16, torch.bfloat16
    else:
        P, eps, mp, dt = synth.uniform_ints(3_000, 2, 4_000, 62), 1.0, 4, torch.float32
    _, _, label = gpu_run(P, eps, mp, dt)
    ref, k_ref = oracle.compact_labels(label)
    lab = torch.from_numpy(label.astype(np.int32)).cuda()
    out, k = binding.dbscan_compact_labels(lab)
    assert k == k_ref
    assert_same(out.cpu().numpy(), ref, f"{case} compacted labels")
    # in place
    out2, k2 = binding.dbscan_compact_labels(lab, out=lab)
    assert k2 == k_ref
    assert_same(lab.cpu().numpy(), ref, f"{case} compacted in place")


def test_compact_labels_many_blocks():
    # 3M labels in many 1024-label scan blocks: representatives at random
    # positions, every other point on one of them or noise
    rng = np.random.default_rng(63)
    n = 3_000_000
    reps = np.sort(rng.choice(n, size=40_000, replace=False))
    lab = np.full(n, -1, np.int64)
    others = rng.random(n) < 0.8
    lab[others] = reps[rng.integers(0, reps.size, size=int(others.sum()))]
    lab[reps] = reps
    ref, k_ref = oracle.compact_labels(lab)
    out, k = binding.dbscan_compact_labels(torch.from_numpy(lab.astype(np.int32)).cuda())
    assert k == k_ref == reps.size
    assert_same(out.cpu().numpy(), ref, "3M compacted labels")


def test_compact_labels_edge_cases():
    empty = torch.empty(0, dtype=torch.int32, device="cuda")
    out, k = binding.dbscan_compact_labels(empty)
    assert k == 0 and out.numel() == 0
    one = torch.tensor([0], dtype=torch.int32, device="cuda")
    out, k = binding.dbscan_compact_labels(one)
    assert k == 1 and out.tolist() == [0]
    # labels dbscan_fit* cannot produce are rejected and the output is untouched:
    # a label pointing at a point not labelled with itself, out of range, below -1
    for bad in ([1, 0], [5, -1], [-2, 1], [0, 0, 1]):
        lab = torch.tensor(bad, dtype=torch.int32, device="cuda")
        keep = torch.full_like(lab, 77)
        with pytest.raises(RuntimeError):
            binding.dbscan_compact_labels(lab, out=keep)
        assert keep.tolist() == [77] * len(bad)
    # the context is still usable afterwards
    out, k = binding.dbscan_compact_labels(torch.tensor([-1, 1, 1], dtype=torch.int32, device="cuda"))
    assert k == 1 and out.tolist() == [-1, 0, 0]
