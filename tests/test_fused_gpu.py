"""The fused single-launch pipeline (every stage in one cooperative kernel,
taken by default for problems of at most 4,096 points with d <= 4 or 8,192
points with 4 < d <= 32) against the oracle, element by element: counts,
core flags and labels."""
import numpy as np
import pytest
import torch

import oracle
from all_pairs_distance_gb300 import binding, synth
from conftest import GOLDEN_FILES, load_golden
from gpu_util import assert_same, gpu_run

pytestmark = [pytest.mark.gpu, pytest.mark.fused_pipeline]

CASES = {
    # name: (points, eps, min_pts, dtype)
    "c1_full_2k_d2": (lambda: synth.generate("blobs_2k_d2"), 30.0, 5, torch.float32),
    "c2_like_4k_d2": (lambda: synth.scaled("blobs_100k_d2", 4_096, seed=91), 20.0, 10, torch.float32),
    "c4_like_4k_d3": (lambda: synth.scaled("blobs_1m_d3", 4_093, seed=92), 10.0, 8, torch.float32),
    "c3_like_6k_d16": (lambda: synth.scaled("blobs_200k_d16", 6_007, seed=93), 120.0, 20, torch.float32),
    "d16_bf16": (lambda: synth.blob_set(5_000, 16, 255, 10, 6.0, 500, 94), 30.0, 6, torch.bfloat16),
    "d32_bf16": (lambda: synth.blob_set(3_000, 32, 255, 10, 6.0, 300, 95), 45.0, 6, torch.bfloat16),
    "d1_blobs": (lambda: synth.blob_set(4_000, 1, 4095, 6, 30.0, 400, 96), 2.0, 4, torch.float32),
    "d4_blobs": (lambda: synth.blob_set(4_000, 4, 1023, 20, 10.0, 400, 97), 12.0, 6, torch.float32),
    "d5_blobs": (lambda: synth.blob_set(8_000, 5, 1023, 15, 12.0, 800, 98), 20.0, 6, torch.float32),
    "d17_blobs": (lambda: synth.blob_set(3_000, 17, 255, 8, 8.0, 300, 99), 40.0, 5, torch.float32),
    "wide_range_d2": (lambda: synth.uniform_ints(4_000, 2, 3_000, 100), 40.0, 4, torch.float32),
    "corners_d3": (lambda: (np.random.default_rng(101).integers(0, 2, size=(700, 3)) * 2047)
                   .astype(np.float32), 2047.0, 5, torch.float32),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_fused_matches_oracle(name):
    make, eps, min_pts, dtype = CASES[name]
    P = make()
    assert len(P) <= (4_096 if P.shape[1] <= 4 else 8_192) and P.shape[1] <= 32
    ref = oracle.dbscan(P, eps, min_pts)
    info = {}
    got = gpu_run(P, eps, min_pts, dtype, info=info)
    assert info["fused"] and info["path"] == "fp32", info
    assert info["n_core"] == int(ref[1].sum())
    for g, e, w in zip(got, ref, ("cnt", "core", "label")):
        assert_same(g, e, f"{name} fused {w}")


@pytest.mark.parametrize("name", GOLDEN_FILES)
def test_fused_golden_fixtures(name):
    P, eps, min_pts, exp = load_golden(name)
    got = gpu_run(P, eps, min_pts)
    for g, w in zip(got, ("cnt", "core", "label")):
        assert_same(g, exp[w], f"{name} {w}")


@pytest.mark.parametrize("n,d", [(1, 3), (2, 3), (127, 3), (128, 3), (129, 3), (256, 3), (257, 3),
                                 (1000, 3), (4_095, 3), (4_096, 3), (8_191, 8), (8_192, 8)])
def test_fused_tile_boundaries(n, d):
    P = synth.uniform_ints(n, d, 60 if n < 2000 else 200, seed=n + 7)
    for min_pts in (1, 3):
        ref = oracle.dbscan(P, 6.0 if d == 3 else 14.0, min_pts)
        info = {}
        got = gpu_run(P, 6.0 if d == 3 else 14.0, min_pts, info=info)
        assert info["fused"]
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"n={n} d={d} min_pts={min_pts} {w}")


def test_fused_edge_cases():
    P = np.full((700, 3), 17.0, np.float32)              # all duplicates, eps = 0
    cnt, core, label = gpu_run(P, 0.0, 5)
    assert np.all(cnt == 700) and np.all(core == 1) and np.all(label == 0)
    rng = np.random.default_rng(0)
    P = rng.integers(0, 6, size=(900, 2)).astype(np.float32)
    for eps, mp in ((0.0, 3), (1.0, 5), (2.0, 10_000)):
        ref = oracle.dbscan(P, eps, mp)
        for g, e, w in zip(gpu_run(P, eps, mp), ref, ("cnt", "core", "label")):
            assert_same(g, e, f"eps={eps} min_pts={mp} {w}")
    P = (rng.integers(0, 400, size=(3000, 3)) / 4.0).astype(np.float32)   # dyadic fractions
    for eps in (0.5, 1.25):
        ref = oracle.dbscan(P, eps, 4)
        info = {}
        got = gpu_run(P, eps, 4, info=info)
        assert info["fused"] and not info["exact"]
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"fractional eps={eps} {w}")


def test_fused_and_multi_kernel_paths_agree_and_sizes_dispatch():
    P = synth.scaled("blobs_1m_d3", 4_000, seed=102)
    a = gpu_run(P, 10.0, 8, info=(ia := {}))
    with binding.options(fused=0):
        b = gpu_run(P, 10.0, 8, info=(ib := {}))
    assert ia["fused"] and not ib["fused"] and ib["path"] == "f16"
    for x, y, w in zip(a, b, ("cnt", "core", "label")):
        assert_same(x, y, f"fused vs multi-kernel {w}")
    # just above the size limits, or above the dimension limit: multi-kernel
    info = {}
    gpu_run(synth.scaled("blobs_1m_d3", 4_097, seed=103), 10.0, 8, info=info, counts=False)
    assert not info["fused"]
    info = {}
    gpu_run(synth.uniform_ints(8_193, 8, 200, 108), 14.0, 5, info=info, counts=False)
    assert not info["fused"]
    info = {}
    gpu_run(synth.blob_set(1_000, 33, 127, 4, 4.0, 100, 104), 30.0, 5, info=info, counts=False)
    assert not info["fused"]


def test_fused_entry_points_and_errors():
    P = synth.scaled("blobs_100k_d2", 4_000, seed=105)
    _, core_ref, label_ref = oracle.dbscan(P, 20.0, 10)
    x = torch.from_numpy(P).cuda()
    labels, core = binding.dbscan_fit(x, 20.0, 10)
    assert_same(labels.cpu().numpy(), label_ref, "dbscan_fit labels")
    assert_same(core.cpu().numpy(), core_ref, "dbscan_fit core")
    hl, hc = binding.dbscan_fit_host(torch.from_numpy(P).pin_memory(), 20.0, 10)
    assert_same(hl.numpy(), label_ref, "dbscan_fit_host labels")
    lc, cc = binding.dbscan_fit_culled(x, 20.0, 10)
    assert_same(lc.cpu().numpy(), label_ref, "dbscan_fit_culled labels")
    # a non-finite coordinate is reported, and the context stays usable
    y = torch.tensor([[0.0, 1.0], [float("nan"), 2.0], [3.0, 3.0]], device="cuda")
    ws = binding.workspace_for(y)
    binding.dbscan_fit_ex(y, 1.0, 2, workspace=ws)
    assert binding.dbscan_workspace_status(ws) == binding.Status.INVALID_ARG
    cnt, _, _ = gpu_run(np.zeros((5, 2), np.float32), 0.0, 2)
    assert np.all(cnt == 5)


def test_fused_graph_replay_follows_the_buffers():
    sets = [synth.scaled("blobs_100k_d2", 4_001, seed=s) for s in (106, 107)]
    stream = torch.cuda.Stream()
    x = torch.from_numpy(sets[0]).to("cuda")
    ws = binding.workspace_for(x)
    labels = torch.empty(len(sets[0]), dtype=torch.int32, device="cuda")
    core = torch.empty(len(sets[0]), dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream), binding.options(graphs=1):
        for call in range(4):
            P = sets[call % 2]
            x.copy_(torch.from_numpy(P).to("cuda"))
            binding.dbscan_fit_ex(x, 20.0, 10, labels=labels, is_core=core, workspace=ws,
                                  stream=stream)
            assert binding.dbscan_workspace_status(ws, stream) == 0
            stream.synchronize()
            _, core_ref, label_ref = oracle.dbscan(P, 20.0, 10)
            assert_same(core.cpu().numpy(), core_ref, f"call {call} core flags")
            assert_same(labels.cpu().numpy(), label_ref, f"call {call} labels")
