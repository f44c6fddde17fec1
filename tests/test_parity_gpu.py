"""Element-by-element parity of the CUDA path with the CPU oracle.

Sizes are ones the oracle finishes in seconds while still spanning many
128-point tiles and a ragged last tile; every kernel family (d <= 4 packed,
d > 4 shared-memory, float32 and bfloat16 inputs) is exercised.  Counts,
core flags and labels are integers and must match exactly.
"""
import numpy as np
import pytest
import torch

import oracle
from all_pairs_distance_gb300 import binding, synth
from conftest import GOLDEN_FILES, load_golden
from gpu_util import assert_same, gpu_run

pytestmark = pytest.mark.gpu


def _blobs(n, d, hi, nb, sigma, noise, seed):
    return synth.blob_set(n, d, hi, nb, sigma, noise, seed)


CASES = {
    # name: (points factory, eps, min_pts, dtype)
    "c1_full_2k_d2": (lambda: synth.generate("blobs_2k_d2"), 30.0, 5, torch.float32),
    "c2_like_20k_d2": (lambda: synth.scaled("blobs_100k_d2", 20_000), 20.0, 10, torch.float32),
    "c4_like_20k_d3": (lambda: synth.scaled("blobs_1m_d3", 20_011), 10.0, 8, torch.float32),
    "c3_like_6k_d16": (lambda: synth.scaled("blobs_200k_d16", 6_007), 120.0, 20, torch.float32),
    "c5_like_4k_d64_bf16": (lambda: synth.scaled("blobs_500k_d64", 4_003), 100.0, 16, torch.bfloat16),
    "c5_like_3k_d64_f32": (lambda: synth.scaled("blobs_500k_d64", 3_001, seed=9), 100.0, 16, torch.float32),
    "d1_uniform": (lambda: synth.uniform_ints(5_000, 1, 4_000, 1), 1.0, 3, torch.float32),
    "d1_blobs": (lambda: _blobs(4_100, 1, 4095, 6, 30.0, 400, 2), 2.0, 4, torch.float32),
    "d4_blobs": (lambda: _blobs(9_000, 4, 1023, 20, 10.0, 900, 3), 12.0, 6, torch.float32),
    "d5_blobs": (lambda: _blobs(7_000, 5, 1023, 15, 12.0, 700, 4), 20.0, 6, torch.float32),
    "d8_blobs": (lambda: _blobs(6_000, 8, 255, 12, 6.0, 600, 5), 14.0, 5, torch.float32),
    "d17_blobs": (lambda: _blobs(3_000, 17, 255, 8, 8.0, 300, 6), 40.0, 5, torch.float32),
    "d33_blobs": (lambda: _blobs(2_500, 33, 127, 8, 4.0, 250, 7), 30.0, 5, torch.float32),
    "d16_bf16": (lambda: _blobs(5_000, 16, 255, 10, 6.0, 500, 8), 30.0, 6, torch.bfloat16),
    "d32_bf16": (lambda: _blobs(3_000, 32, 255, 10, 6.0, 300, 10), 45.0, 6, torch.bfloat16),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_parity_with_oracle(name):
    make, eps, min_pts, dtype = CASES[name]
    P = make()
    cnt_ref, core_ref, label_ref = oracle.dbscan(P, eps, min_pts)
    cnt, core, label = gpu_run(P, eps, min_pts, dtype)
    assert_same(cnt, cnt_ref, f"{name} counts")
    assert_same(core, core_ref, f"{name} core flags")
    assert_same(label, label_ref, f"{name} labels")
    # the case must exercise clusters and noise (and, at low d, border points)
    if name.startswith("c"):
        assert core_ref.sum() > 0 and (label_ref == -1).sum() > 0
    if name in ("c1_full_2k_d2", "c2_like_20k_d2", "c4_like_20k_d3"):
        assert ((core_ref == 0) & (label_ref >= 0)).sum() > 0


@pytest.mark.parametrize("name", GOLDEN_FILES)
def test_golden_fixture_on_gpu(name):
    P, eps, min_pts, exp = load_golden(name)
    cnt, core, label = gpu_run(P, eps, min_pts)
    assert_same(cnt, exp["cnt"], "cnt")
    assert_same(core, exp["core"], "core")
    assert_same(label, exp["label"], "label")


@pytest.mark.parametrize("n", [1, 2, 127, 128, 129, 255, 256, 257, 1000])
@pytest.mark.parametrize("d", [2, 3, 6])
def test_tile_boundaries(n, d):
    P = synth.uniform_ints(n, d, 40, seed=n * 10 + d)
    for min_pts in (1, 3):
        ref = oracle.dbscan(P, 6.0, min_pts)
        got = gpu_run(P, 6.0, min_pts)
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"n={n} d={d} min_pts={min_pts} {w}")


def test_n_zero_is_noop():
    x = torch.empty((0, 3), device="cuda")
    labels, core = binding.dbscan_fit_ex(x, 1.0, 2)
    assert labels.numel() == 0 and core.numel() == 0


def test_all_duplicates_one_cluster():
    P = np.full((700, 3), 17.0, np.float32)
    cnt, core, label = gpu_run(P, 0.0, 5)
    assert np.all(cnt == 700) and np.all(core == 1) and np.all(label == 0)


def test_eps_zero_and_min_pts_above_n():
    rng = np.random.default_rng(0)
    P = rng.integers(0, 6, size=(900, 2)).astype(np.float32)   # many duplicates
    for eps, mp in ((0.0, 3), (1.0, 5), (2.0, 10_000)):
        ref = oracle.dbscan(P, eps, mp)
        got = gpu_run(P, eps, mp)
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"eps={eps} min_pts={mp} {w}")


def test_min_pts_one_every_point_is_core():
    P = synth.scaled("blobs_100k_d2", 6_000, seed=11)
    ref = oracle.dbscan(P, 20.0, 1)
    got = gpu_run(P, 20.0, 1)
    assert np.all(got[1] == 1)
    for g, e, w in zip(got, ref, ("cnt", "core", "label")):
        assert_same(g, e, f"min_pts=1 {w}")


@pytest.mark.parametrize("order", ["sorted", "reversed", "interleaved"])
def test_input_order_does_not_matter(order):
    # the kernels sort the points into a locality order of their own; results
    # are defined on input indices, so any input order must match the oracle
    # run on that same order (already sorted input included)
    P = synth.scaled("blobs_1m_d3", 12_000, seed=12)
    if order == "sorted":
        P = P[np.lexsort(P.T[::-1])]
    elif order == "reversed":
        P = P[np.lexsort(P.T[::-1])][::-1]
    else:
        idx = np.lexsort(P.T[::-1])
        P = P[np.concatenate([idx[0::2], idx[1::2]])]
    P = np.ascontiguousarray(P)
    ref = oracle.dbscan(P, 10.0, 8)
    for path in ("fp32", "default"):
        with binding.options(paths=(["fp32"] if path == "fp32" else binding.PATHS_DEFAULT)):
            got = gpu_run(P, 10.0, 8)
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"{order} path={path} {w}")


def test_inclusive_boundary_at_full_range():
    # two points at the ends of [0, 2047] with eps equal to their distance:
    # the squared distance 2047^2 equals eps^2 and must count (<=)
    P = np.array([[0.0], [2047.0]], np.float32)
    cnt, core, label = gpu_run(P, 2047.0, 2)
    assert_same(cnt, [2, 2], "cnt")
    assert_same(label, [0, 0], "label")
    cnt, core, label = gpu_run(P, 2046.0, 2)
    assert_same(cnt, [1, 1], "cnt")


@pytest.mark.parametrize("d,hi", [(3, 2047), (2, 2047), (16, 511)])
def test_extreme_corners_all_pairs(d, hi):
    # corners of the box: the largest squared distance (d * hi^2) sits at the
    # edge of exact float32 integers; eps above it makes every pair a neighbour
    rng = np.random.default_rng(d)
    P = (rng.integers(0, 2, size=(300, d)) * hi).astype(np.float32)
    for eps in (float(hi), float(hi) * np.sqrt(d) + 1.0):
        ref = oracle.dbscan(P, eps, 4)
        got = gpu_run(P, eps, 4)
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"d={d} eps={eps} {w}")


def test_extremes_bf16_d64():
    # rows of all-0 and all-255 in bf16 (largest norms of the d=64 workload)
    rng = np.random.default_rng(3)
    P = (rng.integers(0, 2, size=(400, 64)) * 255).astype(np.float32)
    P[:100] = rng.integers(250, 256, size=(100, 64))
    for eps in (100.0, 2040.0, 2041.0):
        ref = oracle.dbscan(P, eps, 4)
        got = gpu_run(P, eps, 4, torch.bfloat16)
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"eps={eps} {w}")


def test_extremes_bf16_d128():
    # all-0 and all-255 rows at d = 128: the widest operand rows the bf16 path
    # stages (144 elements); the corner distance is 255 * sqrt(128) = 2884.9
    rng = np.random.default_rng(4)
    P = (rng.integers(0, 2, size=(400, 128)) * 255).astype(np.float32)
    P[:100] = rng.integers(250, 256, size=(100, 128))
    for eps in (100.0, 2884.0, 2885.0):
        ref = oracle.dbscan(P, eps, 4)
        info = {}
        got = gpu_run(P, eps, 4, torch.bfloat16, info=info)
        assert info["path"] == "bf16", info
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"eps={eps} {w}")


def test_extremes_bf16_d256():
    # all-0 and all-255 rows at d = 256: 544-byte operand rows, and the
    # exactness bound met with equality (4 S = 2^24 after centring); eps up to
    # 2896 keeps 2 S + thrx within 2^24 (tensor cores), larger eps leaves the
    # data to the CUDA cores, which must agree as well
    rng = np.random.default_rng(5)
    P = (rng.integers(0, 2, size=(600, 256)) * 255).astype(np.float32)
    P[:150] = rng.integers(250, 256, size=(150, 256))
    for eps, path in ((80.0, "bf16"), (2896.0, "bf16"), (4080.0, "fp32"), (4079.0, "fp32")):
        ref = oracle.dbscan(P, eps, 4)
        info = {}
        got = gpu_run(P, eps, 4, torch.bfloat16, info=info)
        assert info["path"] == path, (eps, info)
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"d=256 eps={eps} {w}")


def test_dyadic_fractional_coordinates():
    # quarter-integer coordinates are exact in float32 as well; the
    # non-integer branch of the threshold must still give "<= eps^2"
    rng = np.random.default_rng(7)
    P = (rng.integers(0, 400, size=(3000, 3)) / 4.0).astype(np.float32)
    for eps in (0.5, 1.25, 2.0):
        ref = oracle.dbscan(P, eps, 4)
        got = gpu_run(P, eps, 4)
        for g, e, w in zip(got, ref, ("cnt", "core", "label")):
            assert_same(g, e, f"eps={eps} {w}")


def test_deterministic_repeats():
    P = synth.scaled("blobs_1m_d3", 30_000, seed=77)
    first = gpu_run(P, 10.0, 8)
    for _ in range(4):
        again = gpu_run(P, 10.0, 8)
        for g, e in zip(again, first):
            assert np.array_equal(g, e)


def test_sync_and_host_entry_points_agree():
    P = synth.scaled("blobs_100k_d2", 12_000, seed=5)
    _, core_ref, label_ref = oracle.dbscan(P, 20.0, 10)
    x = torch.from_numpy(P).cuda()
    labels, core = binding.dbscan_fit(x, 20.0, 10)
    assert_same(labels.cpu().numpy(), label_ref, "dbscan_fit labels")
    assert_same(core.cpu().numpy(), core_ref, "dbscan_fit core")
    hl, hc = binding.dbscan_fit_host(torch.from_numpy(P).pin_memory(), 20.0, 10)
    assert_same(hl.numpy(), label_ref, "dbscan_fit_host labels")
    assert_same(hc.numpy(), core_ref, "dbscan_fit_host core")
    hl, hc = binding.dbscan_fit_host(P, 20.0, 10)    # pageable numpy input
    assert_same(hl.numpy(), label_ref, "dbscan_fit_host (pageable) labels")


def test_device_side_errors_and_bad_pointers():
    x = torch.tensor([[0.0, 1.0], [float("nan"), 2.0], [3.0, 3.0]], device="cuda")
    ws = binding.workspace_for(x)
    binding.dbscan_fit_ex(x, 1.0, 2, workspace=ws)
    assert binding.dbscan_workspace_status(ws) == binding.Status.INVALID_ARG
    # a host pointer where device memory is required is refused, not run
    lib = binding.load()
    h = torch.zeros((10, 3))
    lab = torch.empty(10, dtype=torch.int32, device="cuda")
    core = torch.empty(10, dtype=torch.uint8, device="cuda")
    st = lib.dbscan_fit_ex(h.data_ptr(), 0, 10, 3, 1.0, 2, lab.data_ptr(), core.data_ptr(),
                           None, 0, None)
    assert st == binding.Status.INVALID_ARG
    # workspace too small
    y = torch.zeros((1000, 3), device="cuda")
    small = torch.empty(1024, dtype=torch.uint8, device="cuda")
    with pytest.raises(binding.DbscanError):
        binding.dbscan_fit_ex(y, 1.0, 2, workspace=small)
    # the context is still usable afterwards
    cnt, core_, label = gpu_run(np.zeros((5, 2), np.float32), 0.0, 2)
    assert np.all(cnt == 5)


ALL_TC = {"tf32", "bf16", "f16", "f16acc16"}
PATH_CASES = {
    # name: (points, eps, min_pts, dtype, tensor-core paths the data qualifies for)
    "c4_like_12k_d3": (lambda: synth.scaled("blobs_1m_d3", 12_007, seed=31), 10.0, 8, torch.float32,
                       {"tf32", "f16", "f16acc16"}),
    "c2_like_9k_d2": (lambda: synth.scaled("blobs_100k_d2", 9_001, seed=32), 20.0, 10, torch.float32,
                      {"tf32", "f16", "f16acc16"}),
    "c3_like_3k_d16": (lambda: synth.scaled("blobs_200k_d16", 3_001, seed=33), 120.0, 20,
                       torch.float32, {"tf32", "f16"}),
    "c5_like_3k_d64": (lambda: synth.scaled("blobs_500k_d64", 2_999, seed=34), 100.0, 16,
                       torch.bfloat16, {"bf16", "tf32", "f16"}),
    "small_box_d3": (lambda: synth.uniform_ints(4_000, 3, 200, 35), 9.0, 6, torch.float32, ALL_TC),
    "corners_d3": (lambda: (np.random.default_rng(36).integers(0, 2, size=(700, 3)) * 2047)
                   .astype(np.float32), 2047.0, 5, torch.float32, {"tf32", "f16", "f16acc16"}),
    # d = 10 with two threshold digits fills the f16 accumulator's single K = 16 MMA
    "d10_two_digits": (lambda: synth.blob_set(3_000, 10, 511, 12, 20.0, 300, 37), 60.0, 4,
                       torch.float32, {"tf32", "f16", "f16acc16"}),
    # d = 11 no longer fits one K = 16 MMA: the f16 accumulator is not eligible,
    # f16 operands with an f32 accumulator take two K steps
    "d11_blobs": (lambda: synth.blob_set(2_500, 11, 511, 10, 20.0, 250, 38), 60.0, 5,
                  torch.float32, {"tf32", "f16"}),
    # wide rows: 144 bf16/f16 or 136 tf32 elements at d = 128, 72 tf32 elements at
    # d = 64 (a range of 400 is too wide for bf16 and narrow enough for exact tf32
    # and f16)
    "d128_bf16": (lambda: synth.blob_set(2_500, 128, 255, 8, 6.0, 250, 39), 110.0, 5,
                  torch.bfloat16, {"bf16", "f16", "tf32"}),
    "d64_tf32_wide": (lambda: synth.blob_set(2_000, 64, 400, 8, 12.0, 200, 40), 150.0, 5,
                      torch.float32, {"tf32", "f16"}),
    # the widest rows: 272 bf16/f16 elements at d = 256 (one row buffer and
    # one-tile stages in the sweeps)
    "d256_bf16": (lambda: synth.blob_set(2_000, 256, 255, 6, 5.0, 200, 42), 140.0, 5,
                  torch.bfloat16, {"bf16", "f16"}),
    # a threshold constant of three base-2048 digits (eps^2 >= 2048^2): f16
    # operands hold at most two, tf32 takes three
    "d3_three_digits": (lambda: synth.uniform_ints(1_500, 3, 2047, 41), 2100.0, 40, torch.float32,
                        {"tf32"}),
}


@pytest.mark.parametrize("path", ["fp32", "tf32", "bf16", "f16", "f16acc16"])
@pytest.mark.parametrize("name", sorted(PATH_CASES))
def test_parity_every_path(name, path):
    # the library picks a path per call from the data; allowing one path only
    # narrows the choice (a path the data cannot use exactly falls back to CUDA
    # cores)
    make, eps, min_pts, dtype, eligible = PATH_CASES[name]
    P = make()
    ref = oracle.dbscan(P, eps, min_pts)
    info = {}
    with binding.options(paths=[path]):
        got = gpu_run(P, eps, min_pts, dtype, info=info)
    assert info["path"] == (path if path in eligible else "fp32")
    assert info["exact"]
    assert info["n_core"] == int(ref[1].sum())
    for g, e, w in zip(got, ref, ("cnt", "core", "label")):
        assert_same(g, e, f"{name} [{path}] {w}")


def test_default_path_choice():
    # by default integer data in a 256-wide box go to bf16, in a 2048-wide box
    # to f16 (both f32 accumulation), threshold constants too large for f16
    # operands to tf32, and wider or fractional data stay on CUDA cores; the
    # f16 accumulator is never chosen unless allowed
    for P, eps, expect in ((synth.uniform_ints(3000, 3, 2047, 1), 4.0, "f16"),
                           (synth.uniform_ints(3000, 3, 255, 2), 4.0, "bf16"),
                           (synth.uniform_ints(3000, 16, 255, 5), 4.0, "bf16"),
                           (synth.uniform_ints(3000, 12, 511, 6), 4.0, "f16"),
                           (synth.uniform_ints(3000, 128, 255, 7), 4.0, "bf16"),
                           (synth.uniform_ints(1500, 256, 255, 10), 4.0, "bf16"),
                           (synth.uniform_ints(3000, 64, 400, 8), 4.0, "f16"),
                           (synth.uniform_ints(3000, 3, 2047, 9), 2100.0, "tf32"),
                           (synth.uniform_ints(3000, 2, 3000, 3), 4.0, "fp32"),
                           (synth.uniform_ints(3000, 2, 100, 4) + np.float32(0.5), 4.0, "fp32")):
        info = {}
        gpu_run(P, eps, 3, info=info, counts=False)
        assert info["path"] == expect, (expect, info)
    with binding.options(paths=binding.PATHS_DEFAULT | binding.PATH_BITS["f16acc16"]):
        info = {}
        gpu_run(synth.uniform_ints(3000, 3, 2047, 1), 4.0, 3, info=info, counts=False)
        assert info["path"] == "f16acc16", info


def gpu_run_culled(P, eps, min_pts, dtype=torch.float32):
    x = torch.from_numpy(np.ascontiguousarray(P)).to("cuda").to(dtype)
    ws = binding.workspace_for(x)
    labels, core = binding.dbscan_fit_culled(x, eps, min_pts, workspace=ws)
    st = binding.dbscan_workspace_status(ws)
    assert st == 0, binding.dbscan_strerror(st)
    return core.cpu().numpy(), labels.cpu().numpy()


CULL_CASES = {
    # tile culling engages (integer data, d <= 8) or must leave results untouched
    "c1_full_2k_d2": (lambda: synth.generate("blobs_2k_d2"), 30.0, 5, torch.float32),
    "c2_like_20k_d2": (lambda: synth.scaled("blobs_100k_d2", 20_000, seed=41), 20.0, 10, torch.float32),
    "c4_like_20k_d3": (lambda: synth.scaled("blobs_1m_d3", 20_011, seed=42), 10.0, 8, torch.float32),
    "d8_blobs": (lambda: _blobs(6_000, 8, 255, 12, 6.0, 600, 43), 14.0, 5, torch.float32),
    "d1_blobs": (lambda: _blobs(4_100, 1, 4095, 6, 30.0, 400, 44), 2.0, 4, torch.float32),
    "corners_d3": (lambda: (np.random.default_rng(45).integers(0, 2, size=(700, 3)) * 2047)
                   .astype(np.float32), 2047.0, 5, torch.float32),
    "d16_blobs": (lambda: synth.scaled("blobs_200k_d16", 4_001, seed=46), 120.0, 20, torch.float32),
    "d33_no_cull": (lambda: _blobs(2_500, 33, 127, 8, 4.0, 250, 48), 30.0, 5, torch.float32),
    # dyadic fractions: the float test is exact, the tile test keeps a margin
    "fractional_d3": (lambda: synth.scaled("blobs_1m_d3", 5_003, seed=47) * np.float32(0.5),
                           5.0, 8, torch.float32),
}


@pytest.mark.parametrize("path", ["default", "tf32", "bf16", "f16", "fp32"])
@pytest.mark.parametrize("name", sorted(CULL_CASES))
def test_culled_matches_oracle(name, path):
    make, eps, min_pts, dtype = CULL_CASES[name]
    P = make()
    _, core_ref, label_ref = oracle.dbscan(P, eps, min_pts)
    with binding.options(paths=binding.PATHS_DEFAULT if path == "default" else [path]):
        core, label = gpu_run_culled(P, eps, min_pts, dtype)
    assert_same(core, core_ref, f"{name} [{path}] culled core flags")
    assert_same(label, label_ref, f"{name} [{path}] culled labels")


ROW_CASES = {
    # the tensor-core sweeps take one or two row blocks per unit; the rows switch
    # forces either for every sweep or per sweep (count, union, border)
    "c4_like_9k_d3": (lambda: synth.scaled("blobs_1m_d3", 9_001, seed=51), 10.0, 8, torch.float32),
    "c5_like_2k_d64": (lambda: synth.scaled("blobs_500k_d64", 2_177, seed=52), 100.0, 16,
                       torch.bfloat16),
    "d16_blobs": (lambda: synth.scaled("blobs_200k_d16", 3_203, seed=53), 120.0, 20, torch.float32),
    # 9 row tiles: the last unit of two row blocks holds one
    "odd_tiles_d2": (lambda: synth.scaled("blobs_100k_d2", 1_074, seed=54), 20.0, 4, torch.float32),
    # fractional data: exact tests off, no tile culling, tensor cores not used
    "fractional_d3": (lambda: synth.scaled("blobs_1m_d3", 4_001, seed=55) * np.float32(0.5), 5.0, 8,
                      torch.float32),
}


@pytest.mark.parametrize("rows", ["1", "2", "212", "121"])
@pytest.mark.parametrize("name", sorted(ROW_CASES))
def test_row_units_match_oracle(name, rows):
    make, eps, min_pts, dtype = ROW_CASES[name]
    P = make()
    assert len(P) == {"c4_like_9k_d3": 9_001, "c5_like_2k_d64": 2_177, "d16_blobs": 3_203,
                      "odd_tiles_d2": 1_074, "fractional_d3": 4_001}[name]
    cnt_ref, core_ref, label_ref = oracle.dbscan(P, eps, min_pts)
    r = [int(c) for c in rows] * (3 if len(rows) == 1 else 1)
    with binding.options(rows=r):
        cnt, core, label = gpu_run(P, eps, min_pts, dtype)
        core_c, label_c = gpu_run_culled(P, eps, min_pts, dtype)
    assert_same(cnt, cnt_ref, f"{name} [rows {rows}] counts")
    assert_same(core, core_ref, f"{name} [rows {rows}] core flags")
    assert_same(label, label_ref, f"{name} [rows {rows}] labels")
    assert_same(core_c, core_ref, f"{name} [rows {rows}] culled core flags")
    assert_same(label_c, label_ref, f"{name} [rows {rows}] culled labels")


SPAN_CASES = {
    # more than 256 column tiles (the CUDA-core sweeps test the boxes of at most
    # 256 column tiles at a time): every span boundary of the union and border
    # sweeps, and of the count sweep when the caller asks for culling
    "d3_41k": (lambda: synth.scaled("blobs_1m_d3", 41_003, seed=61), 10.0, 8),
    "d2_40k": (lambda: synth.scaled("blobs_100k_d2", 40_001, seed=62), 20.0, 10),
    "d8_34k": (lambda: _blobs(34_000, 8, 255, 40, 6.0, 3_400, 63), 14.0, 5),
    # fractional coordinates: the tile test with its rounding margin
    "d3_fractional_34k": (lambda: synth.scaled("blobs_1m_d3", 34_001, seed=64) * np.float32(0.5),
                          5.0, 8),
}


@pytest.mark.parametrize("culled", [False, True])
@pytest.mark.parametrize("name", sorted(SPAN_CASES))
def test_cuda_core_culling_spans(name, culled):
    make, eps, min_pts = SPAN_CASES[name]
    P = make()
    assert len(P) > 256 * 128
    cnt_ref, core_ref, label_ref = oracle.dbscan(P, eps, min_pts)
    with binding.options(paths=["fp32"]):
        if culled:
            core, label = gpu_run_culled(P, eps, min_pts)
        else:
            info = {}
            cnt, core, label = gpu_run(P, eps, min_pts, info=info)
            assert info["path"] == "fp32"
            assert_same(cnt, cnt_ref, f"{name} counts")
    assert_same(core, core_ref, f"{name} core flags")
    assert_same(label, label_ref, f"{name} labels")
    assert core_ref.sum() > 0 and (label_ref == -1).sum() > 0


FLOAT_CASES = {
    # data off the exact path (non-integer, or a range too wide for the
    # exactness flag), where the tile test keeps every tile pair within eps
    # plus a bound on the float test's rounding; the coordinates are chosen so
    # that the float arithmetic itself is exact (multiples of 1/8, or integers
    # whose sums stay below 2^24), so the sweeps are deterministic and the
    # oracle decides every pair the same way; more than 256 row tiles
    "d3_eighths_41k": (lambda: synth.scaled("blobs_1m_d3", 41_003, seed=81) * np.float32(0.125),
                       1.25, 8),
    "d2_eighths_34k": (lambda: synth.scaled("blobs_100k_d2", 34_001, seed=82) * np.float32(0.125),
                       2.5, 10),
    "d16_eighths_34k": (lambda: synth.scaled("blobs_200k_d16", 34_001, seed=83) * np.float32(0.125),
                        15.0, 20),
    # integers over [0, 3070]: range^2 sum >= 2^24 (not flagged exact), sums below 2^24
    "d2_wide_ints_34k": (lambda: np.rint(synth.scaled("blobs_100k_d2", 34_001, seed=84) *
                                         np.float32(1.5)).astype(np.float32), 30.0, 10),
}


_FLOAT_REF = {}


@pytest.mark.parametrize("culled", [False, True])
@pytest.mark.parametrize("name", sorted(FLOAT_CASES))
def test_float_tile_test_matches_oracle(name, culled):
    make, eps, min_pts = FLOAT_CASES[name]
    P = make()
    if name not in _FLOAT_REF:   # one oracle run per case for both entry points
        _FLOAT_REF[name] = oracle.dbscan(P, eps, min_pts)
    cnt_ref, core_ref, label_ref = _FLOAT_REF[name]
    for cull in (0, 1):
        with binding.options(cull=cull):
            if culled:
                core, labels = gpu_run_culled(P, eps, min_pts)
            else:
                info = {}
                cnt, core, labels = gpu_run(P, eps, min_pts, info=info)
                assert info["path"] == "fp32" and not info["exact"], info
                assert_same(cnt, cnt_ref, f"{name} cull={cull} counts")
        assert_same(core, core_ref, f"{name} cull={cull} core flags")
        assert_same(labels, label_ref, f"{name} cull={cull} labels")
    assert core_ref.sum() > 0 and (label_ref == -1).sum() > 0
    assert len(np.unique(label_ref[label_ref >= 0])) > 1


def _jittered(P, scale, seed):
    # continuous (non-dyadic) float coordinates
    rng = np.random.default_rng(seed)
    return (P * np.float32(scale) + rng.random(P.shape, dtype=np.float32) * np.float32(scale))


ACCURACY_CASES = {
    # float data whose spread is large against eps (range ~200 against eps 1,
    # ~190 against 44): the direct form of the test is accurate to a few
    # roundings of d^2 itself
    "d3_41k": (lambda: _jittered(synth.scaled("blobs_1m_d3", 41_003, seed=91), 0.1, 11), 1.0, 8),
    "d16_34k": (lambda: _jittered(synth.scaled("blobs_200k_d16", 34_001, seed=93), 0.37, 13), 44.4, 20),
}


@pytest.mark.parametrize("name", sorted(ACCURACY_CASES))
def test_float_data_counts_within_rounding_and_repeatable(name):
    # on float data a pair can be decided either way only when its squared
    # distance lies within a relative 1e-5 of eps^2: every count lies between
    # the oracle's counts at those two radii, and a second call (the points
    # may land in other tiles) repeats every count, flag and label
    make, eps, min_pts = ACCURACY_CASES[name]
    P = make()
    lo = oracle.counts(P, eps * np.sqrt(1.0 - 1e-5))
    hi = oracle.counts(P, eps * np.sqrt(1.0 + 1e-5))
    info = {}
    first = gpu_run(P, eps, min_pts, info=info)
    assert info["path"] == "fp32" and not info["exact"], info
    cnt, core, labels = first
    bad = np.flatnonzero((cnt < lo) | (cnt > hi))
    assert bad.size == 0, (f"{bad.size} counts outside the rounding window, first at {bad[:8].tolist()}: "
                           f"got {cnt[bad[:8]].tolist()} in [{lo[bad[:8]].tolist()}, "
                           f"{hi[bad[:8]].tolist()}]")
    assert np.all(core >= (lo >= min_pts)) and np.all(core <= (hi >= min_pts))
    second = gpu_run(P, eps, min_pts)
    for g, e, w in zip(second, first, ("counts", "core flags", "labels")):
        assert_same(g, e, f"{name} repeated call {w}")
