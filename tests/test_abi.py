"""C-ABI checks that need no GPU: the library builds for sm_103a, loads,
exports every function include/dbscan.h declares, and rejects bad arguments
on the host before touching the device."""
import ctypes
import os
import re

import pytest

from all_pairs_distance_gb300 import build as lib_build

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dbscan.h")


@pytest.fixture(scope="module")
def lib():
    path = lib_build.build()
    return ctypes.CDLL(path)


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(dbscan_\w+)\s*\(", src)))


def test_header_declares_the_boundary():
    names = declared_functions()
    for must in ("dbscan_fit", "dbscan_fit_ex", "dbscan_workspace_size", "dbscan_strerror"):
        assert must in names


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), f"{name} declared in dbscan.h but not exported"


def test_strerror(lib):
    lib.dbscan_strerror.restype = ctypes.c_char_p
    lib.dbscan_strerror.argtypes = [ctypes.c_int]
    for code in range(-5, 1):
        assert lib.dbscan_strerror(code).startswith(b"DBSCAN_")
    assert b"unknown" in lib.dbscan_strerror(42)


def test_workspace_size(lib):
    f = lib.dbscan_workspace_size
    f.restype = ctypes.c_size_t
    f.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
    assert f(-1, 3, 0) == 0            # negative n
    assert f(10, 0, 0) == 0            # d < 1
    assert f(10, 257, 0) == 0          # d above the maximum
    assert f(10, 3, 1) == 0            # bf16 needs d % 16 == 0
    assert f(10, 3, 7) == 0            # unknown dtype
    assert f(1 << 31, 3, 0) == 0       # n beyond int32 labels
    assert f(0, 3, 0) > 0
    small, big = f(1000, 3, 0), f(1_000_000, 3, 0)
    assert 0 < small < big
    # O(N d) memory: no N x N term anywhere
    assert big < 200 * 1_000_000 * 4
    assert f(1_000_000, 3, 0) % 256 == 0
    assert f(500_000, 64, 1) > f(500_000, 16, 1)


def _fit_ex(lib):
    f = lib.dbscan_fit_ex
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    f.argtypes = [P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                  ctypes.c_int32, P, P, P, ctypes.c_size_t, P]
    return f


def test_host_side_argument_errors(lib):
    f = _fit_ex(lib)
    fake = ctypes.c_void_p(0x1000)   # never dereferenced: these calls fail validation first
    INVALID, UNSUP = -1, -2
    assert f(fake, 0, -5, 3, 1.0, 2, fake, fake, None, 0, None) == INVALID
    assert f(fake, 0, 10, 0, 1.0, 2, fake, fake, None, 0, None) == INVALID
    assert f(fake, 0, 10, 300, 1.0, 2, fake, fake, None, 0, None) == UNSUP
    assert f(fake, 1, 10, 3, 1.0, 2, fake, fake, None, 0, None) == UNSUP
    assert f(fake, 5, 10, 3, 1.0, 2, fake, fake, None, 0, None) == INVALID
    assert f(fake, 0, 10, 3, -1.0, 2, fake, fake, None, 0, None) == INVALID
    assert f(fake, 0, 10, 3, float("nan"), 2, fake, fake, None, 0, None) == INVALID
    assert f(fake, 0, 10, 3, float("inf"), 2, fake, fake, None, 0, None) == INVALID
    assert f(fake, 0, 10, 3, 1.0, 0, fake, fake, None, 0, None) == INVALID
    assert f(None, 0, 10, 3, 1.0, 2, fake, fake, None, 0, None) == INVALID
    assert f(fake, 0, 10, 3, 1.0, 2, None, fake, None, 0, None) == INVALID
    assert f(fake, 0, 10, 3, 1.0, 2, fake, None, None, 0, None) == INVALID
    assert f(fake, 0, (1 << 31), 3, 1.0, 2, fake, fake, None, 0, None) == UNSUP
    # workspace too small, or not 256-byte aligned
    assert f(fake, 0, 10, 3, 1.0, 2, fake, fake, ctypes.c_void_p(0x10000), 16, None) == INVALID
    assert f(fake, 0, 10, 3, 1.0, 2, fake, fake, ctypes.c_void_p(0x10010), 1 << 30, None) == INVALID
    # n == 0 is a no-op, whatever the pointers
    assert f(None, 0, 0, 3, 1.0, 2, None, None, None, 0, None) == 0


def test_compact_labels_host_side_errors(lib):
    f = lib.dbscan_compact_labels
    f.restype = ctypes.c_int
    P = ctypes.c_void_p
    f.argtypes = [P, ctypes.c_int64, P, P, P]
    INVALID, UNSUP = -1, -2
    k = ctypes.c_int32(-7)
    assert f(None, -1, None, ctypes.byref(k), None) == INVALID       # negative n
    assert f(None, 10, None, None, None) == INVALID                  # no place for k
    assert f(None, 1 << 31, None, ctypes.byref(k), None) == UNSUP    # beyond int32 labels
    assert f(None, 10, None, ctypes.byref(k), None) == INVALID       # null buffers with n > 0
    assert k.value == -7                                             # untouched on error
    assert f(None, 0, None, ctypes.byref(k), None) == 0               # n == 0: k = 0
    assert k.value == 0


def test_options_roundtrip_and_validation(lib, monkeypatch):
    # the tuning switches are process-wide host state: no GPU involved
    from all_pairs_distance_gb300 import binding
    binding.dbscan_set_options(reset=True)
    try:
        o = binding.dbscan_get_options()
        assert o == {"paths": binding.PATHS_DEFAULT, "rows": (0, 0, 0), "graphs": 1, "fused": 1,
                     "cull": 1} or \
            os.environ.get("DBSCAN_FORCE_PATH") or os.environ.get("DBSCAN_TC_ROWS") or \
            os.environ.get("DBSCAN_GRAPHS") or os.environ.get("DBSCAN_FUSED") or \
            os.environ.get("DBSCAN_CULL")
        binding.dbscan_set_options(paths=["f16"], rows=(1, 2, 1), graphs=0, fused=0, cull=0)
        want = {"paths": 4, "rows": (1, 2, 1), "graphs": 0, "fused": 0, "cull": 0}
        assert binding.dbscan_get_options() == want
        with binding.options(paths=["fp32"], rows=2, fused=1, cull=1):
            assert binding.dbscan_get_options() == {"paths": 0, "rows": (2, 2, 2), "graphs": 0,
                                                    "fused": 1, "cull": 1}
        assert binding.dbscan_get_options() == want
        # out-of-range switches are refused and leave the state alone
        bad = binding.Options()
        bad.paths = 16
        assert lib.dbscan_set_options(ctypes.byref(bad)) == -1
        bad.paths, bad.rows[1] = 1, 3
        assert lib.dbscan_set_options(ctypes.byref(bad)) == -1
        bad.rows[1], bad.graphs = 0, 2
        assert lib.dbscan_set_options(ctypes.byref(bad)) == -1
        bad.graphs, bad.fused = 1, 5
        assert lib.dbscan_set_options(ctypes.byref(bad)) == -1
        bad.fused, bad.cull = 1, 2
        assert lib.dbscan_set_options(ctypes.byref(bad)) == -1
        assert lib.dbscan_get_options(None) == -1
        assert binding.dbscan_get_options() == want
        # the environment is read once per process and again only on a reset
        monkeypatch.setenv("DBSCAN_FORCE_PATH", "f16acc16")
        monkeypatch.setenv("DBSCAN_TC_ROWS", "212")
        monkeypatch.setenv("DBSCAN_GRAPHS", "0")
        monkeypatch.setenv("DBSCAN_FUSED", "0")
        monkeypatch.setenv("DBSCAN_CULL", "0")
        assert binding.dbscan_get_options()["paths"] == 4
        binding.dbscan_set_options(reset=True)
        assert binding.dbscan_get_options() == {"paths": 8, "rows": (2, 1, 2), "graphs": 0,
                                                "fused": 0, "cull": 0}
    finally:
        monkeypatch.delenv("DBSCAN_FORCE_PATH", raising=False)
        monkeypatch.delenv("DBSCAN_TC_ROWS", raising=False)
        monkeypatch.delenv("DBSCAN_GRAPHS", raising=False)
        monkeypatch.delenv("DBSCAN_FUSED", raising=False)
        monkeypatch.delenv("DBSCAN_CULL", raising=False)
        binding.dbscan_set_options(reset=True)


def test_shard_host_side_checks(lib):
    # argument errors are found on the host before any device work
    f = lib.dbscan_fit_shard
    P = ctypes.c_void_p
    f.argtypes = [ctypes.c_int32, P, ctypes.c_int32, ctypes.c_int64, ctypes.c_int32, ctypes.c_float,
                  ctypes.c_int32, ctypes.c_int32, ctypes.c_int32, P, P, P, P, ctypes.c_size_t, P]
    f.restype = ctypes.c_int
    fake = ctypes.c_void_p(0x1000)
    INVALID, UNSUP = -1, -2
    for stage, rank, world in ((-1, 0, 1), (5, 0, 1), (0, 1, 1), (0, -1, 2), (0, 0, 0)):
        assert f(stage, fake, 0, 10, 3, 1.0, 2, rank, world, None, None, None, fake, 1 << 20, None) == INVALID
    assert f(0, fake, 0, 10, 3, 1.0, 2, 0, 1, None, None, None, None, 0, None) == INVALID   # no workspace
    assert f(0, fake, 0, 10, 300, 1.0, 2, 0, 1, None, None, None, fake, 1 << 20, None) == UNSUP
    assert f(0, fake, 0, 10, 3, -1.0, 2, 0, 1, None, None, None, fake, 1 << 20, None) == INVALID
    assert f(2, None, 0, 0, 3, 1.0, 2, 0, 2, None, None, None, None, 0, None) == 0   # n == 0: no-op
    # the combined buffers lie inside the workspace, one int per point each
    g = lib.dbscan_shard_buffer
    g.argtypes = [P, ctypes.c_int64, ctypes.c_int32, ctypes.c_int32, P, P]
    g.restype = ctypes.c_int
    size = lib.dbscan_workspace_size
    size.restype = ctypes.c_size_t
    size.argtypes = [ctypes.c_int64, ctypes.c_int32, ctypes.c_int32]
    base = 1 << 32
    total = size(50_000, 3, 0)
    spans = []
    for which in (0, 1, 2):
        ptr, cnt = ctypes.c_void_p(), ctypes.c_int64()
        assert g(ctypes.c_void_p(base), 50_000, 3, which, ctypes.byref(ptr), ctypes.byref(cnt)) == 0
        assert cnt.value == 50_000 and base <= ptr.value and ptr.value + 4 * cnt.value <= base + total
        spans.append((ptr.value, ptr.value + 4 * cnt.value))
    for a in range(3):
        for b in range(a):
            assert spans[a][1] <= spans[b][0] or spans[b][1] <= spans[a][0]
    ptr, cnt = ctypes.c_void_p(), ctypes.c_int64()
    assert g(ctypes.c_void_p(base), 50_000, 3, 3, ctypes.byref(ptr), ctypes.byref(cnt)) == INVALID
