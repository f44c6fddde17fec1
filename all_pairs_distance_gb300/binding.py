"""ctypes binding of ``include/dbscan.h`` -- argument marshalling only.

Every step of the computation runs in the CUDA library; these functions pass
tensor pointers, sizes and the current torch stream through the C ABI and turn
status codes into exceptions.  There is no CPU path: if the library is not
built (``__graft_entry__.build()``), every call raises.
"""
from __future__ import annotations

import contextlib
import ctypes
import enum
import os
import threading

import numpy as np
import torch

from .build import LIB as _LIB_PATH


class Status(enum.IntEnum):
    OK = 0
    INVALID_ARG = -1
    UNSUPPORTED = -2
    ALLOC = -3
    CUDA = -4
    INTERNAL = -5


DTYPES = {torch.float32: 0, torch.bfloat16: 1}

# Tensor-core path bits of dbscan_options.paths (dbscan.h DBSCAN_PATH_*).
PATH_BITS = {"tf32": 1, "bf16": 2, "f16": 4, "f16acc16": 8}
PATHS_DEFAULT = 1 | 2 | 4


class Options(ctypes.Structure):
    _fields_ = [("paths", ctypes.c_uint32), ("rows", ctypes.c_int32 * 3),
                ("graphs", ctypes.c_int32), ("fused", ctypes.c_int32), ("cull", ctypes.c_int32)]


class DbscanError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = int(status)
        super().__init__(f"{where}: {dbscan_strerror(status)} ({status})")


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _LIB_PATH


def load():
    """Load the CUDA library; raises when it has not been built."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"CUDA library not built: {_LIB_PATH} is missing "
                               "(run __graft_entry__.build())")
        lib = ctypes.CDLL(_LIB_PATH)
        P, i64, i32, f32, sz = (ctypes.c_void_p, ctypes.c_int64, ctypes.c_int32,
                                ctypes.c_float, ctypes.c_size_t)
        lib.dbscan_fit.argtypes = [P, i64, i32, f32, i32, P, P]
        lib.dbscan_fit.restype = ctypes.c_int
        lib.dbscan_fit_ex.argtypes = [P, i32, i64, i32, f32, i32, P, P, P, sz, P]
        lib.dbscan_fit_ex.restype = ctypes.c_int
        lib.dbscan_fit_culled.argtypes = [P, i32, i64, i32, f32, i32, P, P, P, sz, P]
        lib.dbscan_fit_culled.restype = ctypes.c_int
        lib.dbscan_fit_host.argtypes = [P, i32, i64, i32, f32, i32, P, P, P]
        lib.dbscan_fit_host.restype = ctypes.c_int
        lib.dbscan_compact_labels.argtypes = [P, i64, P, P, P]
        lib.dbscan_compact_labels.restype = ctypes.c_int
        lib.dbscan_neighbor_counts.argtypes = [P, i32, i64, i32, f32, P, P, sz, P]
        lib.dbscan_neighbor_counts.restype = ctypes.c_int
        lib.dbscan_workspace_size.argtypes = [i64, i32, i32]
        lib.dbscan_workspace_size.restype = sz
        lib.dbscan_workspace_status.argtypes = [P, P]
        lib.dbscan_workspace_status.restype = ctypes.c_int
        lib.dbscan_workspace_info.argtypes = [P, P, P, i32]
        lib.dbscan_workspace_info.restype = ctypes.c_int
        lib.dbscan_profile_begin.argtypes = []
        lib.dbscan_profile_begin.restype = ctypes.c_int
        lib.dbscan_profile_end.argtypes = [P, i32, P, P]
        lib.dbscan_profile_end.restype = ctypes.c_int
        lib.dbscan_strerror.argtypes = [ctypes.c_int]
        lib.dbscan_strerror.restype = ctypes.c_char_p
        lib.dbscan_fit_shard.argtypes = [i32, P, i32, i64, i32, f32, i32, i32, i32, P, P, P, P, sz, P]
        lib.dbscan_fit_shard.restype = ctypes.c_int
        lib.dbscan_shard_buffer.argtypes = [P, i64, i32, i32, P, P]
        lib.dbscan_shard_buffer.restype = ctypes.c_int
        lib.dbscan_set_options.argtypes = [P]
        lib.dbscan_set_options.restype = ctypes.c_int
        lib.dbscan_get_options.argtypes = [P]
        lib.dbscan_get_options.restype = ctypes.c_int
        _lib = lib
        return _lib


def _check(st, where):
    if st != 0:
        raise DbscanError(st, where)


def _stream_handle(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _points(points: torch.Tensor):
    if points.dim() != 2:
        raise ValueError("points must be [n, d]")
    if points.dtype not in DTYPES:
        raise TypeError("points must be float32 or bfloat16")
    return points.contiguous()


def dbscan_get_options() -> dict:
    """The process-wide tuning switches in force."""
    o = Options()
    _check(load().dbscan_get_options(ctypes.byref(o)), "dbscan_get_options")
    return {"paths": int(o.paths), "rows": tuple(int(r) for r in o.rows), "graphs": int(o.graphs),
            "fused": int(o.fused), "cull": int(o.cull)}


def dbscan_set_options(paths=None, rows=None, graphs=None, fused=None, cull=None, *,
                       reset=False) -> None:
    """Change the switches (arguments left None keep their value); ``paths``
    is a bit mask or an iterable of names from PATH_BITS ("fp32" alone, or an
    empty iterable, allows CUDA cores only); ``rows`` one int for every sweep
    or three (count, union, border); ``fused`` 0 keeps small problems on the
    multi-kernel path; ``cull`` 0 makes every sweep visit every tile pair;
    ``reset`` restores the defaults."""
    lib = load()
    if reset:
        _check(lib.dbscan_set_options(None), "dbscan_set_options")
        return
    cur = dbscan_get_options()
    o = Options()
    if paths is None:
        o.paths = cur["paths"]
    elif isinstance(paths, int):
        o.paths = paths
    else:
        names = [paths] if isinstance(paths, str) else list(paths)
        o.paths = sum(PATH_BITS[p] for p in names if p != "fp32")
    r = cur["rows"] if rows is None else ((rows,) * 3 if isinstance(rows, int) else tuple(rows))
    for i in range(3):
        o.rows[i] = int(r[i])
    o.graphs = cur["graphs"] if graphs is None else int(bool(graphs))
    o.fused = cur["fused"] if fused is None else int(bool(fused))
    o.cull = cur["cull"] if cull is None else int(bool(cull))
    _check(lib.dbscan_set_options(ctypes.byref(o)), "dbscan_set_options")


@contextlib.contextmanager
def options(**kw):
    """Switches changed inside a ``with`` block, restored afterwards."""
    saved = dbscan_get_options()
    dbscan_set_options(**kw)
    try:
        yield
    finally:
        dbscan_set_options(paths=saved["paths"], rows=saved["rows"], graphs=saved["graphs"],
                           fused=saved["fused"], cull=saved["cull"])


SHARD_COUNTS, SHARD_PARENTS, SHARD_ORDER = 0, 1, 2


def dbscan_fit_shard(stage: int, points: torch.Tensor, eps: float, min_pts: int, rank: int,
                     world: int, *, workspace: torch.Tensor, labels=None, is_core=None,
                     gathered=None, stream=None) -> None:
    """One stage (0-4) of the sharded pipeline on this rank (dbscan.h)."""
    p = _points(points)
    n, d = p.shape
    ptr = lambda t: None if t is None else t.data_ptr()
    _check(load().dbscan_fit_shard(int(stage), p.data_ptr(), DTYPES[p.dtype], n, d, float(eps),
                                   int(min_pts), int(rank), int(world), ptr(gathered), ptr(labels),
                                   ptr(is_core), workspace.data_ptr(), workspace.numel(),
                                   _stream_handle(stream)), f"dbscan_fit_shard stage {stage}")


def dbscan_shard_buffer(workspace: torch.Tensor, n: int, d: int, which: int) -> torch.Tensor:
    """The int32 workspace array the ranks combine between stages, as a view."""
    ptr = ctypes.c_void_p()
    count = ctypes.c_int64()
    _check(load().dbscan_shard_buffer(workspace.data_ptr(), int(n), int(d), int(which),
                                      ctypes.byref(ptr), ctypes.byref(count)), "dbscan_shard_buffer")
    off = ptr.value - workspace.data_ptr()
    return workspace[off:off + 4 * count.value].view(torch.int32)


def dbscan_strerror(status: int) -> str:
    return load().dbscan_strerror(int(status)).decode()


def dbscan_workspace_size(n: int, d: int, dtype=torch.float32) -> int:
    code = DTYPES[dtype] if isinstance(dtype, torch.dtype) else int(dtype)
    return int(load().dbscan_workspace_size(int(n), int(d), code))


def workspace_for(points: torch.Tensor) -> torch.Tensor:
    """A torch-owned workspace big enough for ``points`` (256-byte aligned)."""
    n, d = points.shape
    nbytes = dbscan_workspace_size(n, d, points.dtype)
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=points.device)


def dbscan_fit(points: torch.Tensor, eps: float, min_pts: int):
    """Synchronous float32 DBSCAN on device points -> (labels int32, is_core uint8)."""
    p = _points(points)
    n, d = p.shape
    labels = torch.empty(n, dtype=torch.int32, device=p.device)
    is_core = torch.empty(n, dtype=torch.uint8, device=p.device)
    _check(load().dbscan_fit(p.data_ptr(), n, d, float(eps), int(min_pts),
                             labels.data_ptr(), is_core.data_ptr()), "dbscan_fit")
    return labels, is_core


def dbscan_fit_ex(points: torch.Tensor, eps: float, min_pts: int, *, labels=None,
                  is_core=None, workspace=None, stream=None):
    """Asynchronous DBSCAN on the current torch stream with a torch-owned
    workspace -> (labels, is_core).  Device-side errors: dbscan_workspace_status."""
    p = _points(points)
    n, d = p.shape
    if labels is None:
        labels = torch.empty(n, dtype=torch.int32, device=p.device)
    if is_core is None:
        is_core = torch.empty(n, dtype=torch.uint8, device=p.device)
    if workspace is None:
        workspace = workspace_for(p)
    _check(load().dbscan_fit_ex(p.data_ptr(), DTYPES[p.dtype], n, d, float(eps), int(min_pts),
                                labels.data_ptr(), is_core.data_ptr(), workspace.data_ptr(),
                                workspace.numel(), _stream_handle(stream)), "dbscan_fit_ex")
    return labels, is_core



def dbscan_fit_culled(points: torch.Tensor, eps: float, min_pts: int, *, labels=None,
                  is_core=None, workspace=None, stream=None):
    """dbscan_fit_ex with tile culling (tile pairs whose bounding boxes are eps
    or more apart are skipped; identical results for exact data, d <= 64)."""
    p = _points(points)
    n, d = p.shape
    if labels is None:
        labels = torch.empty(n, dtype=torch.int32, device=p.device)
    if is_core is None:
        is_core = torch.empty(n, dtype=torch.uint8, device=p.device)
    if workspace is None:
        workspace = workspace_for(p)
    _check(load().dbscan_fit_culled(p.data_ptr(), DTYPES[p.dtype], n, d, float(eps), int(min_pts),
                                labels.data_ptr(), is_core.data_ptr(), workspace.data_ptr(),
                                workspace.numel(), _stream_handle(stream)), "dbscan_fit_culled")
    return labels, is_core

def dbscan_neighbor_counts(points: torch.Tensor, eps: float, *, out=None, workspace=None,
                           stream=None):
    """eps-neighbourhood sizes (self included), int32 on the device."""
    p = _points(points)
    n, d = p.shape
    if out is None:
        out = torch.empty(n, dtype=torch.int32, device=p.device)
    if workspace is None:
        workspace = workspace_for(p)
    _check(load().dbscan_neighbor_counts(p.data_ptr(), DTYPES[p.dtype], n, d, float(eps),
                                         out.data_ptr(), workspace.data_ptr(), workspace.numel(),
                                         _stream_handle(stream)), "dbscan_neighbor_counts")
    return out


def dbscan_fit_host(points, eps: float, min_pts: int, *, labels=None, is_core=None,
                    stream=None):
    """DBSCAN on host buffers (numpy arrays or CPU tensors, ideally pinned);
    the library copies in and out and synchronises."""
    if isinstance(points, np.ndarray):
        points = torch.from_numpy(np.ascontiguousarray(points))
    p = _points(points)
    if p.is_cuda:
        raise ValueError("dbscan_fit_host takes host buffers")
    n, d = p.shape
    if labels is None:
        labels = torch.empty(n, dtype=torch.int32)
    if is_core is None:
        is_core = torch.empty(n, dtype=torch.uint8)
    _check(load().dbscan_fit_host(p.data_ptr(), DTYPES[p.dtype], n, d, float(eps), int(min_pts),
                                  labels.data_ptr(), is_core.data_ptr(),
                                  _stream_handle(stream)), "dbscan_fit_host")
    return labels, is_core


def dbscan_compact_labels(labels: torch.Tensor, *, out=None, stream=None):
    """Labels renumbered 0..k-1 (noise -1) and k; ``out`` may be ``labels``."""
    if not (labels.is_cuda and labels.dtype == torch.int32 and labels.dim() == 1
            and labels.is_contiguous()):
        raise ValueError("labels must be a contiguous 1-D int32 CUDA tensor")
    if out is None:
        out = torch.empty_like(labels)
    k = ctypes.c_int32(0)
    _check(load().dbscan_compact_labels(labels.data_ptr(), labels.numel(), out.data_ptr(),
                                        ctypes.byref(k), _stream_handle(stream)),
           "dbscan_compact_labels")
    return out, int(k.value)


def dbscan_workspace_status(workspace: torch.Tensor, stream=None) -> int:
    return int(load().dbscan_workspace_status(workspace.data_ptr(), _stream_handle(stream)))


# path codes of dbscan_workspace_info: f16 accumulates in f32; f16acc16 is the
# opt-in f16 accumulator
PATHS = {0: "fp32", 1: "tf32", 2: "bf16", 3: "f16", 4: "f16acc16"}


def dbscan_workspace_info(workspace: torch.Tensor, stream=None) -> dict:
    """Path chosen, core / candidate counts and exactness of the last call."""
    out = (ctypes.c_int64 * 6)()
    _check(load().dbscan_workspace_info(workspace.data_ptr(), _stream_handle(stream), out, 6),
           "dbscan_workspace_info")
    return {"path": PATHS.get(int(out[0]), str(out[0])), "n_core": int(out[1]),
            "n_cand": int(out[2]), "exact": bool(out[3]), "kpad": int(out[4]),
            "fused": bool(out[5])}


STAGES = ("prep", "count", "compact", "union", "flatten", "border", "finalize")


def dbscan_profile_begin() -> None:
    _check(load().dbscan_profile_begin(), "dbscan_profile_begin")


def dbscan_profile_end():
    """-> (per-stage ms dict summed over calls, calls, kernel launches)."""
    ms = (ctypes.c_float * len(STAGES))()
    calls = ctypes.c_int64()
    launches = ctypes.c_int64()
    _check(load().dbscan_profile_end(ms, len(STAGES), ctypes.byref(calls), ctypes.byref(launches)),
           "dbscan_profile_end")
    return dict(zip(STAGES, [float(v) for v in ms])), int(calls.value), int(launches.value)
