"""CPU DBSCAN oracle -- test infrastructure only.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg may import this package.  The CUDA library never calls it and has no CPU
fallback of any kind.

The C source (``dbscan_oracle.c``) is a plain single-threaded DBSCAN written
from the definitions of "Design and optimization of DBSCAN Algorithm based on
CUDA", §II; its header lists the readings taken where the page is silent.
This module compiles it with gcc into ``oracle/_build/`` and wraps it with
ctypes.  Inputs are converted to float64 here (exact for float32/bf16 data).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dbscan_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_LIB = os.path.join(_BUILD, "liboracle.so")
_LIB_OMP = os.path.join(_BUILD, "liboracle_omp.so")
_lock = threading.Lock()
_lib = None
_lib_omp = None


def build(force: bool = False) -> str:
    """Compile the oracle shared library (gcc, -O2, no -march flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared",
                               "-o", tmp, _SRC])
        os.replace(tmp, _LIB)
    return _LIB


def build_parallel(force: bool = False):
    """The same source built with OpenMP (its count loop on all host cores),
    or None when the compiler cannot build it.  A separately timed baseline
    only: the tests and the single-threaded baseline use ``build()``."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_OMP) or os.path.getmtime(_LIB_OMP) < os.path.getmtime(_SRC):
        tmp = _LIB_OMP + f".tmp{os.getpid()}"
        try:
            subprocess.check_call(["gcc", "-O2", "-std=c99", "-fPIC", "-shared", "-fopenmp",
                                   "-o", tmp, _SRC], stderr=subprocess.DEVNULL)
        except (subprocess.CalledProcessError, OSError):
            return None
        os.replace(tmp, _LIB_OMP)
    return _LIB_OMP


def _declare(lib):
    P = ctypes.c_void_p
    i64, i32, f32 = ctypes.c_int64, ctypes.c_int32, ctypes.c_float
    lib.oracle_counts.argtypes = [P, i64, i32, f32, P]
    lib.oracle_counts.restype = None
    lib.oracle_row_counts.argtypes = [P, i64, i32, f32, P, i64, P]
    lib.oracle_row_counts.restype = None
    lib.oracle_row_neighbours.argtypes = [P, i64, i32, f32, i64, P, i64]
    lib.oracle_row_neighbours.restype = i64
    lib.oracle_dbscan.argtypes = [P, i64, i32, f32, i32, P, P, P]
    lib.oracle_dbscan.restype = ctypes.c_int
    lib.oracle_threads.argtypes = []
    lib.oracle_threads.restype = ctypes.c_int
    return lib


def _load_parallel():
    global _lib_omp
    with _lock:
        if _lib_omp is None:
            path = build_parallel()
            if path is None:
                return None
            _lib_omp = _declare(ctypes.CDLL(path))
    return _lib_omp


def parallel_threads() -> int:
    """Threads of the OpenMP build's count loop (0 when it cannot be built)."""
    lib = _load_parallel()
    return int(lib.oracle_threads()) if lib is not None else 0


def dbscan_parallel(points, eps: float, min_pts: int):
    """``dbscan`` through the OpenMP build (same source; identical results)."""
    lib = _load_parallel()
    if lib is None:
        raise RuntimeError("the OpenMP build of the oracle is not available")
    p = _as_f64(points)
    n, d = p.shape
    cnt = np.zeros(n, np.int32)
    core = np.zeros(n, np.uint8)
    label = np.zeros(n, np.int32)
    rc = lib.oracle_dbscan(_ptr(p), n, d, float(eps), int(min_pts), _ptr(cnt), _ptr(core),
                           _ptr(label))
    if rc != 0:
        raise MemoryError("oracle_dbscan could not allocate its queue")
    return cnt, core, label


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def _as_f64(points) -> np.ndarray:
    p = np.asarray(points)
    if p.ndim != 2:
        raise ValueError("points must be [n, d]")
    return np.ascontiguousarray(p, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def dbscan(points, eps: float, min_pts: int):
    """Full DBSCAN: returns ``(cnt int32[n], core uint8[n], label int32[n])``."""
    p = _as_f64(points)
    n, d = p.shape
    cnt = np.zeros(n, np.int32)
    core = np.zeros(n, np.uint8)
    label = np.zeros(n, np.int32)
    rc = _load().oracle_dbscan(_ptr(p), n, d, float(eps), int(min_pts),
                               _ptr(cnt), _ptr(core), _ptr(label))
    if rc != 0:
        raise MemoryError("oracle_dbscan could not allocate its queue")
    return cnt, core, label


def counts(points, eps: float) -> np.ndarray:
    """eps-neighbourhood sizes (self included) of every point."""
    p = _as_f64(points)
    n, d = p.shape
    cnt = np.zeros(n, np.int32)
    _load().oracle_counts(_ptr(p), n, d, float(eps), _ptr(cnt))
    return cnt


def row_counts(points, eps: float, rows) -> np.ndarray:
    """eps-neighbourhood sizes of the listed rows only."""
    p = _as_f64(points)
    n, d = p.shape
    r = np.ascontiguousarray(rows, dtype=np.int64)
    out = np.zeros(r.shape[0], np.int32)
    _load().oracle_row_counts(_ptr(p), n, d, float(eps), _ptr(r), r.shape[0], _ptr(out))
    return out


def row_neighbours(points, eps: float, i: int) -> np.ndarray:
    """Ascending indices of the eps-neighbours of point ``i`` (itself included)."""
    p = _as_f64(points)
    n, d = p.shape
    cap = 1024
    while True:
        out = np.zeros(cap, np.int64)
        c = _load().oracle_row_neighbours(_ptr(p), n, d, float(eps), int(i), _ptr(out), cap)
        if c <= cap:
            return out[:c]
        cap = int(c)


def compact_labels(labels):
    """Cluster labels renumbered 0..k-1 (noise stays -1) and k.

    The optional compacted output named among the scope's next steps: the
    distinct non-negative labels, taken in increasing order, become 0, 1, ...
    (DBSCAN labels are smallest core indices, so clusters keep the order of
    their first core point).  A plain definition: no page fixes it.
    """
    lab = np.asarray(labels, dtype=np.int64)
    keys = np.unique(lab[lab >= 0])
    out = np.full(lab.shape, -1, dtype=np.int32)
    pos = lab >= 0
    out[pos] = np.searchsorted(keys, lab[pos]).astype(np.int32)
    return out, int(keys.size)
