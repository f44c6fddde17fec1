"""Seeded synthetic point sets for the DBSCAN workloads.

This module only draws random numbers: it holds none of the clustering
arithmetic, and both the CUDA path's tests/benchmark and the CPU oracle's
tests take their inputs from here.

Workloads (the pages' own data set is unnamed -- "Design and optimization of
DBSCAN Algorithm based on CUDA", §I and Table I describe only "a test set with
23040 points" in 3-D -- so these synthetic sets stand in for it):

* ``blobs_2k_d2``    N=2,000   d=2   [0,2047]  8 blobs sigma=40 + 10% noise, eps=30,  minPts=5
* ``blobs_100k_d2``  N=100,000 d=2   [0,2047]  50 blobs sigma=25 (Dirichlet(1) sizes) + 10% noise, eps=20, minPts=10
* ``blobs_200k_d16`` N=200,000 d=16  [0,511]   100 blobs sigma=20 + 15% noise, eps=120, minPts=20
* ``blobs_1m_d3``    N=1,000,000 d=3 [0,2047]  500 blobs sigma=12 + 3 filaments + 20% noise, eps=10, minPts=8
* ``blobs_500k_d64`` N=500,000 d=64  [0,255]   200 blobs sigma=8 + 10% noise, eps=100, minPts=16 (bf16)

Recipe shared by all of them: ``numpy.random.default_rng(seed)``; blob centres
uniform in the box; blob points ``rint`` (half-to-even) of a normal draw,
clipped to the box; noise uniform integers in ``[0, hi]``; the concatenation is
shuffled with one permutation from the same generator, so clusters are not
contiguous in index space.  Every coordinate is an integer stored as float32.
"""
from __future__ import annotations

from dataclasses import dataclass

import numpy as np


@dataclass(frozen=True)
class Workload:
    name: str
    n: int
    d: int
    hi: int
    eps: float
    min_pts: int
    dtype: str  # "f32" or "bf16": the type the points are handed to the library in
    seed: int


WORKLOADS = {
    "blobs_2k_d2": Workload("blobs_2k_d2", 2_000, 2, 2047, 30.0, 5, "f32", 1),
    "blobs_100k_d2": Workload("blobs_100k_d2", 100_000, 2, 2047, 20.0, 10, "f32", 2),
    "blobs_200k_d16": Workload("blobs_200k_d16", 200_000, 16, 511, 120.0, 20, "f32", 3),
    "blobs_1m_d3": Workload("blobs_1m_d3", 1_000_000, 3, 2047, 10.0, 8, "f32", 4),
    "blobs_500k_d64": Workload("blobs_500k_d64", 500_000, 64, 255, 100.0, 16, "bf16", 5),
}


def _split_even(total: int, parts: int) -> np.ndarray:
    """Equal sizes, remainder to the first parts."""
    sizes = np.full(parts, total // parts, dtype=np.int64)
    sizes[: total % parts] += 1
    return sizes


def _blob_points(rng, centres, sizes, sigma, hi):
    chunks = []
    d = centres.shape[1]
    for c, m in zip(centres, sizes):
        if m == 0:
            continue
        p = rng.normal(loc=c, scale=sigma, size=(int(m), d))
        chunks.append(np.clip(np.rint(p), 0, hi))
    if not chunks:
        return np.zeros((0, centres.shape[1]))
    return np.concatenate(chunks, axis=0)


def _noise(rng, m, d, hi):
    return rng.integers(0, hi, size=(m, d), endpoint=True).astype(np.float64)


def _filament(rng, a, b, m, hi):
    """Points uniform along segment a->b plus N(0,1) jitter perpendicular to it."""
    t = rng.uniform(0.0, 1.0, size=(m, 1))
    base = a[None, :] + t * (b - a)[None, :]
    u = (b - a) / max(np.linalg.norm(b - a), 1e-12)
    jit = rng.normal(0.0, 1.0, size=(m, a.shape[0]))
    jit -= (jit @ u)[:, None] * u[None, :]
    return np.clip(np.rint(base + jit), 0, hi)


def blob_set(n, d, hi, n_blobs, sigma, noise, seed, *, sizes="even",
             filaments=0, filament_pts=0):
    """General recipe: ``n`` points = blobs + ``noise`` uniform points (+ filaments).

    ``sizes`` is "even" (equal, remainder first) or "dirichlet" (multinomial
    over Dirichlet(1) weights).  Filaments join random pairs of distinct blob
    centres.  Returns float32 ``[n, d]`` with integer values in ``[0, hi]``.
    """
    rng = np.random.default_rng(seed)
    n_blob_pts = n - noise - filaments * filament_pts
    if n_blob_pts < 0:
        raise ValueError("noise + filament points exceed n")
    centres = rng.uniform(0.0, hi, size=(max(n_blobs, 1), d))
    if n_blobs == 0:
        blob_sizes = np.zeros(1, dtype=np.int64)
    elif sizes == "even":
        blob_sizes = _split_even(n_blob_pts, n_blobs)
    elif sizes == "dirichlet":
        w = rng.dirichlet(np.ones(n_blobs))
        blob_sizes = rng.multinomial(n_blob_pts, w)
    else:
        raise ValueError(sizes)
    parts = [_blob_points(rng, centres, blob_sizes, sigma, hi)]
    for _ in range(filaments):
        a, b = rng.choice(n_blobs, size=2, replace=False)
        parts.append(_filament(rng, centres[a], centres[b], filament_pts, hi))
    parts.append(_noise(rng, noise, d, hi))
    pts = np.concatenate(parts, axis=0)
    assert pts.shape == (n, d), pts.shape
    perm = rng.permutation(n)
    return np.ascontiguousarray(pts[perm]).astype(np.float32)


def generate(name: str) -> np.ndarray:
    """The named workload's points, float32 ``[N, d]`` (integer-valued)."""
    w = WORKLOADS[name]
    if name == "blobs_2k_d2":
        return blob_set(w.n, w.d, w.hi, 8, 40.0, 200, w.seed)
    if name == "blobs_100k_d2":
        return blob_set(w.n, w.d, w.hi, 50, 25.0, 10_000, w.seed, sizes="dirichlet")
    if name == "blobs_200k_d16":
        return blob_set(w.n, w.d, w.hi, 100, 20.0, 30_000, w.seed)
    if name == "blobs_1m_d3":
        return blob_set(w.n, w.d, w.hi, 500, 12.0, 200_000, w.seed,
                        filaments=3, filament_pts=5_000)
    if name == "blobs_500k_d64":
        return blob_set(w.n, w.d, w.hi, 200, 8.0, 50_000, w.seed)
    raise KeyError(name)


def scaled(name: str, n: int, seed: int | None = None) -> np.ndarray:
    """A smaller set with the named workload's range, spread and noise share.

    The blob count is scaled with ``n`` (at least 2 blobs) so that blob
    densities -- and hence the mix of core, border and noise points -- stay
    close to the full workload's.  Used for element-by-element parity at sizes
    the oracle finishes in seconds.
    """
    w = WORKLOADS[name]
    s = w.seed * 1000 + 7 if seed is None else seed
    frac = n / w.n
    if name == "blobs_2k_d2":
        return blob_set(n, w.d, w.hi, max(2, round(8 * frac)), 40.0, n // 10, s)
    if name == "blobs_100k_d2":
        return blob_set(n, w.d, w.hi, max(2, round(50 * frac)), 25.0, n // 10, s,
                        sizes="dirichlet")
    if name == "blobs_200k_d16":
        return blob_set(n, w.d, w.hi, max(2, round(100 * frac)), 20.0, (n * 3) // 20, s)
    if name == "blobs_1m_d3":
        nb = max(2, round(500 * frac))
        fp = max(1, round(5_000 * frac))
        return blob_set(n, w.d, w.hi, nb, 12.0, n // 5, s, filaments=3, filament_pts=fp)
    if name == "blobs_500k_d64":
        return blob_set(n, w.d, w.hi, max(2, round(200 * frac)), 8.0, n // 10, s)
    raise KeyError(name)


def uniform_ints(n: int, d: int, hi: int, seed: int) -> np.ndarray:
    """Uniform integer points in ``[0, hi]^d`` as float32."""
    rng = np.random.default_rng(seed)
    return rng.integers(0, hi, size=(n, d), endpoint=True).astype(np.float32)
