"""Writes the expected results of the full-size workloads, computed by the
oracle alone, as digests: tests/golden/fullsize_<workload>.json.

For each workload the seeded input comes from the synthetic generator
(``all_pairs_distance_gb300.synth``, random numbers only) and the expected
neighbour counts, core flags and labels from the oracle's OpenMP build
(``oracle.dbscan_parallel``: the same source as ``oracle.dbscan``, with its
count loop and the scan of each expansion step spread over the host cores;
identical results, tested in tests/test_oracle.py).  The file stores the
SHA-256 of the input and of each output array, plus a few totals, so that a
GPU test can compare all N values of a result without shipping them:

    python tests/golden/make_fullsize.py [workload ...]

Run times on 8 x86 cores: blobs_200k_d16 a few minutes, blobs_1m_d3 about
half an hour, blobs_500k_d64 about an hour.
"""
from __future__ import annotations

import hashlib
import json
import os
import sys
import time

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(os.path.dirname(HERE))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

DEFAULT = ("blobs_200k_d16", "blobs_1m_d3", "blobs_500k_d64")


def digest(a: np.ndarray, dtype: str) -> str:
    """SHA-256 of the array's values as contiguous little-endian ``dtype``."""
    return hashlib.sha256(np.ascontiguousarray(a, dtype=dtype).tobytes()).hexdigest()


def input_digest(P: np.ndarray) -> str:
    return digest(P, "<f4")


def path_for(name: str) -> str:
    return os.path.join(HERE, f"fullsize_{name}.json")


def make(name: str) -> dict:
    import oracle
    from all_pairs_distance_gb300 import synth

    w = synth.WORKLOADS[name]
    P = synth.generate(name)
    t = time.time()
    cnt, core, label = oracle.dbscan_parallel(P, w.eps, w.min_pts)
    dt = time.time() - t
    rec = {
        "workload": name, "n": int(P.shape[0]), "d": int(P.shape[1]),
        "eps": w.eps, "min_pts": w.min_pts,
        "input_sha256": input_digest(P),
        "cnt_sha256": digest(cnt, "<i4"),
        "core_sha256": digest(core, "<u1"),
        "label_sha256": digest(label, "<i4"),
        "n_core": int(core.sum()),
        "n_noise": int((label == -1).sum()),
        "n_clusters": int(np.unique(label[label >= 0]).size),
        "cnt_sum": int(cnt.astype(np.int64).sum()),
        "producer": "oracle.dbscan_parallel (OpenMP build of oracle/dbscan_oracle.c)",
        "oracle_threads": oracle.parallel_threads(),
        "oracle_seconds": round(dt, 1),
    }
    with open(path_for(name), "w") as f:
        json.dump(rec, f, indent=1)
        f.write("\n")
    return rec


if __name__ == "__main__":
    for nm in (sys.argv[1:] or DEFAULT):
        print(json.dumps(make(nm)), flush=True)
