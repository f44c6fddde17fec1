"""The sharded pipeline's collectives (all_pairs_distance_gb300.shard) over
two and three gloo ranks on CPU: each rank runs the choreography with a CPU
stand-in for the GPU stages (tests/shard_cpu.py) and must end with the
oracle's core flags and labels."""
import json
import os
import socket
import subprocess
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

RANK_SCRIPT = r'''
import json, os, sys
sys.path.insert(0, {root!r}); sys.path.insert(0, {tests!r})
import numpy as np
import torch.distributed as dist
import oracle
from all_pairs_distance_gb300 import synth
from all_pairs_distance_gb300.shard import run_sharded
from shard_cpu import CpuStages
dist.init_process_group("gloo")
rank, world = dist.get_rank(), dist.get_world_size()
out = {{}}
for name, P, eps, mp in (
        ("c1", synth.scaled("blobs_2k_d2", 700, seed=3), 30.0, 5),
        ("c4", synth.scaled("blobs_1m_d3", 900, seed=4), 10.0, 8),
        ("bridge", np.array([[0, 0], [1, 0], [2, 0], [3, 0], [10, 0], [11, 0], [12, 0],
                             [4, 0], [5, 0], [6, 0], [7, 0], [8, 0], [9, 0]], np.float32), 1.0, 3)):
    lab, core = run_sharded(CpuStages(P, eps, mp, rank, world))
    _, core_ref, lab_ref = oracle.dbscan(P, eps, mp)
    out[name] = bool(np.array_equal(lab, lab_ref) and np.array_equal(core, core_ref))
with open(os.path.join({outdir!r}, f"rank{{rank}}.json"), "w") as f:
    json.dump(out, f)
dist.destroy_process_group()
'''


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


@pytest.mark.parametrize("world", [2, 3])
def test_sharded_choreography_over_gloo(tmp_path, world):
    script = tmp_path / "rank.py"
    script.write_text(RANK_SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests"),
                                         outdir=str(tmp_path)))
    env = dict(os.environ, PYTHONPATH=ROOT)
    env.pop("CUDA_VISIBLE_DEVICES", None)
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node",
           str(world), "--master-addr", "127.0.0.1", "--master-port", str(_free_port()), str(script)]
    r = subprocess.run(cmd, cwd=ROOT, env=env, capture_output=True, text=True, timeout=300)
    assert r.returncode == 0, r.stderr[-3000:]
    for rank in range(world):
        res = json.loads((tmp_path / f"rank{rank}.json").read_text())
        assert res and all(res.values()), (rank, res)
