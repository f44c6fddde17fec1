"""The sharded pipeline's GPU stages (dbscan_fit_shard) on one GPU.

* world = 2 and 3: the ranks' stages run one after another in this process,
  each with its own workspace, and torch sums, stacks and minimises their
  buffers where the collectives would (no kernel waits on another rank's).
  This checks the split of the work units and the merge of the forests.
* world = 1: the real choreography over a one-rank NCCL process group.
Results must equal the oracle's, element by element."""
import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist

import oracle
from all_pairs_distance_gb300 import binding, synth
from all_pairs_distance_gb300.shard import GpuStages, dbscan_fit_sharded
from gpu_util import assert_same

pytestmark = pytest.mark.gpu

CASES = {
    "c4_like_20k_d3": (lambda: synth.scaled("blobs_1m_d3", 20_011, seed=111), 10.0, 8, torch.float32),
    "c2_like_12k_d2": (lambda: synth.scaled("blobs_100k_d2", 12_003, seed=112), 20.0, 10, torch.float32),
    "c3_like_6k_d16": (lambda: synth.scaled("blobs_200k_d16", 6_007, seed=113), 120.0, 20, torch.float32),
    "c5_like_4k_d64": (lambda: synth.scaled("blobs_500k_d64", 4_003, seed=114), 100.0, 16, torch.bfloat16),
}


def emulate(P, eps, min_pts, dtype, world):
    x = torch.from_numpy(P).cuda().to(dtype)
    ranks = [GpuStages(x, eps, min_pts, r, world) for r in range(world)]
    orders = [s.order() for s in ranks]
    for o in orders[1:]:
        o.copy_(orders[0])
    cnts = [s.count() for s in ranks]
    total = torch.stack(cnts).sum(0, dtype=torch.int32)
    for c in cnts:
        c.copy_(total)
    gathered = torch.stack([s.union() for s in ranks]).contiguous()
    labels = [s.border(gathered) for s in ranks]
    low = torch.stack(labels).amin(0)
    for lab in labels:
        lab.copy_(low)
    out = [s.finish() for s in ranks]
    for s in ranks:
        assert binding.dbscan_workspace_status(s.ws) == 0
    torch.cuda.synchronize()
    return [(lab.cpu().numpy(), core.cpu().numpy()) for lab, core in out]


@pytest.mark.parametrize("world", [2, 3])
@pytest.mark.parametrize("name", sorted(CASES))
def test_emulated_ranks_match_oracle(name, world):
    make, eps, min_pts, dtype = CASES[name]
    P = make()
    _, core_ref, label_ref = oracle.dbscan(P, eps, min_pts)
    for r, (lab, core) in enumerate(emulate(P, eps, min_pts, dtype, world)):
        assert_same(core, core_ref, f"{name} world {world} rank {r} core flags")
        assert_same(lab, label_ref, f"{name} world {world} rank {r} labels")


def test_emulated_ranks_on_cuda_cores():
    P = synth.scaled("blobs_100k_d2", 9_001, seed=115)
    _, core_ref, label_ref = oracle.dbscan(P, 20.0, 10)
    with binding.options(paths=["fp32"]):
        out = emulate(P, 20.0, 10, torch.float32, 2)
    for lab, core in out:
        assert_same(core, core_ref, "fp32 core flags")
        assert_same(lab, label_ref, "fp32 labels")


def test_one_rank_nccl_group():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    dist.init_process_group("nccl", init_method=f"tcp://127.0.0.1:{port}", rank=0, world_size=1)
    try:
        P = synth.scaled("blobs_1m_d3", 15_007, seed=116)
        _, core_ref, label_ref = oracle.dbscan(P, 10.0, 8)
        lab, core = dbscan_fit_sharded(torch.from_numpy(P).cuda(), 10.0, 8)
        torch.cuda.synchronize()
        assert_same(core.cpu().numpy(), core_ref, "core flags")
        assert_same(lab.cpu().numpy(), label_ref, "labels")
    finally:
        dist.destroy_process_group()


def test_shard_argument_errors():
    x = torch.zeros((100, 3), device="cuda")
    ws = binding.workspace_for(x)
    lib = binding.load()
    for stage, rank, world in ((5, 0, 1), (0, 1, 1), (0, -1, 2), (0, 0, 0)):
        st = lib.dbscan_fit_shard(stage, x.data_ptr(), 0, 100, 3, 1.0, 2, rank, world, None, None,
                                  None, ws.data_ptr(), ws.numel(), None)
        assert st == binding.Status.INVALID_ARG
    # no workspace: the stages keep their state in it
    assert lib.dbscan_fit_shard(0, x.data_ptr(), 0, 100, 3, 1.0, 2, 0, 1, None, None, None,
                                None, 0, None) == binding.Status.INVALID_ARG
