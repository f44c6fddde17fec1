"""Graph replay of repeated calls (a caller's stream and workspace): the
replayed call must give the oracle's result for whatever the buffers hold."""
import numpy as np
import pytest
import torch

import oracle
from all_pairs_distance_gb300 import binding, synth
from gpu_util import assert_same

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("case", ["d3", "d64_bf16", "d2_culled"])
def test_replay_follows_the_buffers(case):
    if case == "d3":
        sets = [synth.scaled("blobs_1m_d3", 9_001, seed=s) for s in (71, 72)]
        eps, mp, dt = 10.0, 8, torch.float32
    elif case == "d64_bf16":
        sets = [synth.scaled("blobs_500k_d64", 2_501, seed=s) for s in (73, 74)]
        eps, mp, dt = 100.0, 16, torch.bfloat16
    else:
        sets = [synth.scaled("blobs_100k_d2", 6_001, seed=s) for s in (75, 76)]
        eps, mp, dt = 20.0, 10, torch.float32
    fit = binding.dbscan_fit_culled if case.endswith("culled") else binding.dbscan_fit_ex
    stream = torch.cuda.Stream()
    x = torch.from_numpy(sets[0]).to("cuda").to(dt)
    ws = binding.workspace_for(x)
    labels = torch.empty(len(sets[0]), dtype=torch.int32, device="cuda")
    core = torch.empty(len(sets[0]), dtype=torch.uint8, device="cuda")
    with torch.cuda.stream(stream), binding.options(graphs=1):
        # the same arguments four times (captured once, then replayed), the
        # input overwritten in place between calls
        for call in range(4):
            P = sets[call % 2]
            x.copy_(torch.from_numpy(P).to("cuda").to(dt))
            fit(x, eps, mp, labels=labels, is_core=core, workspace=ws, stream=stream)
            st = binding.dbscan_workspace_status(ws, stream)
            assert st == 0, binding.dbscan_strerror(st)
            stream.synchronize()
            _, core_ref, label_ref = oracle.dbscan(P, eps, mp)
            assert_same(core.cpu().numpy(), core_ref, f"{case} call {call} core flags")
            assert_same(labels.cpu().numpy(), label_ref, f"{case} call {call} labels")


def test_replay_and_direct_launches_agree():
    P = synth.scaled("blobs_1m_d3", 7_001, seed=77)
    x = torch.from_numpy(P).to("cuda")
    ws = binding.workspace_for(x)
    stream = torch.cuda.Stream()
    out = {}
    for mode in ("1", "0"):
        with torch.cuda.stream(stream), binding.options(graphs=int(mode)):
            for _ in range(2):
                lab, core = binding.dbscan_fit_ex(x, 10.0, 8, workspace=ws, stream=stream)
                cnt = binding.dbscan_neighbor_counts(x, 10.0, workspace=ws, stream=stream)
            stream.synchronize()
        out[mode] = (lab.cpu().numpy(), core.cpu().numpy(), cnt.cpu().numpy())
    for a, b, w in zip(out["1"], out["0"], ("labels", "core", "counts")):
        assert_same(a, b, f"graph vs direct {w}")


def test_graph_cache_evicts_beyond_its_capacity():
    # more distinct argument sets than the cache holds (16): the least recently
    # used graphs are destroyed to make room and every call stays correct
    P = synth.scaled("blobs_100k_d2", 3_001, seed=78)
    _, core_ref, label_ref = oracle.dbscan(P, 20.0, 10)
    x = torch.from_numpy(P).to("cuda")
    ws = binding.workspace_for(x)
    stream = torch.cuda.Stream()
    outs = [(torch.empty(len(P), dtype=torch.int32, device="cuda"),
             torch.empty(len(P), dtype=torch.uint8, device="cuda")) for _ in range(20)]
    with torch.cuda.stream(stream), binding.options(graphs=1):
        for sweep in range(2):
            for lab, core in outs:   # 20 keys (output pointers differ)
                lab.fill_(-7)
                binding.dbscan_fit_ex(x, 20.0, 10, labels=lab, is_core=core, workspace=ws,
                                      stream=stream)
            stream.synchronize()
            for lab, core in outs:
                assert_same(lab.cpu().numpy(), label_ref, f"sweep {sweep} labels")
                assert_same(core.cpu().numpy(), core_ref, f"sweep {sweep} core flags")
