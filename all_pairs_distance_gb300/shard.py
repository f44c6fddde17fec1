"""DBSCAN sharded across the ranks of a torch.distributed process group, one
GPU per rank.

Every rank passes the same points.  The library splits the work units of the
count, union and border sweeps between the ranks (dbscan.h, dbscan_fit_shard)
and this module runs the four collectives between its five stages:

    stage 0  statistics + locality order       -> broadcast of rank 0's order
    stage 1  staging + this rank's count        -> all-reduce SUM of the counts
    stage 2  core flags + this rank's union     -> all-gather of the union-find forests
    stage 3  merge + this rank's border labels  -> all-reduce MIN of the labels
    stage 4  finalize

With NCCL the collectives run on the current CUDA stream's order, so the
stages and the collectives form one stream-ordered pipeline.  The choreography
(``run_sharded``) takes any object with the five stage methods, which is how
the CPU tests run it over gloo without a GPU.
"""
from __future__ import annotations

import torch
import torch.distributed as dist

from . import binding


class GpuStages:
    """The five stages on this rank's GPU, through the C ABI."""

    def __init__(self, points: torch.Tensor, eps: float, min_pts: int, rank: int, world: int,
                 workspace: torch.Tensor | None = None):
        self.p = points.contiguous()
        self.n, self.d = self.p.shape
        self.eps, self.min_pts, self.rank, self.world = eps, min_pts, rank, world
        self.ws = binding.workspace_for(self.p) if workspace is None else workspace
        dev = self.p.device
        self.labels = torch.empty(self.n, dtype=torch.int32, device=dev)
        self.is_core = torch.empty(self.n, dtype=torch.uint8, device=dev)

    def _stage(self, k, **kw):
        binding.dbscan_fit_shard(k, self.p, self.eps, self.min_pts, self.rank, self.world,
                                 workspace=self.ws, **kw)

    def order(self) -> torch.Tensor:
        self._stage(0)
        return binding.dbscan_shard_buffer(self.ws, self.n, self.d, binding.SHARD_ORDER)

    def count(self) -> torch.Tensor:
        self._stage(1)
        return binding.dbscan_shard_buffer(self.ws, self.n, self.d, binding.SHARD_COUNTS)

    def union(self) -> torch.Tensor:
        self._stage(2, labels=self.labels, is_core=self.is_core)
        return binding.dbscan_shard_buffer(self.ws, self.n, self.d, binding.SHARD_PARENTS)

    def border(self, gathered: torch.Tensor) -> torch.Tensor:
        self._stage(3, labels=self.labels, gathered=gathered)
        return self.labels

    def finish(self):
        self._stage(4, labels=self.labels)
        return self.labels, self.is_core


def run_sharded(stages, group=None):
    """The five stages with the collectives between them -> stages.finish()."""
    world = dist.get_world_size(group)
    order = stages.order()
    dist.broadcast(order, src=dist.get_global_rank(group, 0) if group is not None else 0, group=group)
    cnt = stages.count()
    dist.all_reduce(cnt, op=dist.ReduceOp.SUM, group=group)
    parents = stages.union()
    gathered = torch.empty((world, parents.numel()), dtype=parents.dtype, device=parents.device)
    dist.all_gather(list(gathered.unbind(0)), parents, group=group)
    labels = stages.border(gathered)
    dist.all_reduce(labels, op=dist.ReduceOp.MIN, group=group)
    return stages.finish()


def dbscan_fit_sharded(points: torch.Tensor, eps: float, min_pts: int, group=None, *,
                       workspace: torch.Tensor | None = None):
    """DBSCAN over all ranks of ``group`` (every rank passes the same device
    points) -> (labels int32, is_core uint8), identical on every rank."""
    stages = GpuStages(points, eps, min_pts, dist.get_rank(group), dist.get_world_size(group),
                       workspace)
    return run_sharded(stages, group)
