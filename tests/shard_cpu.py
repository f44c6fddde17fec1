"""CPU stand-in for the five GPU stages of the sharded pipeline (test helper).

Same contract as ``all_pairs_distance_gb300.shard.GpuStages``: rank r takes the
rows i with i % world == r of the upper triangle in the count, union and
border steps (the library splits 128-point work units the same way), and the
buffers it returns are what the collectives combine.  Brute force in numpy, for
the small sets of the gloo tests."""
import numpy as np
import torch

BIG = np.iinfo(np.int32).max


class CpuStages:
    def __init__(self, P, eps, min_pts, rank, world):
        self.P = np.asarray(P, dtype=np.int64)
        self.n = len(P)
        self.thr = int(np.float32(eps) * np.float32(eps))
        self.min_pts, self.rank, self.world = min_pts, rank, world
        d2 = ((self.P[:, None, :] - self.P[None, :, :]) ** 2).sum(-1)
        self.nb = d2 <= self.thr
        self.mine = np.arange(self.n) % world == rank

    def _find(self, x):
        while self.parent[x] != x:
            self.parent[x] = self.parent[self.parent[x]]
            x = self.parent[x]
        return x

    def _unite(self, a, b):
        a, b = self._find(a), self._find(b)
        if a != b:
            self.parent[max(a, b)] = min(a, b)

    def order(self):
        # the GPU stages share rank 0's locality order; this stand-in works in
        # input order and only checks that the broadcast arrives
        self.perm = torch.full((self.n,), -1 if self.rank else 0, dtype=torch.int32)
        if self.rank == 0:
            self.perm = torch.arange(self.n, dtype=torch.int32)
        return self.perm

    def count(self):
        assert torch.equal(self.perm, torch.arange(self.n, dtype=torch.int32)), "order not broadcast"
        cnt = np.zeros(self.n, np.int64)
        for i in np.flatnonzero(self.mine):
            js = np.flatnonzero(self.nb[i, i:]) + i
            cnt[i] += len(js)
            cnt[js[js != i]] += 1
        self.cnt = torch.from_numpy(cnt.astype(np.int32))
        return self.cnt

    def union(self):
        c = self.cnt.numpy()
        self.core = c >= self.min_pts
        self.parent = np.arange(self.n)
        for i in np.flatnonzero(self.mine & self.core):
            for j in np.flatnonzero(self.nb[i, i + 1:] & self.core[i + 1:]) + i + 1:
                self._unite(i, j)
        return torch.from_numpy(self.parent.astype(np.int32))

    def border(self, gathered):
        for r in range(gathered.shape[0]):
            for i, p in enumerate(gathered[r].numpy()):
                if self.core[i] and p != i:
                    self._unite(i, int(p))
        c = self.cnt.numpy()
        lab = np.full(self.n, -1, np.int64)
        for i in np.flatnonzero(self.core):
            lab[i] = self._find(i)
        cand = ~self.core & (c >= 2)
        lab[cand] = BIG
        for i in np.flatnonzero(self.mine & cand):
            js = np.flatnonzero(self.nb[i] & self.core)
            if len(js):
                lab[i] = min(lab[i], lab[js].min())
        self.labels = torch.from_numpy(lab.astype(np.int32))
        return self.labels

    def finish(self):
        lab = self.labels.numpy().copy()
        lab[lab == BIG] = -1
        return lab, self.core.astype(np.uint8)
