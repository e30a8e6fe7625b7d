"""Data-parallel use of the step across the ranks of a torch.distributed group.

Matrices are independent and each update needs a whole matrix (Canzona page,
section 2.1), so the matrices are split over the ranks: each rank runs the
step on the matrices it owns and the updated matrices are exchanged afterwards
(every rank broadcasts its own, in one flat buffer: a non-uniform all-gather,
section 4.1.2).  The owner of each matrix comes from

* "plan": the micro-group planner with one simulated rank per process -- the
  min-heap host-rank assignment of section 3.2.2 (rot_plan_create_ex), or
* "alpha": the α-balanced partition of section 3.2.1 over caller-given
  buckets (rot_partition_alpha), or
* "static": ownership by parameter start within each bucket (section 3.1.1).

Every rank computes the owner map itself; construction checks that all ranks
hold the same map (section 6.2's remedy for uneven buffers running out of
memory is to check the partition map's consistency) and raises on every rank
if they do not.

No optimizer arithmetic here: the local step is RotatedAdam's (the C ABI), or
whatever `make_local` builds; this module only selects, gathers and moves
tensors.
"""

from __future__ import annotations

import hashlib
from typing import Callable, List, Optional, Sequence, Tuple

import numpy as np
import torch
import torch.distributed as dist

from . import binding as B


def owner_map(shapes: Sequence[Tuple[int, int]], ranks: int, partition: str = "plan",
              c_max: int = 512 << 20, buckets: Optional[Sequence[int]] = None,
              alpha: float = 1.0) -> List[int]:
    """Owner rank of every matrix (computed on the host by the C ABI)."""
    if partition == "plan":
        return B.Plan(shapes, c_max, ranks=ranks).owners()
    sizes = list(buckets) if buckets is not None else [len(shapes)]
    if partition == "alpha":
        return B.partition_alpha(B.item_work(shapes), sizes, ranks, alpha)[0]
    if partition == "static":
        return B.partition_static([m * n for m, n in shapes], sizes, ranks)
    raise ValueError(f"unknown partition {partition!r}")


def imbalance(shapes: Sequence[Tuple[int, int]], owners: Sequence[int],
              ranks: int) -> Tuple[float, float]:
    """(work, memory) imbalance of an owner map: max over ranks / mean, with
    work = the planner's cost and memory = elements (section 5.2.1 reports the
    same two ratios)."""
    work = B.item_work(shapes)
    w = [0] * ranks
    e = [0] * ranks
    for i, o in enumerate(owners):
        w[o] += work[i]
        e[o] += shapes[i][0] * shapes[i][1]

    def ratio(v):
        mean = sum(v) / ranks
        return max(v) / mean if mean > 0 else 1.0

    return ratio(w), ratio(e)


class ShardedRotatedAdam:
    """Each rank steps the matrices it owns, then all ranks exchange them.

    shapes, c_max and the hyper-parameters are as for RotatedAdam (c_max also
    caps the planner's groups).  make_local(shapes) builds the local stepper
    (default: RotatedAdam on `device`); it must offer step(W, G, refresh).
    """

    def __init__(self, shapes: Sequence[Tuple[int, int]], c_max: int, group=None,
                 partition: str = "plan", buckets: Optional[Sequence[int]] = None,
                 alpha: float = 1.0, make_local: Optional[Callable] = None, device="cuda",
                 **hyper):
        self.group = group
        self.rank = dist.get_rank(group)
        self.world = dist.get_world_size(group)
        self.shapes = [tuple(s) for s in shapes]
        self.owners = owner_map(self.shapes, self.world, partition, c_max, buckets, alpha)
        self.check_consistency()
        self.mine = [i for i, o in enumerate(self.owners) if o == self.rank]
        self.by_rank = [[i for i, o in enumerate(self.owners) if o == r]
                        for r in range(self.world)]
        if make_local is None:
            from .optimizer import RotatedAdam

            def make_local(sh):
                return RotatedAdam(sh, c_max, device, **hyper)
        self.local = make_local([self.shapes[i] for i in self.mine]) if self.mine else None

    def _src(self, r: int) -> int:
        return r if self.group is None else dist.get_global_rank(self.group, r)

    def check_consistency(self) -> None:
        """All ranks must hold the same owner map; raises on every rank if not."""
        h = hashlib.sha256(np.asarray(self.owners, dtype=np.int64).tobytes()).digest()
        mine = torch.tensor([int.from_bytes(h[:7], "little")], dtype=torch.int64)
        if dist.get_backend(self.group) == "nccl":
            mine = mine.cuda()
        every = [torch.empty_like(mine) for _ in range(self.world)]
        dist.all_gather(every, mine, group=self.group)
        if any(int(x.item()) != int(mine.item()) for x in every):
            raise RuntimeError("owner maps differ across ranks: every rank must build the "
                               "partition from the same shapes, cap and buckets")

    def step(self, W: Sequence[torch.Tensor], G: Sequence[torch.Tensor], refresh: bool) -> None:
        """Local step on the owned matrices, then the exchange of all of them."""
        if self.local is not None:
            self.local.step([W[i] for i in self.mine], [G[i] for i in self.mine], refresh)
        self.exchange(W)

    def exchange(self, W: Sequence[torch.Tensor]) -> None:
        """Every rank broadcasts its updated matrices in one flat buffer."""
        for r, idx in enumerate(self.by_rank):
            if not idx:
                continue
            if r == self.rank:
                flat = torch.cat([W[i].reshape(-1) for i in idx])
            else:
                total = sum(W[i].numel() for i in idx)
                flat = torch.empty(total, dtype=W[idx[0]].dtype, device=W[idx[0]].device)
            dist.broadcast(flat, src=self._src(r), group=self.group)
            if r != self.rank:
                at = 0
                for i in idx:
                    k = W[i].numel()
                    W[i].copy_(flat[at:at + k].view_as(W[i]))
                    at += k
