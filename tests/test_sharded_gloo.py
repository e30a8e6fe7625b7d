"""The data-parallel path on two CPU ranks (gloo): owner maps agree across
ranks, each rank steps only what it owns, and after the exchange every rank
holds the same matrices as a single-process run.  The local step here is the
oracle (this is a test of the host logic around the step; the GPU step itself
is tested against the oracle elsewhere)."""

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

from matrix_optimizer_step_rot_gb300 import build, inputs
from matrix_optimizer_step_rot_gb300 import sharded as S
from oracle import rot_oracle as orc

WORLD = 2


class OracleLocal:
    """Local stepper over float64 torch tensors, driven by the oracle."""

    def __init__(self, shapes, hyper, log):
        self.states = [orc.init_state(m, n) for m, n in shapes]
        self.h = hyper
        self.log = log
        self.shapes = shapes

    def step(self, W, G, refresh):
        h = self.h
        self.log.append(len(W))
        for w, g, st in zip(W, G, self.states):
            new = orc.step(w.numpy(), g.numpy(), st, h.beta1, h.beta2, h.eps, h.lr, refresh,
                           h.rank_rtol)
            w.copy_(torch.from_numpy(new))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, port, out_dir, mode):
    build.build()
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=WORLD)
    try:
        wl = inputs.workload("tiny")
        if mode == "mismatch":
            c_max = wl.c_max if rank == 0 else 1      # rank 1 plans with another cap
            try:
                S.ShardedRotatedAdam(wl.shapes, c_max, make_local=lambda sh: None)
            except RuntimeError as e:
                np.save(os.path.join(out_dir, f"err{rank}.npy"), np.array([str(e)]))
            return
        log = []
        opt = S.ShardedRotatedAdam(wl.shapes, wl.c_max, partition=mode, buckets=[2, 2],
                                   make_local=lambda sh: OracleLocal(sh, wl.hyper, log))
        W = [torch.from_numpy(wl.w0(i).astype(np.float64)) for i in range(wl.count)]
        for t in range(1, wl.steps + 1):
            G = [torch.from_numpy(wl.grad(i, t).astype(np.float64)) for i in range(wl.count)]
            opt.step(W, G, wl.refresh(t))
        np.savez(os.path.join(out_dir, f"rank{rank}.npz"), *[w.numpy() for w in W],
                 owners=np.array(opt.owners), stepped=np.array(log))
    finally:
        dist.destroy_process_group()


def _spawn(tmp_path, mode):
    build.build()
    mp.start_processes(_worker, args=(_free_port(), str(tmp_path), mode), nprocs=WORLD,
                       join=True, start_method="spawn")


@pytest.mark.parametrize("mode", ["plan", "alpha", "static"])
def test_two_ranks_match_single_process(tmp_path, mode):
    _spawn(tmp_path, mode)
    wl = inputs.workload("tiny")
    ref = orc.run(wl)
    res = [np.load(tmp_path / f"rank{r}.npz") for r in range(WORLD)]
    owners = list(res[0]["owners"])
    assert owners == list(res[1]["owners"])
    assert sorted(set(owners)) == [0, 1]               # both ranks own work on this map
    for r in range(WORLD):
        # each rank stepped exactly its own matrices, every step
        assert list(res[r]["stepped"]) == [owners.count(r)] * wl.steps
        for i in range(wl.count):
            np.testing.assert_array_equal(res[r][f"arr_{i}"], ref[i][0])


def test_diverging_owner_maps_raise_on_every_rank(tmp_path):
    _spawn(tmp_path, "mismatch")
    for r in range(WORLD):
        msg = str(np.load(tmp_path / f"err{r}.npy")[0])
        assert "owner maps differ" in msg


def test_owner_maps_and_imbalance_on_the_stack():
    """Owner maps of the three partitions on the 28-block stack at 8 ranks,
    one bucket per block: under the planner and the α-balanced map every rank
    owns work (static ownership by start leaves the same ranks idle in every
    7-matrix bucket), and the α-balanced map's work imbalance is below static
ownership's (the page's section 5.2.1 claim, in kind).  The planner's global
LPT, free of bucket contiguity, is the most even of the three here."""
    build.build()
    wl = inputs.workload("full")
    ratios = {}
    for mode in ("plan", "alpha", "static"):
        own = S.owner_map(wl.shapes, 8, mode, wl.c_max, [7] * 28, 1.0)
        if mode != "static":
            assert sorted(set(own)) == list(range(8))
        ratios[mode] = S.imbalance(wl.shapes, own, 8)
    print(ratios)
    assert ratios["alpha"][0] < ratios["static"][0]
    assert ratios["plan"][0] <= ratios["alpha"][0]
