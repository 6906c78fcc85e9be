"""Multi-rank host logic of bench.py on CPU (gloo, world size 2): every rank
gets its own seeded inputs of the same shape (weak scaling), timing is the
maximum over ranks, and the job value counts all ranks' work over that time.
No GPU and no collective on the data path are involved."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        import workloads
        w = workloads.WORKLOADS["tiny"]
        x = workloads.make_inputs(w.B, w.H, w.N, w.d, seed=bench.rank_seed(w, rank))
        ms = 1.0 + rank  # rank 1 is the slower one
        worst = bench._max_over_ranks(ms, world)
        bench._barrier(world)
        out[rank] = (worst, bench.job_tflops(world, 1e12, worst), float(x["q"].float().sum()))
    finally:
        dist.destroy_process_group()


def test_two_ranks_weak_scaling_host_logic():
    world, port = 2, _free_port()
    with mp.Manager() as m:
        out = m.dict()
        mp.spawn(_worker, args=(world, port, out), nprocs=world, join=True)
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.0              # max over ranks
    assert res[0][1] == pytest.approx(2 * 1e12 / 2e-3 / 1e12)  # all ranks' flops over the slowest time
    assert res[0][2] != res[1][2]                      # each rank has its own inputs
