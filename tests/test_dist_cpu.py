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


# --------------------------------------------------------------------------- local replica spawn
_ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

_CHILD = """
import json, os, sys
sys.path.insert(0, {root!r})
import torch.distributed as dist
import bench
if os.environ["RANK"] == "1" and {fail_rank1}:
    sys.exit(3)
world, rank, local = bench._dist("gloo")
worst = bench._max_over_ranks(1.0 + rank, world)
bench._barrier(world)
with open(os.path.join({out!r}, "rank%d.json" % rank), "w") as f:
    json.dump({{"world": world, "rank": rank, "local": local, "worst": worst,
               "addr": os.environ["MASTER_ADDR"]}}, f)
dist.destroy_process_group()
"""


def _child(tmp_path, fail_rank1=False):
    script = tmp_path / "child.py"
    script.write_text(_CHILD.format(root=_ROOT, out=str(tmp_path), fail_rank1=fail_rank1))
    return str(script)


def test_spawn_local_replicas_two_gloo_ranks(tmp_path):
    # bench.py --gpus N without torchrun starts N ranks itself: each gets the
    # torchrun environment (its own RANK / LOCAL_RANK, a shared WORLD_SIZE and
    # a rendezvous on 127.0.0.1), so they form one process group.
    import bench
    assert bench.spawn_local_replicas(2, [], script=_child(tmp_path)) == 0
    import json
    res = [json.loads((tmp_path / f"rank{r}.json").read_text()) for r in (0, 1)]
    assert [r["rank"] for r in res] == [0, 1] and [r["local"] for r in res] == [0, 1]
    assert all(r["world"] == 2 and r["worst"] == 2.0 and r["addr"] == "127.0.0.1" for r in res)


def test_spawn_local_replicas_reports_a_failed_rank(tmp_path):
    # Rank 1 exits with status 3 before it joins; rank 0, waiting for it at
    # the rendezvous, is stopped and the launcher returns the failure.
    import bench
    t0 = __import__("time").time()
    assert bench.spawn_local_replicas(2, [], script=_child(tmp_path, fail_rank1=True)) == 3
    assert __import__("time").time() - t0 < 60
    assert not (tmp_path / "rank0.json").exists()


def test_reference_arm_with_two_replicas_prints_one_line():
    # The reference arm under --gpus 2 without torchrun: two ranks start,
    # rank 0 alone runs the oracle and prints, n_gpus says 2.
    import json
    import subprocess
    import sys
    r = subprocess.run([sys.executable, os.path.join(_ROOT, "bench.py"), "--impl", "reference", "--gpus", "2",
                        "--workload", "tiny", "--steps", "1", "--warmup", "1"],
                       capture_output=True, text=True, timeout=300, cwd=_ROOT)
    assert r.returncode == 0, r.stderr
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    line = json.loads(lines[0])
    assert line["impl"] == "reference" and line["n_gpus"] == 2
