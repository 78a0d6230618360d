"""The benchmark's multi-rank host logic on CPU with two gloo ranks: the job
time is the slowest rank's, the value is whole-job (weak scaling: every rank
adds its own bucket), and only rank 0 of the reference arm does any work."""
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    t = bench.reduce_max(10.0 + 5.0 * rank, torch.device("cpu"))
    v = bench.weak_scaling_value(2e9, 10, world, t)
    dist.barrier()
    dist.destroy_process_group()
    q.put((rank, t, v))


def test_two_rank_max_and_weak_scaling_value():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
    assert all(p.exitcode == 0 for p in procs)
    res = sorted(q.get(timeout=5) for _ in range(2))
    for rank, t, v in res:
        assert t == 15.0                                   # the slowest rank's time
        assert abs(v - 2e9 * 10 * 2 / 15e-3 / 1e12) < 1e-12  # both ranks' work counted


def test_single_process_reduce_is_identity():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_max(3.5, torch.device("cpu")) == 3.5
    assert bench.weak_scaling_value(1e12, 1, 1, 1000.0) == 1.0


def test_reference_arm_nonzero_rank_exits_without_work():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                        "--gpus", "2", "--steps", "1", "--warmup", "3"],
                       capture_output=True, text=True, env=env, timeout=300)
    assert r.returncode == 0
    assert r.stdout.strip() == ""
