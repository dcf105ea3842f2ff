"""The benchmark's N > 1 path on CPU: two gloo ranks run its barrier, its max over ranks and
its weak-scaling aggregation, with the same calls the NCCL path makes on several GPUs."""
import os
import socket
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    sys.path.insert(0, ROOT)
    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        bench.barrier(world)
        # rank r took (r + 1) ms for the same work: the job is as slow as its slowest rank
        ms_max = bench.max_over_ranks(world, float(rank + 1))
        neg = bench.max_over_ranks(world, -float(10 * (rank + 1)))  # min via max of negatives
        value = bench.weak_scaling_value(world, 32768, ms_max)
        q.put((rank, ms_max, neg, value))
        bench.barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_aggregate_like_the_bench():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(2))
    for rank, ms_max, neg, value in res:
        assert ms_max == 2.0            # the slower rank's time, on every rank
        assert neg == -10.0             # the smaller of -10 and -20
        assert value == pytest.approx(2 * 32768 / 2e-3)   # all ranks' tokens over the max time


def test_reference_arm_prints_only_on_rank_zero():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference", "--steps", "1",
                        "--warmup", "0"], capture_output=True, text=True, env=env, timeout=120)
    assert r.returncode == 0 and r.stdout.strip() == ""
