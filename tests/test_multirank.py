"""Multi-rank host logic on the CPU: two gloo ranks, no GPU.

The path shards over (batch, head) with no exchange, so several GPUs run
independent replicas.  What is tested here is the bench's whole-job
aggregation: every rank's time, the max over ranks, and the value of N
replicas.
"""
import os
import socket

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    return dist


def _bench_worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import bench
    dist = _init(rank, world, port)
    ms = [3.0, 5.0][rank]  # the second rank is slower
    got = bench.max_over_ranks(ms, world, "cpu")
    val = bench.whole_job_value(1e12, got, world)
    gathered = [None] * world
    dist.all_gather_object(gathered, (got, val))
    if rank == 0:
        out.put(gathered)
    dist.destroy_process_group()


def test_bench_aggregation_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.spawn(_bench_worker, args=(2, _free_port(), q), nprocs=2, join=True)
    res = q.get(timeout=60)
    for got, val in res:
        assert got == 5.0                       # every rank sees the slowest time
        assert abs(val - 2 * 1e12 / 5e-3 / 1e12) < 1e-9  # two replicas in 5 ms
