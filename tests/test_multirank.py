"""Multi-rank host logic on the CPU: two gloo ranks, no GPU.

- The bench's whole-job aggregation: every rank's time, the max over ranks,
  and the value of N replicas.
- Context parallelism across ranks with the zigzag assignment: each rank
  localizes the mask for its own query chunks against every key chunk (no
  communication: it needs only the global boundary vectors) and computes
  them with the oracle; rank 0 gathers the chunks and checks them against
  the attention of the whole sequence.
"""
import os
import socket

import numpy as np
import pytest
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


def _cp_worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import oracle
    from sparse_masked_attention_gb300 import workloads as W
    from sparse_masked_attention_gb300.attention import zigzag_assignment
    dist = _init(rank, world, port)
    N, d, C = 320, 16, 2 * world
    L = N // C
    rng = np.random.default_rng(0)          # every rank draws the same inputs
    mask = W.share_question(N, [W.share_question_groups(rng, N, (40, 90), (2, 3), (15, 40))])
    q, k, v = (rng.standard_normal((N, d)) for _ in range(3))
    ms = mask.slice(0)
    mine = {}
    for qc in zigzag_assignment(C, world)[rank]:
        q0 = qc * L
        o = np.zeros((L, d))
        lse = np.full(L, -np.inf)
        for kc in range(C):
            local, lc = oracle.localize(ms, N, mask.causal, q0, kc * L, L)
            if local is None:
                continue
            po, pl = oracle.attention_fwd(q[q0:q0 + L], k[kc * L:(kc + 1) * L],
                                          v[kc * L:(kc + 1) * L], local, lc)
            new = np.logaddexp(lse, pl)
            fin = np.isfinite(new)
            wa = np.where(fin, np.exp(lse - np.where(fin, new, 0)), 0.0)
            wb = np.where(fin, np.exp(pl - np.where(fin, new, 0)), 0.0)
            o = o * wa[:, None] + po * wb[:, None]
            lse = new
        mine[qc] = (o, lse)
    gathered = [None] * world
    dist.all_gather_object(gathered, mine)
    if rank == 0:
        o_all = np.zeros((N, d))
        l_all = np.zeros(N)
        owners = {}
        for r, part in enumerate(gathered):
            for qc, (o, lse) in part.items():
                owners[qc] = r
                o_all[qc * L:(qc + 1) * L] = o
                l_all[qc * L:(qc + 1) * L] = lse
        ro, rl = oracle.attention_fwd(q, k, v, ms, mask.causal)
        out.put((sorted(owners.items()), float(np.max(np.abs(o_all - ro))),
                 float(np.max(np.abs(l_all - rl)))))
    dist.destroy_process_group()


def test_zigzag_context_parallel_over_two_gloo_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    mp.spawn(_cp_worker, args=(2, _free_port(), q), nprocs=2, join=True)
    owners, err_o, err_l = q.get(timeout=120)
    assert owners == [(0, 0), (1, 1), (2, 1), (3, 0)]  # rank r owns chunks r and 3 - r
    assert err_o < 1e-12 and err_l < 1e-12
