"""Multi-rank host logic of bench.py with two gloo ranks on the CPU: every
rank gets its own batch of the same shape (weak scaling), the job time is the
slowest rank's and the positions add up."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        p = bench.make_problem("skewed", rank)
        seconds = 1.0 + rank            # rank 1 is the slow one
        t, pos = bench.reduce_over_ranks(seconds, p.positions, dist, torch.device("cpu"))
        q.put((rank, p.positions, int(p.seq_lens.sum()), t, pos,
               bench.config_of("skewed", p, world)["parallelism"]))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_weak_scaling():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=180) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    (r0, pos0, _, t0, tot0, par0), (r1, pos1, _, t1, tot1, par1) = res
    assert pos0 != pos1                      # each rank has its own batch
    assert t0 == t1 == 2.0                   # slowest rank's time everywhere
    assert tot0 == tot1 == pos0 + pos1       # positions add up
    assert par0 == "dp2 (independent batches)"


def test_single_process_reduction_is_identity():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    assert bench.reduce_over_ranks(1.5, 7, None, None) == (1.5, 7)
