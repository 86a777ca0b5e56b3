"""bench.py's multi-rank logic on CPU with gloo, world size 2: the step time
is the slowest rank's, the job value counts every rank's drafted tokens, and
the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    p = s.getsockname()[1]
    s.close()
    return p


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = bench.max_over_ranks(1.0 + rank * 0.5)             # rank 1 is slower
    val = bench.job_throughput(ms, 15, world)
    args = type("A", (), dict(warmup=0, steps=1, workload="tiny"))()
    ref = bench.run_reference(args, rank, world, 0) if rank == 1 else None   # non-zero rank: no work
    q.put((rank, ms, val, ref))
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_agree_on_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    out = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, val, ref in out:
        assert ms == pytest.approx(1.5)
        assert val == pytest.approx(2 * 15 / 1.5e-3)
    assert out[1][3] is None


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks(2.5) == 2.5
    assert bench.job_throughput(2.0, 15, 1) == pytest.approx(7500.0)
