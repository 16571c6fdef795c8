"""bench.py's whole-job aggregation over ranks, on CPU with the gloo backend
and two processes: bytes add up over ranks, the step time is the slowest
rank's, and every rank sees the same result."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    try:
        ws, r, local = bench.dist_env()
        assert (ws, r, local) == (world, rank, rank)
        tot, ms = bench.aggregate(1000.0 * (rank + 1), 2.0 + rank)
        q.put((rank, tot, ms))
    finally:
        dist.destroy_process_group()


def test_aggregate_over_two_gloo_ranks():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, tot, ms in res:
        assert tot == pytest.approx(3000.0)  # 1000 + 2000 bytes
        assert ms == pytest.approx(3.0)      # the slower rank


def test_aggregate_single_process_is_identity():
    import bench
    assert bench.aggregate(123.0, 4.5) == (123.0, 4.5)
