"""The bench's N > 1 path on CPU: world-size-2 gloo ranks (one process per
rank, as torchrun runs one per GPU) agree on the slowest rank's time and on
the whole-job throughput (units of all ranks over that time). Replicas only:
the decode step has no data-path collective."""
import os
import socket

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank: int, world: int, port: int, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        t_local = 0.010 + 0.005 * rank  # rank 1 is the slow one
        t, value = bench.job_rate(t_local, 2.0e9, world, torch.device("cpu"))
        q.put((rank, t, value))
    finally:
        dist.destroy_process_group()


def test_job_rate_world_2():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, t, value in res:
        assert t == pytest.approx(0.015)          # max over ranks
        assert value == pytest.approx(2.0e9 * world / 0.015 / 1e9)  # all ranks' units


def test_job_rate_single():
    import bench
    t, value = bench.job_rate(0.02, 1.0e9, 1, torch.device("cpu"))
    assert t == 0.02 and value == pytest.approx(50.0)
