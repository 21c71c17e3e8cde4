"""Multi-rank timing of bench.py on CPU: two gloo ranks (the replicated
N > 1 path without GPUs).  Every rank must see the slowest rank's time and
the whole-job value must count all ranks' bytes."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        ms_local = 10.0 * (rank + 1)  # rank 1 is the slow one
        ms, value = bench.aggregate_ranks(ms_local, world, wbytes=1_000_000, steps=100, dist=dist)
        out.put((rank, ms, value))
        dist.barrier()
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_job_value():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    world = 2
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    res = sorted(q.get(timeout=10) for _ in range(world))
    for rank, ms, value in res:
        assert ms == 20.0                            # the slowest rank's time
        assert value == pytest.approx(2 * 1_000_000 * 100 / 0.020 / 1e9)  # both ranks' bytes


def test_single_rank_is_local_time():
    import bench
    ms, value = bench.aggregate_ranks(4.0, 1, wbytes=2_000_000, steps=10)
    assert ms == 4.0 and value == pytest.approx(2_000_000 * 10 / 0.004 / 1e9)
