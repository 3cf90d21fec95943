"""The replica path of the benchmark: one process per GPU and no collective on
the data path, only a barrier around the timed steps and the maximum step
time over ranks.  Run as world-size-2 gloo process groups on the CPU."""
import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, ms, q):
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        bench.sync_ranks(torch)
        q.put((rank,) + bench.aggregate_ranks(torch, ms[rank], 1000, "cpu"))
        bench.sync_ranks(torch)
    finally:
        dist.destroy_process_group()


def test_single_process_is_its_own_job():
    import torch
    sys.path.insert(0, ROOT)
    import bench
    bench.sync_ranks(torch)   # no process group: nothing to wait for
    ms, value = bench.aggregate_ranks(torch, 2.0, 1000, "cpu")
    assert ms == 2.0 and value == pytest.approx(1000 / 2e-3)


def test_two_replicas_take_the_slowest_rank():
    """Both ranks report all rows of the job over the slowest rank's time."""
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ms = [1.5, 4.0]
    procs = [ctx.Process(target=_worker, args=(r, 2, port, ms, q)) for r in range(2)]
    for p in procs:
        p.start()
    out = [q.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for rank, m, value in out:
        assert m == 4.0, rank
        assert value == pytest.approx(2 * 1000 / 4e-3), rank
