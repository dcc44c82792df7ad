"""The bench's multi-rank aggregation on two gloo ranks (CPU): every rank sees
the slowest rank's timings, and the job throughput counts all ranks' calls over
that time."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, out):
    sys.path.insert(0, ROOT)
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    # rank r took 100 + 10 r ms for the device-timed steps and 300 - r ms end to end
    got = bench.max_over_ranks([100.0 + 10 * rank, 300.0 - rank], torch.device("cpu"), world)
    dist.barrier()
    out.put((rank, got, bench.job_throughput(world, 2, got[0])))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    import bench
    for rank, got, thr in res:
        assert got == [110.0, 300.0]
        assert thr == pytest.approx(world * bench.CALLS_PER_CHUNK * 2 / 0.110)


def test_single_rank_is_identity():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.max_over_ranks([1.5, 2.5], torch.device("cpu"), 1) == [1.5, 2.5]
    assert bench.job_throughput(1, 10, 1000.0) == pytest.approx(bench.CALLS_PER_CHUNK * 10)
