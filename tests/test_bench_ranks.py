"""The multi-rank bench arithmetic on CPU: two gloo ranks reduce their timings (max) and bytes
(sum) and report the whole-job throughput every rank agrees on."""
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
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    times = [[12.0, 20.0], [15.0, 18.0]][rank]       # per-rank (step total, e2e total) in ms
    nbytes = [[3.0e9], [2.0e9]][rank]                 # per-rank bytes over the timed steps
    slow, slow_e2e = bench.reduce_across_ranks(times, "max", world, torch.device("cpu"))
    (total,) = bench.reduce_across_ranks(nbytes, "sum", world, torch.device("cpu"))
    q.put((rank, slow, slow_e2e, total, bench.job_throughput(total, slow)))
    dist.destroy_process_group()


def test_two_rank_reduction_and_throughput():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    procs = [ctx.Process(target=_rank, args=(r, world, port, q)) for r in range(world)]
    for p in procs:
        p.start()
    got = sorted(q.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, slow, slow_e2e, total, gbs in got:
        assert slow == 15.0 and slow_e2e == 20.0     # the slowest rank sets the time
        assert total == 5.0e9                         # every rank's bytes count
        assert gbs == pytest.approx(5.0e9 / 15.0e-3 / 1e9)


def test_single_rank_is_identity():
    import bench
    assert bench.reduce_across_ranks([1.5, 2.5], "max", 1, torch.device("cpu")) == [1.5, 2.5]
    assert bench.job_throughput(1e9, 1000.0) == pytest.approx(1.0)
