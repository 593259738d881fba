"""The multi-GPU path is replicas only: each rank times the same work and the
job's value is all ranks' units over the slowest rank's time. Covered here
with two gloo ranks on the CPU."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    import bench
    ms = [3.0, 5.0][rank]                       # rank 1 is the slow one
    worst = bench.max_over_ranks(ms, world, torch.device("cpu"))
    q.put((rank, worst, bench.job_throughput(1000, world, worst)))
    dist.destroy_process_group()


def test_two_rank_aggregation():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    ps = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in ps:
        p.start()
    for p in ps:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert [g[1] for g in got] == [5.0, 5.0]
    assert all(abs(g[2] - 2 * 1000 / 5e-3) < 1e-6 for g in got)


def test_single_rank_is_identity():
    import bench
    assert bench.max_over_ranks(2.5, 1, torch.device("cpu")) == 2.5
    assert bench.job_throughput(10, 1, 2.0) == 10 / 2e-3
