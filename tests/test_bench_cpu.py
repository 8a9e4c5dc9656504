"""The replica aggregation of bench.py under torch.distributed (gloo, world_size 2, CPU): every rank
streams the same bytes; the whole-job value is the total over ranks divided by the slowest rank's
time, which every rank learns through the all-gather."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist

    import bench
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        t = 1.0 + rank  # rank 1 is the slower replica
        times = bench.max_over_ranks(t, world)
        value, tmax = bench.aggregate(1e9, times)
        q.put((rank, times, value, tmax))
    finally:
        dist.destroy_process_group()


def test_replica_aggregation_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, times, value, tmax in res:
        assert times == [1.0, 2.0]
        assert tmax == 2.0
        assert value == pytest.approx(2 * 1e9 / 2.0 / 1e9)  # 2 ranks x 1 GB over the slowest 2 s


def test_aggregate_single_rank():
    import bench
    v, t = bench.aggregate(17555292160, [0.0075])
    assert t == 0.0075 and v == pytest.approx(17555292160 / 0.0075 / 1e9)
