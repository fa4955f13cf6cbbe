"""The N > 1 host logic of bench.py on CPU: two gloo ranks agree on the
max-over-ranks time and report whole-job throughput (units of all ranks over
that time).  The path itself is replicas only (independent (batch, kv-head)
groups per rank, no data-path collective)."""
import os
import socket

import pytest
import torch.multiprocessing as mp


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, secs, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import torch.distributed as dist

    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (world, rank, rank)
        value, t = bench.aggregate_throughput(1000.0, secs[rank], world, "gloo")
        out[rank] = (value, t)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation():
    world = 2
    port = _free_port()
    secs = [2.0, 5.0]
    ctx = mp.get_context("spawn")
    out = ctx.Manager().dict()
    procs = [ctx.Process(target=_worker, args=(r, world, port, secs, out)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    for r in range(world):
        value, t = out[r]
        assert t == 5.0
        assert value == pytest.approx(2 * 1000.0 / 5.0)


def test_single_process_is_identity():
    import bench

    assert bench.reduce_max(3.5, None) == 3.5
    assert bench.aggregate_throughput(10.0, 2.0, 1, None) == (5.0, 2.0)
