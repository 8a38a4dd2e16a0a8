"""The benchmark's multi-rank aggregation on CPU: two gloo ranks report
different elapsed times and unit counts; every rank gets the slowest time
and the summed units (the whole-job throughput the JSON line reports)."""
import os
import socket

import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import bench


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        elapsed = [12.5, 20.0][rank]
        units = [1000.0, 1536.0][rank]
        t, u = bench._aggregate(elapsed, units, torch.device("cpu"))
        out[rank] = (t, u)
    finally:
        dist.destroy_process_group()


def test_two_rank_aggregation_gloo():
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, 2, port, out)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        assert out[0] == out[1] == (20.0, 2536.0)


def test_single_process_passthrough():
    assert bench._aggregate(3.0, 7.0, torch.device("cpu")) == (3.0, 7.0)
