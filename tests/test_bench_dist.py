"""The benchmark's multi-GPU host logic on CPU: two gloo ranks, as torchrun
would launch them (replicas, barrier, max over ranks, whole-job value)."""
import os
import socket

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _rank_main(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    import torch
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    bench.barrier(ws)
    # each replica "took" a different time; the job took the slowest one's
    t = bench.max_over_ranks(0.001 * (rank + 1), ws, torch.device("cpu"))
    value = bench.job_value(1 << 30, 16, t, ws)
    out[rank] = (t, value)
    bench.barrier(ws)
    dist.destroy_process_group()


def test_two_gloo_replicas_take_the_slowest_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        results = dict(out)
    import bench
    for r in range(world):
        t, value = results[r]
        assert t == pytest.approx(0.002)
        _, bus = bench.bus_bw(1 << 30, 16, 0.002)
        assert value == pytest.approx(2 * bus)


def test_busbw_formula():
    import bench
    alg, bus = bench.bus_bw(1 << 30, 16, 0.5)
    assert alg == pytest.approx((1 << 30) / 0.5 / 1e9)
    assert bus == pytest.approx(alg * 2 * 15 / 16)
