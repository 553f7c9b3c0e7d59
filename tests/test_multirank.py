"""The multi-rank host logic of bench.py on CPU: two gloo ranks, each timing
its own replica, reduce to the max time and the summed unit count that the
aggregate value is computed from (no GPU and no data-path collective)."""
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


def _rank(rank, world, port, out):
    import torch.distributed as dist
    import bench
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    ws, r, local = bench.dist_env()
    assert (ws, r, local) == (world, rank, rank)
    t_ms = 10.0 + 5.0 * rank               # rank 1 is the slow one
    steps = 100
    t_max = bench.max_over_ranks(t_ms, ws)
    units = bench.sum_over_ranks(float(steps), ws)
    out[rank] = (t_max, units, 1000.0 * t_max / units)
    dist.barrier()
    dist.destroy_process_group()


def test_two_gloo_ranks_reduce_time_and_units():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_rank, args=(r, world, port, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(120)
            assert p.exitcode == 0
        res = dict(out)
    for r in range(world):
        t_max, units, us = res[r]
        assert t_max == pytest.approx(15.0)
        assert units == pytest.approx(200.0)
        assert us == pytest.approx(75.0)   # 15 ms over 200 layer-steps of both replicas
