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


# ---- sequence sharding of one decode step (the exchange a 1M+ context split
# over ranks would use), on gloo ranks with the oracle's arithmetic ----------
def _shard_rank(rank, world, port, out):
    import numpy as np
    import torch.distributed as dist

    import oracle as orc
    from workloads.gen import bits, make_decode
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    wl = make_decode("tiny")  # 4 query heads / 1 KV head, K = 64, window 4 + 64
    L = wl.lens(0)[0]
    cut = [0, 2345, L]  # ragged shards of the sequence
    s0, s1 = cut[rank], cut[rank + 1]
    k, v = bits(wl.k[0, 0, s0:s1]), bits(wl.v[0, 0, s0:s1])
    res = {}
    for h in range(wl.Hq):
        q = bits(wl.q(0)[0, h])
        z = orc.scores(q, k, wl.scale)                       # this shard's logits
        win = [i for i in range(s1 - s0) if orc.in_window(s0 + i, L, wl.n_init, wl.n_recent)]
        pool = [i for i in range(s1 - s0) if not orc.in_window(s0 + i, L, wl.n_init,
                                                                wl.n_recent)]
        loc = orc.topk(z, pool, wl.K)                        # local top-K (shard indices)
        mine = [(float(z[i]), s0 + int(i)) for i in loc]
        # exchange 1: every shard's K (logit, position) pairs -> the global top-K
        allp = [None] * world
        dist.all_gather_object(allp, mine)
        pairs = sorted((p for part in allp for p in part), key=lambda p: (-p[0], p[1]))
        omega = {pos for _, pos in pairs[: wl.K]}
        sel = [pos - s0 for pos in range(s0, s1) if pos in omega]
        # this shard's partials over its window rows and its selected rows
        pw = orc.partial(z, win, v)[:3] if win else (np.zeros(wl.d), -np.inf, 0.0)
        po = orc.partial(z, sel, v)[:3] if sel else (np.zeros(wl.d), -np.inf, 0.0)
        # exchange 2: (o, m, l) per set -> Eq. 4-5 across shards, then W with Omega
        allw, allo = [None] * world, [None] * world
        dist.all_gather_object(allw, pw)
        dist.all_gather_object(allo, po)

        def fold(parts):
            o, m, l = parts[0]
            for o2, m2, l2 in parts[1:]:
                o, lse = orc.merge(o, m, l, o2, m2, l2)
                m, l = (lse, 1.0) if lse > -np.inf else (-np.inf, 0.0)
            return o, m, l

        ow, mw, lw = fold(allw)
        oo, mo, lo = fold(allo)
        o, lse = orc.merge(ow, mw, lw, oo, mo, lo)
        res[h] = (sorted(omega), o.tolist(), lse)
    out[rank] = res
    dist.barrier()
    dist.destroy_process_group()


def test_sequence_shards_reproduce_the_unsharded_step():
    """Two ranks each hold a ragged half of the sequence: local top-K, one
    all-gather of K (logit, position) pairs for the global top-K, per-shard
    partials over their window and selected rows, a second all-gather and the
    Eq. 4-5 merge give the oracle's unsharded step (same set, same output)."""
    import numpy as np

    import oracle as orc
    from workloads.gen import bits, make_decode
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        procs = [ctx.Process(target=_shard_rank, args=(r, world, port, out))
                 for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(300)
            assert p.exitcode == 0
        res = dict(out)
    wl = make_decode("tiny")
    L = wl.lens(0)[0]
    for h in range(wl.Hq):
        ref = orc.decode_head(bits(wl.q(0)[0, h]), bits(wl.k[0, 0, :L]), bits(wl.v[0, 0, :L]),
                              wl.K, wl.n_init, wl.n_recent, wl.scale)
        for r in range(world):
            omega, o, lse = res[r][h]
            assert omega == sorted(ref["sel"].tolist())
            np.testing.assert_allclose(o, ref["out"], rtol=0, atol=1e-12)
            assert abs(lse - ref["lse"]) <= 1e-12 * max(1.0, abs(ref["lse"]))
