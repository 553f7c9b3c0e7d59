"""A sequence split over shards, in the library (RetrievalAttention Eq. 4-5:
attention partials over disjoint sets merge exactly).

Two shards of one cache run in one process on one GPU: each runs
sparse_attn_decode_shard (its local top-K outside the global window), the K
(logit, global position) pairs of both are merged on the host into the global
top-K, each shard runs attend_set over the selected rows it holds plus its
window rows, and lse_merge folds the two (out, lse).  The result must equal
the unsharded step under the oracle's rules (top-K set up to the near-tie
rule, output within 2e-3).  The exchange itself across processes is covered
by the gloo test in test_multirank.py.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from helpers import LSE_TOL, OUT_TOL, TIE_REL
from workloads.gen import bits, make_decode

pytestmark = pytest.mark.gpu


def split_step(wl, cuts, K):
    import top_retrieval_sparse_gb300 as tsa
    dev = "cuda"
    L = wl.lens(0)[0]
    q = wl.q(0)[0].to(dev).contiguous()          # [Hq][128]
    Hq, d = q.shape
    bounds = [0] + list(cuts) + [L]
    shards = []
    for s in range(len(bounds) - 1):
        lo, hi = bounds[s], bounds[s + 1]
        kv = tsa.kv_contiguous(wl.k[:, :, lo:hi].to(dev).contiguous(),
                               wl.v[:, :, lo:hi].to(dev).contiguous())
        idx = torch.full((Hq, K), -1, dtype=torch.int32, device=dev)
        sc = torch.empty((Hq, K), dtype=torch.float32, device=dev)
        tsa.decode_shard(q, kv, hi - lo, lo, L, K, wl.n_init, wl.n_recent, wl.scale,
                         topk_idx=idx, topk_score=sc)
        shards.append((lo, hi, kv, idx.cpu().numpy(), sc.cpu().numpy()))
    torch.cuda.synchronize()
    # host merge of the exchanged pairs: order (logit desc, global position asc)
    sel = []
    for h in range(Hq):
        pairs = [(float(sc[h, j]), lo + int(idx[h, j]))
                 for lo, hi, kv, idx, sc in shards for j in range(K) if idx[h, j] >= 0]
        pairs.sort(key=lambda p: (-p[0], p[1]))
        sel.append(np.array(sorted(p for _, p in pairs[:K]), np.int64))
    # per shard: its selected rows plus its window rows, attended as one set
    win = orc.window_positions(L, wl.n_init, wl.n_recent)
    outs, lses = [], []
    for lo, hi, kv, _, _ in shards:
        rows = [sorted([p - lo for p in sel[h] if lo <= p < hi] +
                       [p - lo for p in win if lo <= p < hi]) for h in range(Hq)]
        M = max(1, max(len(r) for r in rows))
        pos = torch.full((1, Hq, M), -1, dtype=torch.int32)
        cnt = torch.tensor([[len(r) for r in rows]], dtype=torch.int32)
        for h, r in enumerate(rows):
            pos[0, h, :len(r)] = torch.tensor(r, dtype=torch.int32)
        lse = torch.empty((1, Hq), dtype=torch.float32, device=dev)
        o = tsa.attend_set(q[None], kv, pos.to(dev), cnt.to(dev), wl.scale, lse_out=lse)
        outs.append(o[0])
        lses.append(lse[0])
    o, lse = outs[0], lses[0]
    for o2, l2 in zip(outs[1:], lses[1:]):
        o, lse = tsa.lse_merge(o, lse, o2, l2)
    torch.cuda.synchronize()
    return sel, o.cpu().numpy(), lse.cpu().numpy()


@pytest.mark.parametrize("cuts", [(17_000,), (29_700,), (9_000, 21_000)])
def test_shards_reproduce_the_unsharded_step(cuts):
    """Two or three shards; with the cut at L - 300 the recent window (512
    positions) spans both shards, and the initial window always lies in the
    first."""
    K = 256
    wl = make_decode("llama128k", L0=30_000, steps=1, K=K)
    L = wl.lens(0)[0]
    sel, out, lse = split_step(wl, cuts, K)
    G = wl.Hq // wl.Hkv
    pool = np.array([i for i in range(L) if not orc.in_window(i, L, wl.n_init, wl.n_recent)],
                    np.int64)
    for h in range(wl.Hq):
        kb, vb, qb = bits(wl.k[0, h // G, :L]), bits(wl.v[0, h // G, :L]), bits(wl.q(0)[0, h])
        r = orc.decode_head(qb, kb, vb, K, wl.n_init, wl.n_recent, wl.scale)
        verdict = orc.topk_check(r["z"], pool, K, sel[h], TIE_REL)
        assert verdict in (1, 2), f"h={h}: merged top-K rejected"
        ref_out, ref_lse = orc.decode_eval_set(r["z"], vb, wl.n_init, wl.n_recent, sel[h])
        assert np.max(np.abs(out[h] - ref_out)) <= OUT_TOL, f"h={h}"
        assert abs(lse[h] - ref_lse) <= LSE_TOL, f"h={h}"


def test_attend_set_matches_oracle_and_ignores_rows_past_the_cache():
    """attend_set over random sets (sizes 0..M, one head with an empty set)
    equals the oracle's partial (Eq. 3) on the same rows; a position past the
    cache is left out and reported as a device-side check."""
    import top_retrieval_sparse_gb300 as tsa
    wl = make_decode("tiny", L0=5000, steps=1)
    dev = "cuda"
    L = wl.lens(0)[0]
    kv = tsa.kv_contiguous(wl.k.to(dev), wl.v.to(dev))
    rng = np.random.default_rng(5)
    M = 300
    Hq = wl.Hq
    sets = [np.sort(rng.choice(L, size=s, replace=False)) for s in (300, 17, 0, 129)]
    pos = torch.full((1, Hq, M), -1, dtype=torch.int32)
    cnt = torch.tensor([[len(x) for x in sets]], dtype=torch.int32)
    for h, x in enumerate(sets):
        pos[0, h, :len(x)] = torch.tensor(x, dtype=torch.int32)
    lse = torch.empty((1, Hq), dtype=torch.float32, device=dev)
    n = tsa.lib().tsa_attend_set_workspace_size(1, Hq, M)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    out = tsa.attend_set(wl.q(0).to(dev).contiguous(), kv, pos.to(dev), cnt.to(dev), wl.scale,
                         lse_out=lse, workspace=ws)
    torch.cuda.synchronize()
    out, lse = out.cpu().numpy(), lse.cpu().numpy()
    for h, x in enumerate(sets):
        z = orc.scores(bits(wl.q(0)[0, h]), bits(wl.k[0, 0, :L]), wl.scale)
        o, m, l, ls = orc.partial(z, x, bits(wl.v[0, 0, :L]))
        if len(x):
            assert np.max(np.abs(out[0, h] - o)) <= OUT_TOL and abs(lse[0, h] - ls) <= LSE_TOL
        else:
            assert np.all(out[0, h] == 0) and lse[0, h] == -np.inf
    assert tsa.workspace_status(ws) == 0
    # one row past the cache: ignored, flagged
    pos[0, 1, 3] = kv.l_cap + 7
    out2 = tsa.attend_set(wl.q(0).to(dev).contiguous(), kv, pos.to(dev), cnt.to(dev), wl.scale,
                          workspace=ws)
    torch.cuda.synchronize()
    assert tsa.workspace_status(ws) == -5
    x = np.delete(sets[1], 3)
    z = orc.scores(bits(wl.q(0)[0, 1]), bits(wl.k[0, 0, :L]), wl.scale)
    o, _, _, _ = orc.partial(z, x, bits(wl.v[0, 0, :L]))
    assert np.max(np.abs(out2.cpu().numpy()[0, 1] - o)) <= OUT_TOL
