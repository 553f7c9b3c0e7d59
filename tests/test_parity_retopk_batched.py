"""Batched ReTopK with per-request state (continuous batching), in lockstep
with one oracle instance per sequence.

Four sequences of different lengths share one paged cache (16-token pages in
a seeded random order).  Each has its own handle, FIFO state, step counter and
oracle; a call takes the sequences active at that step in a shuffled order:
sequences 0-2 from step 0, sequence 3 joins at step 10 (its own step 0, a
refresh), sequence 1 retires after step 14.  For every sequence and head the
path, the candidate set A_t and the support S_t must equal its own oracle's
(bit-exact, the lockstep rules of test_parity_retopk), and the output must be
within 2e-3.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from helpers import OUT_TOL, TIE_REL
from workloads.gen import bits, make_retopk

pytestmark = pytest.mark.gpu


def test_batched_retopk_mixed_lengths_join_and_retire():
    import top_retrieval_sparse_gb300 as tsa
    dev = "cuda"
    lens0 = [5000, 7300, 6100, 8200]
    steps = 24
    joins = {0: 0, 1: 0, 2: 0, 3: 10}
    retires = {1: 15}  # not active from step 15 on
    wls = [make_retopk(L0=L0, steps=steps, K=64, C=8, R=2, W=8, T_r=16, seed=11 + i)
           for i, L0 in enumerate(lens0)]
    Hq, Hkv, d, K = wls[0].Hq, wls[0].Hkv, wls[0].d, wls[0].K
    G = Hq // Hkv
    ps = 16
    lcap = max(w.lcap for w in wls)
    max_pages = lcap // ps
    pages = [w.lcap // ps for w in wls]
    total = sum(pages)
    perm = torch.randperm(total, generator=torch.Generator().manual_seed(5)).to(torch.int32)
    kp = torch.zeros((total, Hkv, ps, d), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    rows = torch.zeros((len(wls), max_pages), dtype=torch.int32)
    base = 0
    for i, w in enumerate(wls):
        pg = perm[base:base + pages[i]].long()
        kp[pg.to(dev)] = w.k[0].reshape(Hkv, pages[i], ps, d).transpose(0, 1).to(dev)
        vp[pg.to(dev)] = w.v[0].reshape(Hkv, pages[i], ps, d).transpose(0, 1).to(dev)
        rows[i, :pages[i]] = pg.to(torch.int32)
        base += pages[i]
    rows = rows.to(dev)

    handles, oracles, t_of = [], [], []
    kb = [[bits(w.k[0, g]) for g in range(Hkv)] for w in wls]
    vb = [[bits(w.v[0, g]) for g in range(Hkv)] for w in wls]
    for i, w in enumerate(wls):
        kv1 = tsa.kv_paged(kp, vp, rows[i:i + 1].contiguous())
        sup, cnt = tsa.prefill_supports(w.q_prefill.to(dev).contiguous(), kv1, w.L0, K, w.scale)
        g = tsa.ReTopK(Hq, Hkv, d, K, w.C, w.R, w.W, w.tau, w.T_r, lcap)
        g.init(w.q_prefill.to(dev).contiguous(), sup, cnt)
        o = orc.ReTopK(Hq, d, K, w.C, w.R, w.W, w.tau, w.T_r, path_abs=1e-5, rho_abs=1e-5,
                       topk_rel=TIE_REL)
        qpre = bits(w.q_prefill)
        sh, ch = sup.cpu().numpy(), cnt.cpu().numpy()
        for c in range(w.C):
            for h in range(Hq):
                o.set_slot(h, c, qpre[c, h], sh[c, h, : ch[c, h]])
        handles.append(g)
        oracles.append(o)
        t_of.append(0)
    ws = torch.zeros(tsa.ReTopK.batched_workspace_size(handles[0], len(wls)), dtype=torch.uint8,
                     device=dev)
    rng = np.random.default_rng(9)
    cap = wls[0].R * K + wls[0].W
    seen = {"exact": 0, "reuse": 0, "adopt": 0}
    for step in range(steps):
        active = [i for i in range(len(wls)) if joins[i] <= step < retires.get(i, steps)]
        rng.shuffle(active)
        n = len(active)
        q = torch.stack([wls[i].q_all[t_of[i]] for i in active]).to(dev).contiguous()
        lens = [wls[i].length(t_of[i]) for i in active]
        kv = tsa.kv_paged(kp, vp, rows[torch.tensor(active, device=dev)].contiguous())
        so = torch.empty((n, Hq, K), dtype=torch.int32, device=dev)
        po = torch.empty((n, Hq), dtype=torch.int32, device=dev)
        mo = torch.empty((n, Hq), dtype=torch.int32, device=dev)
        co = torch.empty((n, Hq, cap), dtype=torch.int32, device=dev)
        out = tsa.ReTopK.step_batched([handles[i] for i in active], q, kv, lens, wls[0].scale,
                                      support_out=so, path_out=po, mcand_out=mo, cand_out=co,
                                      workspace=ws)
        torch.cuda.synchronize()
        out, so, po, mo, co = (x.cpu().numpy() for x in (out, so, po, mo, co))
        for j, i in enumerate(active):
            w, o, t, L = wls[i], oracles[i], t_of[i], lens[j]
            qb = bits(w.q_all[t])
            for h in range(Hq):
                sg = so[j, h][so[j, h] >= 0]
                cg = co[j, h][: mo[j, h]] if po[j, h] == 0 else None
                r = o.step_head(h, qb[h], kb[i][h // G][:L], vb[i][h // G][:L], w.scale,
                                other_path=int(po[j, h]), other_cand=cg, other_sup=sg)
                assert r["path"] == po[j, h], f"seq {i} t={t} h={h}: path"
                if r["path"] == 0:
                    assert r["cand_ok"] in (1, 2), f"seq {i} t={t} h={h}: candidate set"
                    assert mo[j, h] == len(r["cand"])
                else:
                    assert mo[j, h] == L
                assert r["sup_ok"] in (1, 2), f"seq {i} t={t} h={h}: support"
                assert np.max(np.abs(out[j, h] - r["out"])) <= OUT_TOL, f"seq {i} t={t} h={h}"
                seen["exact" if r["path"] else "reuse"] += 1
                seen["adopt"] += r["adopt_path"] + r["adopt_cand"]
            o.advance()
            t_of[i] += 1
            assert handles[i].counters() == (t_of[i], t_of[i] % w.C)
    assert seen["reuse"] > 0 and seen["exact"] > 0 and seen["adopt"] <= 1
    assert t_of == [24, 15, 24, 14]
    assert tsa.workspace_status(ws) == 0


def test_batched_step_equals_single_steps():
    """Two sequences stepped together equal the same sequences stepped one at
    a time (same supports and paths, outputs within 1e-5)."""
    import top_retrieval_sparse_gb300 as tsa
    dev = "cuda"
    wls = [make_retopk(L0=L0, steps=8, K=48, C=6, R=3, W=5, T_r=4, seed=3 + i)
           for i, L0 in enumerate((4000, 4500))]
    lcap = max(w.lcap for w in wls)
    Hq, Hkv, d, K = wls[0].Hq, wls[0].Hkv, wls[0].d, wls[0].K
    k = torch.zeros((2, Hkv, lcap, d), dtype=torch.bfloat16, device=dev)
    v = torch.zeros_like(k)
    for i, w in enumerate(wls):
        k[i, :, :w.lcap] = w.k[0].to(dev)
        v[i, :, :w.lcap] = w.v[0].to(dev)
    kv2 = tsa.kv_contiguous(k, v)
    runs = []
    for batched in (True, False):
        hs = []
        for i, w in enumerate(wls):
            kv1 = tsa.kv_contiguous(k[i:i + 1].contiguous(), v[i:i + 1].contiguous())
            sup, cnt = tsa.prefill_supports(w.q_prefill.to(dev).contiguous(), kv1, w.L0, K, w.scale)
            g = tsa.ReTopK(Hq, Hkv, d, K, w.C, w.R, w.W, w.tau, w.T_r, lcap)
            g.init(w.q_prefill.to(dev).contiguous(), sup, cnt)
            hs.append((g, kv1))
        rec = []
        for t in range(8):
            q = torch.stack([w.q_all[t] for w in wls]).to(dev).contiguous()
            lens = [w.length(t) for w in wls]
            so = torch.empty((2, Hq, K), dtype=torch.int32, device=dev)
            po = torch.empty((2, Hq), dtype=torch.int32, device=dev)
            if batched:
                out = tsa.ReTopK.step_batched([g for g, _ in hs], q, kv2, lens, wls[0].scale,
                                              support_out=so, path_out=po)
            else:
                out = torch.empty((2, Hq, d), dtype=torch.float32, device=dev)
                for i, (g, kv1) in enumerate(hs):
                    g.step(q[i].contiguous(), kv1, lens[i], wls[0].scale, out=out[i],
                           support_out=so[i], path_out=po[i])
            rec.append((out.clone(), so.clone(), po.clone()))
        torch.cuda.synchronize()
        runs.append(rec)
    for t, (a, b) in enumerate(zip(*runs)):
        assert torch.equal(a[2], b[2]), f"t={t}: paths"
        for i in range(2):
            for h in range(Hq):
                assert set(a[1][i, h].tolist()) == set(b[1][i, h].tolist()), (t, i, h)
        assert torch.max(torch.abs(a[0] - b[0])).item() < 1e-5
