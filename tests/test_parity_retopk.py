"""GPU parity of retopk_step against the ReTopK oracle, run in lockstep.

Per step and head: the path decision, the candidate set A_t (bit-exact) and
the support S_t (bit-exact up to the near-tie rule) must match the oracle;
the output must be within 2e-3 max-abs of the oracle evaluated on the support.
Where the oracle's own decision lies within a rounding margin (|max rho - tau|,
rho_(R) vs rho_(R+1), the top-K near-tie) it adopts the GPU's choice, so one
rounding-level tie does not diverge the two caches.  Adoption is bounded: at
most one head-step in a thousand (at least one allowed) may take the GPU's
decision, and the fp32 normalised queries the GPU pushes into its FIFO must be
within 1e-6 (per component) of the fp64 normalisation; with the 128-term fp32
dot product's own rounding that keeps every GPU cosine within a few 1e-6 of
the oracle's, inside the 1e-5 adoption margin.
"""
import numpy as np
import pytest
import torch

import oracle as orc
from helpers import OUT_TOL, TIE_REL
from workloads.gen import bits, make_retopk

pytestmark = pytest.mark.gpu


def gpu_prefill_supports(tsa, wl, kv, dev):
    """Exact top-K of each prefill query over its causal prefix (no window),
    computed with the library's prefill entry point (one call)."""
    return tsa.prefill_supports(wl.q_prefill.to(dev).contiguous(), kv, wl.L0, wl.K, wl.scale)


def decode_prefill_supports(tsa, wl, kv, dev):
    """The same supports from one sparse_attn_decode call per prefill query."""
    Cn, Hq, K = wl.C, wl.Hq, wl.K
    sup = torch.full((Cn, Hq, K), -1, dtype=torch.int32, device=dev)
    for c in range(Cn):
        p = wl.L0 - Cn + c
        q = wl.q_prefill[c].to(dev)[None].contiguous()
        lens = torch.tensor([p + 1], dtype=torch.int32, device=dev)
        idx = torch.empty((1, Hq, K), dtype=torch.int32, device=dev)
        tsa.sparse_attn_decode(q, kv, lens, K, 0, 0, wl.scale, topk_idx=idx)
        sup[c] = idx[0]
    cnt = (sup >= 0).sum(-1).to(torch.int32)
    return sup, cnt


def run_lockstep(wl, steps, check_out=True, verify_prefill=True):
    import top_retrieval_sparse_gb300 as tsa
    dev = "cuda"
    G = wl.Hq // wl.Hkv
    kv = tsa.kv_contiguous(wl.k.to(dev), wl.v.to(dev))
    g = tsa.ReTopK(wl.Hq, wl.Hkv, 128, wl.K, wl.C, wl.R, wl.W, wl.tau, wl.T_r, wl.lcap)
    sup, cnt = gpu_prefill_supports(tsa, wl, kv, dev)
    g.init(wl.q_prefill.to(dev).contiguous(), sup, cnt)

    kb = [bits(wl.k[0, i]) for i in range(wl.Hkv)]
    vb = [bits(wl.v[0, i]) for i in range(wl.Hkv)]
    qpre = bits(wl.q_prefill)
    o = orc.ReTopK(wl.Hq, 128, wl.K, wl.C, wl.R, wl.W, wl.tau, wl.T_r,
                   path_abs=1e-5, rho_abs=1e-5, topk_rel=TIE_REL)
    sup_h, cnt_h = sup.cpu().numpy(), cnt.cpu().numpy()
    for c in range(wl.C):
        p = wl.L0 - wl.C + c
        for h in range(wl.Hq):
            got = sup_h[c, h, : cnt_h[c, h]]
            if verify_prefill:
                z = orc.scores(qpre[c, h], kb[h // G][: p + 1], wl.scale)
                verdict = orc.topk_check(z, np.arange(p + 1), wl.K, got, TIE_REL)
                assert verdict in (1, 2), f"prefill support c={c} h={h} rejected"
            o.set_slot(h, c, qpre[c, h], got)

    cap = wl.R * wl.K + wl.W
    so = torch.empty((wl.Hq, wl.K), dtype=torch.int32, device=dev)
    po = torch.empty((wl.Hq,), dtype=torch.int32, device=dev)
    mo = torch.empty((wl.Hq,), dtype=torch.int32, device=dev)
    co = torch.empty((wl.Hq, cap), dtype=torch.int32, device=dev)
    lo = torch.empty((wl.Hq,), dtype=torch.float32, device=dev)
    stats = {"exact": 0, "reuse": 0, "adopt_path": 0, "adopt_cand": 0, "tie_sup": 0,
             "max_err": 0.0, "qbar_err": 0.0, "mcand": []}
    qbar_cache = g.state[: wl.Hq * wl.C * 128 * 4].view(torch.float32).view(wl.Hq, wl.C, 128)
    for t in range(steps):
        L = wl.length(t)
        q = wl.q_all[t].to(dev).contiguous()
        slot = g.counters()[1]
        out = g.step(q, kv, L, wl.scale, support_out=so, path_out=po, mcand_out=mo,
                     cand_out=co, lse_out=lo)
        torch.cuda.synchronize()
        out_h, sup_g, path_g = out.cpu().numpy(), so.cpu().numpy(), po.cpu().numpy()
        m_g, cand_g = mo.cpu().numpy(), co.cpu().numpy()
        qb = bits(wl.q_all[t])
        # the fp32 normalised queries pushed this step vs the fp64 normalisation
        qf = orc.bf16_to_f64(qb)
        qn = qf / np.linalg.norm(qf, axis=1, keepdims=True)
        pushed = qbar_cache[:, slot].double().cpu().numpy()
        stats["qbar_err"] = max(stats["qbar_err"], float(np.max(np.abs(pushed - qn))))
        for h in range(wl.Hq):
            sg = sup_g[h][sup_g[h] >= 0]
            cg = cand_g[h][: m_g[h]] if path_g[h] == 0 else None
            if path_g[h] == 0:
                assert np.all(cand_g[h][m_g[h]:] == -1)
            r = o.step_head(h, qb[h], kb[h // G][:L], vb[h // G][:L], wl.scale,
                            other_path=int(path_g[h]), other_cand=cg, other_sup=sg)
            assert r["path"] == path_g[h], f"t={t} h={h}: path {path_g[h]} vs {r['path']}"
            if r["path"] == 0:
                assert r["cand_ok"] in (1, 2), f"t={t} h={h}: candidate set differs"
                assert m_g[h] == len(r["cand"])
                assert m_g[h] <= cap
                stats["mcand"].append(int(m_g[h]))
            else:
                assert m_g[h] == L
            assert r["sup_ok"] in (1, 2), f"t={t} h={h}: support rejected"
            err = float(np.max(np.abs(out_h[h] - r["out"])))
            if check_out:
                assert err <= OUT_TOL, f"t={t} h={h}: out err {err}"
            stats["max_err"] = max(stats["max_err"], err)
            stats["exact" if r["path"] else "reuse"] += 1
            stats["adopt_path"] += r["adopt_path"]
            stats["adopt_cand"] += r["adopt_cand"]
            stats["tie_sup"] += r["sup_ok"] == 2
        o.advance()
    assert g.counters() == (steps, steps % wl.C)
    head_steps = steps * wl.Hq
    adopted = stats["adopt_path"] + stats["adopt_cand"]
    assert adopted <= max(1, head_steps // 1000), f"{adopted} adoptions in {head_steps} head-steps"
    assert stats["qbar_err"] <= 1e-6, f"normalised query error {stats['qbar_err']}"
    return stats


def test_retopk_downsized_lockstep():
    wl = make_retopk(L0=6000, steps=40, K=64, C=8, R=2, W=8, T_r=16)
    st = run_lockstep(wl, 40)
    assert st["reuse"] > 0 and st["exact"] > 0
    print("retopk downsized:", {k: v for k, v in st.items() if k != "mcand"},
          "mean M_t", np.mean(st["mcand"]))


def test_retopk_single_recall_keeps_whole_candidate_set():
    """R = 1 and W = 0: A_t is one cached support, |A_t| <= K, so S_t = A_t
    (every candidate selected; the radix is never needed)."""
    wl = make_retopk(L0=4000, steps=12, K=48, C=4, R=1, W=0, T_r=1000, tau=-2.0)
    st = run_lockstep(wl, 12)
    assert st["reuse"] > 0
    assert max(st["mcand"]) <= wl.K


def test_retopk_fallback_mix():
    """A slow-moving walk with tau high enough that the fallback fires."""
    wl = make_retopk(L0=5000, steps=30, K=48, C=6, R=3, W=5, T_r=1000, tau=0.97)
    st = run_lockstep(wl, 30)
    assert st["exact"] > wl.Hq  # more than the step-0 refresh


def test_retopk_always_exact_matches_decode():
    """tau > 1: every step takes the exact path == sparse_attn_decode, no window."""
    import top_retrieval_sparse_gb300 as tsa
    wl = make_retopk(L0=3000, steps=4, K=40, C=4, R=2, W=4, tau=1.5)
    dev = "cuda"
    kv = tsa.kv_contiguous(wl.k.to(dev), wl.v.to(dev))
    g = tsa.ReTopK(wl.Hq, wl.Hkv, 128, wl.K, wl.C, wl.R, wl.W, wl.tau, wl.T_r, wl.lcap)
    sup, cnt = gpu_prefill_supports(tsa, wl, kv, dev)
    g.init(wl.q_prefill.to(dev).contiguous(), sup, cnt)
    for t in range(wl.steps):
        L = wl.length(t)
        q = wl.q_all[t].to(dev).contiguous()
        so = torch.empty((wl.Hq, wl.K), dtype=torch.int32, device=dev)
        out = g.step(q, kv, L, wl.scale, support_out=so)
        idx = torch.empty((1, wl.Hq, wl.K), dtype=torch.int32, device=dev)
        ref, _, _, _ = tsa.sparse_attn_decode(q[None], kv, torch.tensor([L], dtype=torch.int32,
                                              device=dev), wl.K, 0, 0, wl.scale, topk_idx=idx)
        torch.cuda.synchronize()
        for h in range(wl.Hq):
            assert set(so[h].tolist()) == set(idx[0, h].tolist())
        assert torch.max(torch.abs(out - ref[0])).item() < 1e-5


def test_retopk_paged_cache_matches_contiguous():
    """The same stream over a paged copy of the cache (16-token pages in a
    seeded random order): every step's paths, candidate sets, supports and
    outputs equal those of the contiguous run (the kernels read the same rows,
    only through the page table; exact steps included: T_r = 8)."""
    import top_retrieval_sparse_gb300 as tsa
    wl = make_retopk(L0=5000, steps=20, K=48, C=6, R=3, W=5, T_r=8)
    dev = "cuda"
    k, v = wl.k.to(dev), wl.v.to(dev)
    ps = 16
    npg = wl.lcap // ps
    perm = torch.randperm(npg, generator=torch.Generator().manual_seed(7)).to(torch.int32)
    kp = torch.zeros((npg, wl.Hkv, ps, wl.d), dtype=torch.bfloat16, device=dev)
    vp = torch.zeros_like(kp)
    kp[perm.long().to(dev)] = k[0].reshape(wl.Hkv, npg, ps, wl.d).transpose(0, 1)
    vp[perm.long().to(dev)] = v[0].reshape(wl.Hkv, npg, ps, wl.d).transpose(0, 1)
    kvc = tsa.kv_contiguous(k, v)
    kvp = tsa.kv_paged(kp, vp, perm[None].to(dev).contiguous())
    sup, cnt = gpu_prefill_supports(tsa, wl, kvc, dev)
    runs = []
    for kv in (kvc, kvp):
        g = tsa.ReTopK(wl.Hq, wl.Hkv, 128, wl.K, wl.C, wl.R, wl.W, wl.tau, wl.T_r, wl.lcap)
        g.init(wl.q_prefill.to(dev).contiguous(), sup, cnt)
        rec = []
        cap = wl.R * wl.K + wl.W
        for t in range(wl.steps):
            so = torch.empty((wl.Hq, wl.K), dtype=torch.int32, device=dev)
            po = torch.empty((wl.Hq,), dtype=torch.int32, device=dev)
            mo = torch.empty((wl.Hq,), dtype=torch.int32, device=dev)
            co = torch.empty((wl.Hq, cap), dtype=torch.int32, device=dev)
            out = g.step(wl.q_all[t].to(dev).contiguous(), kv, wl.length(t), wl.scale,
                         support_out=so, path_out=po, mcand_out=mo, cand_out=co)
            rec.append((out.clone(), so, po, mo, co))
        torch.cuda.synchronize()
        runs.append(rec)
    n_exact = n_reuse = 0
    for t, (a, b) in enumerate(zip(*runs)):
        assert torch.equal(a[2], b[2]), f"t={t}: paths differ"
        assert torch.equal(a[3], b[3]), f"t={t}: candidate counts differ"
        assert torch.equal(a[4], b[4]), f"t={t}: candidate sets differ"
        for h in range(wl.Hq):
            assert set(a[1][h].tolist()) == set(b[1][h].tolist()), f"t={t} h={h}: supports"
        assert torch.max(torch.abs(a[0] - b[0])).item() < 1e-5, f"t={t}: outputs"
        n_exact += int(a[2].sum())
        n_reuse += int((a[2] == 0).sum())
    assert n_exact >= wl.Hq and n_reuse > 0


@pytest.mark.slow
def test_retopk_full_config_lockstep():
    wl = make_retopk()  # Qwen2.5-7B geometry, 64K, C=32 R=4 K=512 W=32 tau=0.85 T_r=128
    st = run_lockstep(wl, wl.steps)
    print("retopk64k:", {k: v for k, v in st.items() if k != "mcand"},
          "mean M_t", float(np.mean(st["mcand"])), "max M_t", max(st["mcand"]))


@pytest.mark.slow
def test_retopk_1m_context_k1024_first_steps():
    """The long-context setting: 1M keys, K = 1024 (a candidate bitmap of
    128 KiB per head), the first steps of the stream in lockstep: step 0
    refreshes (every head exact over all 1M keys), the next ones mostly reuse.
    The prefill supports come from sparse_attn_decode, whose exactness the
    decode tests cover; they are fed to the oracle as they are."""
    wl = make_retopk("retopk1m", device="cuda", steps=6)
    st = run_lockstep(wl, 6, verify_prefill=False)
    assert st["exact"] >= wl.Hq and st["reuse"] > 0
    print("retopk1m:", {k: v for k, v in st.items() if k != "mcand"},
          "mean M_t", float(np.mean(st["mcand"])), "max M_t", max(st["mcand"]))


@pytest.mark.slow
def test_retopk_4m_context_first_steps():
    """Beyond the 1.5 M positions one CTA's shared memory holds as a bitmap:
    4M keys, K = 1024, where the selector keeps the candidate bitmap in the
    workspace (cleared word by word as the compaction reads it) and only its
    second level in shared memory.  The first steps in lockstep: step 0
    refreshes (every head exact over 4M keys), the next ones mostly reuse, and
    every reuse head's A_t must equal the oracle's union bit for bit."""
    wl = make_retopk("retopk4m", device="cuda", steps=6)
    st = run_lockstep(wl, 6, verify_prefill=False)
    assert st["exact"] >= wl.Hq and st["reuse"] > 0
    print("retopk4m:", {k: v for k, v in st.items() if k != "mcand"},
          "mean M_t", float(np.mean(st["mcand"])), "max M_t", max(st["mcand"]))


@pytest.mark.parametrize("paged", [False, True])
def test_prefill_supports_match_oracle(paged):
    """retopk_prefill_supports: every (prefill query, head)'s support is the
    oracle's exact top-K over its causal prefix (near-tie rule), counts are
    min(K, p + 1), padding is -1; a paged copy of the cache gives the same."""
    import top_retrieval_sparse_gb300 as tsa
    wl = make_retopk(L0=6000, steps=1, K=64, C=8, R=2, W=8)
    dev = "cuda"
    k, v = wl.k.to(dev), wl.v.to(dev)
    if paged:
        ps = 16
        npg = wl.lcap // ps
        perm = torch.randperm(npg, generator=torch.Generator().manual_seed(3)).to(torch.int32)
        kp = torch.zeros((npg, wl.Hkv, ps, wl.d), dtype=torch.bfloat16, device=dev)
        vp = torch.zeros_like(kp)
        kp[perm.long().to(dev)] = k[0].reshape(wl.Hkv, npg, ps, wl.d).transpose(0, 1)
        vp[perm.long().to(dev)] = v[0].reshape(wl.Hkv, npg, ps, wl.d).transpose(0, 1)
        kv = tsa.kv_paged(kp, vp, perm[None].to(dev).contiguous())
    else:
        kv = tsa.kv_contiguous(k, v)
    sup, cnt = gpu_prefill_supports(tsa, wl, kv, dev)
    torch.cuda.synchronize()
    sup, cnt = sup.cpu().numpy(), cnt.cpu().numpy()
    G = wl.Hq // wl.Hkv
    kb = [bits(wl.k[0, i]) for i in range(wl.Hkv)]
    qpre = bits(wl.q_prefill)
    for c in range(wl.C):
        p = wl.L0 - wl.C + c
        for h in range(wl.Hq):
            assert cnt[c, h] == min(wl.K, p + 1)
            got = sup[c, h, : cnt[c, h]]
            assert np.all(sup[c, h, cnt[c, h]:] == -1)
            z = orc.scores(qpre[c, h], kb[h // G][: p + 1], wl.scale)
            assert orc.topk_check(z, np.arange(p + 1), wl.K, got, TIE_REL) in (1, 2), (c, h)


def test_prefill_supports_equal_per_query_decode_and_repeat():
    """The one-call supports equal C separate decode calls (window 0, length
    p + 1), on a fresh workspace and again on the reused one (whose emission
    keys now come from the first call)."""
    import top_retrieval_sparse_gb300 as tsa
    wl = make_retopk(L0=20_000, steps=1, K=128, C=12, R=2, W=8)
    dev = "cuda"
    kv = tsa.kv_contiguous(wl.k.to(dev), wl.v.to(dev))
    ref, rcnt = decode_prefill_supports(tsa, wl, kv, dev)
    n = tsa.prefill_workspace_size(wl.C, wl.Hq, wl.Hkv, wl.d, kv.l_cap, wl.K)
    ws = torch.zeros(n, dtype=torch.uint8, device=dev)
    q = wl.q_prefill.to(dev).contiguous()
    for _ in range(2):
        sup, cnt = tsa.prefill_supports(q, kv, wl.L0, wl.K, wl.scale, workspace=ws)
        torch.cuda.synchronize()
        assert torch.equal(cnt, rcnt)
        for c in range(wl.C):
            for h in range(wl.Hq):
                assert set(sup[c, h].tolist()) == set(ref[c, h].tolist()), (c, h)
    assert tsa.workspace_status(ws) == 0


def test_checkpoint_resume_in_a_fresh_handle():
    """The ReTopK state is the caller's memory plus two host counters: a copy
    of both taken mid-stream, restored into a new handle over new memory (and a
    new, zeroed workspace), continues exactly as the uninterrupted run --
    same paths, candidate sets and supports, outputs within 1e-5."""
    import top_retrieval_sparse_gb300 as tsa
    wl = make_retopk(L0=5000, steps=12, K=48, C=6, R=3, W=5, T_r=5)
    dev = "cuda"
    kv = tsa.kv_contiguous(wl.k.to(dev), wl.v.to(dev))
    sup, cnt = gpu_prefill_supports(tsa, wl, kv, dev)
    a = tsa.ReTopK(wl.Hq, wl.Hkv, 128, wl.K, wl.C, wl.R, wl.W, wl.tau, wl.T_r, wl.lcap)
    a.init(wl.q_prefill.to(dev).contiguous(), sup, cnt)
    cap = wl.R * wl.K + wl.W

    def step(g, t):
        so = torch.empty((wl.Hq, wl.K), dtype=torch.int32, device=dev)
        po = torch.empty((wl.Hq,), dtype=torch.int32, device=dev)
        co = torch.empty((wl.Hq, cap), dtype=torch.int32, device=dev)
        out = g.step(wl.q_all[t].to(dev).contiguous(), kv, wl.length(t), wl.scale,
                     support_out=so, path_out=po, cand_out=co)
        torch.cuda.synchronize()
        return out.cpu(), so.cpu(), po.cpu(), co.cpu()

    for t in range(6):
        step(a, t)
    saved_state, saved_counters = a.state.clone(), a.counters()
    b = tsa.ReTopK(wl.Hq, wl.Hkv, 128, wl.K, wl.C, wl.R, wl.W, wl.tau, wl.T_r, wl.lcap)
    b.state.copy_(saved_state)
    b.set_counters(*saved_counters)
    n_exact = 0
    for t in range(6, 12):
        ra, rb = step(a, t), step(b, t)
        assert torch.equal(ra[2], rb[2]), f"t={t}: paths"
        assert torch.equal(ra[3], rb[3]), f"t={t}: candidate sets"
        for h in range(wl.Hq):
            assert set(ra[1][h].tolist()) == set(rb[1][h].tolist()), (t, h)
        assert torch.max(torch.abs(ra[0] - rb[0])).item() < 1e-5
        n_exact += int(ra[2].sum())
    assert a.counters() == b.counters() == (12, 12 % wl.C)
    assert n_exact >= wl.Hq  # the resumed part crosses a refresh step (t = 10)
