"""Failure detection on the GPU without a GPU fault.

Every wait inside the kernels is bounded.  tsa_inject_scan_stall makes the
next call's key scan use a short limit and makes the scan's first CTA withhold
one tile copy, so that CTA's bounded waits expire: the kernel gives up and
flags a sticky status word, the finish kernel writes NaN outputs, and the
host learns of it through tsa_workspace_status (TSA_ERR_TIMEOUT).  Nothing
traps or faults; the context stays usable and the next call is exact.
"""
import numpy as np
import pytest
import torch

import top_retrieval_sparse_gb300 as tsa
from helpers import check_head, gpu_decode
from workloads.gen import make_decode, make_retopk

pytestmark = pytest.mark.gpu

TIMEOUT, DEVICE_CHECK = -6, -5
STALL_NS = 2_000_000  # 2 ms


def _decode_with(wl, ws, kv, lens, K=None):
    K = wl.K if K is None else K
    q = wl.q(0).cuda().contiguous()
    B, Hq, d = q.shape
    lse = torch.empty((B, Hq), dtype=torch.float32, device="cuda")
    idx = torch.empty((B, Hq, K), dtype=torch.int32, device="cuda")
    sc = torch.empty((B, Hq, K), dtype=torch.float32, device="cuda")
    out, _, _, _ = tsa.sparse_attn_decode(q, kv, lens, K, wl.n_init, wl.n_recent, wl.scale,
                                          lse_out=lse, topk_idx=idx, topk_score=sc,
                                          workspace=ws)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy(), sc.cpu().numpy()


def _setup(name="tiny"):
    wl = make_decode(name)
    kv = tsa.kv_contiguous(wl.k.cuda(), wl.v.cuda())
    lens = torch.tensor(wl.lens(0), dtype=torch.int32, device="cuda")
    n = tsa.decode_workspace_size(wl.B, wl.Hq, wl.Hkv, wl.d, kv.l_cap, wl.K, wl.n_init,
                                  wl.n_recent)
    ws = torch.zeros(n, dtype=torch.uint8, device="cuda")
    return wl, kv, lens, ws


def _check_exact(wl, res):
    out, lse, idx, sc = res
    for b in range(wl.B):
        for h in range(wl.Hq):
            check_head(wl, 0, b, h, out[b, h], lse[b, h], idx[b, h], sc[b, h])


@pytest.mark.parametrize("name", ["tiny", "llama128k"])
def test_scan_timeout_is_reported_and_the_next_call_is_exact(name):
    wl, kv, lens, ws = _setup(name)
    _check_exact(wl, _decode_with(wl, ws, kv, lens))
    assert tsa.workspace_status(ws) == 0

    tsa.inject_scan_stall(STALL_NS)
    out, lse, idx, sc = _decode_with(wl, ws, kv, lens)
    assert np.isnan(out).all() and np.isnan(lse).all() and np.isnan(sc).all()
    assert (idx == -1).all()
    # sticky: a normal call before the status is read still reports NaN
    out2, _, _, _ = _decode_with(wl, ws, kv, lens)
    assert np.isnan(out2).all()
    assert tsa.workspace_status(ws, clear=True) == TIMEOUT
    assert "wait expired" in tsa.lib().tsa_last_error().decode()
    # cleared: the same workspace (not re-zeroed) gives the exact result again
    _check_exact(wl, _decode_with(wl, ws, kv, lens))
    assert tsa.workspace_status(ws) == 0
    # the device never faulted: an unrelated torch op still runs
    assert float(torch.ones(4, device="cuda").sum()) == 4.0


def test_length_beyond_the_cache_is_flagged_and_clamped():
    wl, kv, lens, ws = _setup("tiny")
    bad = torch.tensor([kv.l_cap + 100], dtype=torch.int32, device="cuda")
    out, lse, idx, sc = _decode_with(wl, ws, kv, bad)
    assert np.isfinite(out).all()
    assert tsa.workspace_status(ws) == DEVICE_CHECK
    assert tsa.workspace_status(ws) == 0   # cleared by the first read
    # the clamped call computed the step at L = l_cap
    full = torch.tensor([kv.l_cap], dtype=torch.int32, device="cuda")
    ref = _decode_with(wl, ws, kv, full)
    # same set, same output up to the summation order (pair lists fill by atomics)
    np.testing.assert_allclose(out, ref[0], rtol=0, atol=1e-5)
    for h in range(wl.Hq):
        assert set(idx[0, h].tolist()) == set(ref[2][0, h].tolist())


def test_retopk_step_timeout_keeps_the_fifo_entry():
    """A stalled ReTopK step outputs NaN and does not rewrite its FIFO entry;
    restoring the counters and redoing the step gives the uninterrupted
    run's result."""
    from test_parity_retopk import gpu_prefill_supports
    wl = make_retopk(L0=3000, steps=4, K=40, C=4, R=2, W=4, T_r=2)
    kv = tsa.kv_contiguous(wl.k.cuda(), wl.v.cuda())
    sup, cnt = gpu_prefill_supports(tsa, wl, kv, "cuda")

    def fresh():
        g = tsa.ReTopK(wl.Hq, wl.Hkv, 128, wl.K, wl.C, wl.R, wl.W, wl.tau, wl.T_r, wl.lcap)
        g.init(wl.q_prefill.cuda().contiguous(), sup, cnt)
        return g

    def step(g, t):
        so = torch.empty((wl.Hq, wl.K), dtype=torch.int32, device="cuda")
        out = g.step(wl.q_all[t].cuda().contiguous(), kv, wl.length(t), wl.scale,
                     support_out=so)
        torch.cuda.synchronize()
        return out.cpu().numpy(), so.cpu().numpy()

    ref = fresh()
    want = [step(ref, t) for t in range(wl.steps)]
    g = fresh()
    step(g, 0)
    before = g.state.clone()
    t, head = g.counters()
    tsa.inject_scan_stall(STALL_NS)
    out, _ = step(g, 1)              # T_r = 2: step 1 reuses, but step 2 would refresh;
    assert tsa.workspace_status(g.workspace, clear=True) in (TIMEOUT, 0)
    if np.isnan(out).all():          # the scan ran (some head took the exact path)
        assert torch.equal(g.state, before)
    g.state.copy_(before)
    g.set_counters(t, head)
    for s in range(1, wl.steps):
        o, so = step(g, s)
        np.testing.assert_allclose(o, want[s][0], rtol=0, atol=1e-5)
        for h in range(wl.Hq):
            assert set(so[h].tolist()) == set(want[s][1][h].tolist())
    # a refresh step (every head exact, the scan always runs) under a stall
    g2 = fresh()
    tsa.inject_scan_stall(STALL_NS)
    out, _ = step(g2, 0)
    assert np.isnan(out).all()
    assert tsa.workspace_status(g2.workspace, clear=True) == TIMEOUT
