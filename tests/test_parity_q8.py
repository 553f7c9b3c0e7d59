"""GPU parity of the int8 key codes and of the quantised decode.

Codes: bit-exact against the oracle's quantiser (scales bit-exact, errors an
upper bound within 2^-21 of the oracle's exact ones), fitted and appended,
contiguous and paged.  Decode: the selected set and its logits equal those of
sparse_attn_decode bit for bit, the outputs agree within 1e-5 (fp32 sums in
another order) and the oracle's checking rules hold; covered are ragged
lengths, windows that cover the cache, K = 0 and K >= |P|, GQA groups that
leave columns unused, a paged batch, a decode stream that appends one key a
step (n_new = 1), saturating appends and emission keys that are far off (the
exact fallback).
"""
import numpy as np
import pytest
import torch

import oracle as orc
from helpers import check_head
from workloads.gen import bits, make_decode

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _kv(tsa, wl, paged):
    if paged:
        return tsa.kv_paged(wl.k_pages.to(DEV), wl.v_pages.to(DEV), wl.page_table.to(DEV))
    return tsa.kv_contiguous(wl.k.to(DEV), wl.v.to(DEV))


def _code_rows(kc, wl, b, g, L, paged):
    """Codes of rows [0, L) of (b, g) as [L, 128] uint8 (host)."""
    c = kc.codes.cpu()
    if not paged:
        return c[b, g, :L].numpy()
    ps = wl.k_pages.shape[2]
    pt = wl.page_table[b].tolist()
    rows = [c[pt[i // ps], g, i % ps] for i in range(L)]
    return torch.stack(rows).numpy() if rows else np.zeros((0, 128), np.uint8)


def _check_codes(kc, wl, lens, paged, ref=None):
    """Compare every (sequence, KV head) with the oracle (fit over lens)."""
    sc, er = kc.scale.cpu().numpy(), kc.err.cpu().numpy()
    out = {}
    for b in range(wl.B):
        for g in range(wl.Hkv):
            L = lens[b]
            kb = bits(wl.k[b, g, :L])
            s, codes, err = orc.q8_fit(kb) if ref is None else ref[(b, g)]
            np.testing.assert_array_equal(sc[b, g], s)
            np.testing.assert_array_equal(_code_rows(kc, wl, b, g, L, paged), codes)
            assert np.all(er[b, g] >= err), "the stored error must bound the exact one"
            assert np.all(er[b, g] <= err * (1 + 2.0 ** -21) + 1e-30)
            out[(b, g)] = (s, codes, err)
    return out


@pytest.mark.parametrize("paged", [False, True])
def test_codes_fit_and_append_match_oracle(paged):
    import top_retrieval_sparse_gb300 as tsa
    wl = make_decode("yi_paged", L0=3000, steps=4, B=3, K=100)
    kv = _kv(tsa, wl, paged)
    kc = tsa.KeyCodes(kv, B=wl.B)
    L0 = [l - 1 for l in wl.lens(0)]  # the codes start one row short
    tsa.quantize_keys(kv, kc, torch.tensor(L0, dtype=torch.int32, device=DEV), fit=True)
    torch.cuda.synchronize()
    ref = _check_codes(kc, wl, L0, paged)
    # append 3 rows per sequence, one of them far outside the fitted range
    L1 = [l + 3 for l in L0]
    for b in range(wl.B):
        wl.k[b, :, L1[b] - 2] = (wl.k[b, :, L1[b] - 2].float() * 6.0).to(torch.bfloat16)
    kv = _kv(tsa, _refresh_pages(wl) if paged else wl, paged)
    tsa.quantize_keys(kv, kc, torch.tensor(L1, dtype=torch.int32, device=DEV), fit=False,
                      n_tail=3)
    torch.cuda.synchronize()
    for b in range(wl.B):
        for g in range(wl.Hkv):
            s, codes, err = ref[(b, g)]
            c2, e2 = orc.q8_append(bits(wl.k[b, g, L0[b]:L1[b]]), s, err)
            ref[(b, g)] = (s, np.concatenate([codes, c2]), e2)
    _check_codes(kc, wl, L1, paged, ref)
    assert np.any(kc.err.cpu().numpy() > np.stack(
        [np.stack([orc.q8_fit(bits(wl.k[b, g, :L0[b]]))[2] for g in range(wl.Hkv)])
         for b in range(wl.B)]))  # the saturated row raised the bound


def _refresh_pages(wl):
    """Rewrite the page pool from wl.k (after a test edited wl.k)."""
    ps = wl.k_pages.shape[2]
    for b in range(wl.B):
        for i, p in enumerate(wl.page_table[b].tolist()):
            r0 = i * ps
            if p < 0 or r0 >= wl.lcap:
                continue
            m = min(ps, wl.lcap - r0)
            wl.k_pages[p, :, :m] = wl.k[b, :, r0:r0 + m].to(wl.k_pages.device)
    return wl


def _decode_both(wl, step, kc=None, n_new=0, K=None, paged=False, ws=None, ws8=None):
    """Plain and quantised decode of one step; returns both results (host)."""
    import top_retrieval_sparse_gb300 as tsa
    K = wl.K if K is None else K
    kv = _kv(tsa, wl, paged)
    q = wl.q(step).to(DEV).contiguous()
    lens = torch.tensor(wl.lens(step), dtype=torch.int32, device=DEV)
    if kc is None:
        kc = tsa.KeyCodes(kv, B=wl.B)
        tsa.quantize_keys(kv, kc, lens, fit=True)
    res = []
    for quant in (False, True):
        lse = torch.empty((wl.B, wl.Hq), device=DEV)
        idx = torch.empty((wl.B, wl.Hq, max(K, 1)), dtype=torch.int32, device=DEV)
        sc = torch.empty((wl.B, wl.Hq, max(K, 1)), device=DEV)
        kw = dict(lse_out=lse, topk_idx=idx if K else None, topk_score=sc if K else None)
        if quant:
            out, _, _, _ = tsa.sparse_attn_decode_q8(q, kv, kc, lens, K, wl.n_init,
                                                     wl.n_recent, n_new=n_new, scale=wl.scale,
                                                     workspace=ws8, **kw)
        else:
            out, _, _, _ = tsa.sparse_attn_decode(q, kv, lens, K, wl.n_init, wl.n_recent,
                                                  wl.scale, workspace=ws, **kw)
        torch.cuda.synchronize()
        res.append((out.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()[..., :K],
                    sc.cpu().numpy()[..., :K]))
    return res


def _same_selection(a, b, wl):
    (oa, la, ia, sa), (ob, lb, ib, sb) = a, b
    for bb in range(wl.B):
        for h in range(wl.Hq):
            pa = sorted(zip(ia[bb, h].tolist(), sa[bb, h].view(np.uint32).tolist()))
            pb = sorted(zip(ib[bb, h].tolist(), sb[bb, h].view(np.uint32).tolist()))
            assert pa == pb, f"b={bb} h={h}: selected (position, logit bits) differ"
    np.testing.assert_allclose(ob, oa, atol=1e-5, rtol=0)
    fin = np.isfinite(la)
    assert np.array_equal(fin, np.isfinite(lb))
    np.testing.assert_allclose(lb[fin], la[fin], atol=1e-5, rtol=0)


def _oracle_check(wl, step, res, heads=None, K=None):
    o, l, i, s = res
    for b in range(wl.B):
        for h in (range(wl.Hq) if heads is None else heads):
            check_head(wl, step, b, h, o[b, h], l[b, h], i[b, h], s[b, h] if s.size else None,
                       K=K)


def test_tiny_matches_plain_and_oracle():
    wl = make_decode("tiny", steps=2)
    for t in range(2):
        a, b = _decode_both(wl, t)
        _same_selection(a, b, wl)
        _oracle_check(wl, t, b)


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (12, 4), (28, 4), (32, 8)])
def test_group_sizes_ragged(Hq, Hkv):
    wl = make_decode("llama128k", L0=9001 + 5 * Hq, steps=1, K=300, Hq=Hq, Hkv=Hkv,
                     n_init=16, n_recent=40)
    a, b = _decode_both(wl, 0)
    _same_selection(a, b, wl)
    _oracle_check(wl, 0, b, heads=range(0, Hq, 3))


def test_llama_geometry_downsized():
    """K = 2048 with the 128 + 512 window; several 512-row code tiles per CTA."""
    wl = make_decode("llama128k", L0=40_001, steps=2)
    for t in range(2):
        a, b = _decode_both(wl, t)
        _same_selection(a, b, wl)
    _oracle_check(wl, 1, b, heads=range(0, wl.Hq, 5))


def test_paged_batch():
    wl = make_decode("yi_paged", L0=6000, steps=1, B=5, K=300)
    a, b = _decode_both(wl, 0, paged=True)
    _same_selection(a, b, wl)
    _oracle_check(wl, 0, b, heads=range(0, wl.Hq, 4))


@pytest.mark.parametrize("K", [0, 1, 64, 5000, 50000])
def test_K_edge_cases(K):
    wl = make_decode("tiny", L0=4500, steps=1)
    a, b = _decode_both(wl, 0, K=K)
    _same_selection(a, b, wl)
    _oracle_check(wl, 0, b, K=K)


def test_window_covers_cache_and_tiny_lengths():
    for L0 in (0, 1, 3, 60, 67, 130, 600):
        wl = make_decode("tiny", L0=L0, steps=1, K=16)
        a, b = _decode_both(wl, 0)
        _same_selection(a, b, wl)
        _oracle_check(wl, 0, b)


def test_stream_appends_one_key_a_step():
    """Codes fitted once; every call codes the step's newest key itself
    (n_new = 1) and must select exactly what the plain path selects."""
    import top_retrieval_sparse_gb300 as tsa
    wl = make_decode("llama128k", L0=20_000, steps=6, K=512, n_init=16, n_recent=64)
    kv = _kv(tsa, wl, False)
    kc = tsa.KeyCodes(kv, B=wl.B)
    first = torch.tensor([l - 1 for l in wl.lens(0)], dtype=torch.int32, device=DEV)
    tsa.quantize_keys(kv, kc, first, fit=True)
    ws = torch.zeros(tsa.decode_workspace_size(1, wl.Hq, wl.Hkv, 128, wl.lcap, wl.K,
                                               wl.n_init, wl.n_recent), dtype=torch.uint8,
                     device=DEV)
    ws8 = torch.zeros(tsa.decode_q8_workspace_size(1, wl.Hq, wl.Hkv, 128, wl.lcap, wl.K,
                                                   wl.n_init, wl.n_recent), dtype=torch.uint8,
                      device=DEV)
    for t in range(wl.steps):
        a, b = _decode_both(wl, t, kc=kc, n_new=1, ws=ws, ws8=ws8)
        _same_selection(a, b, wl)
    _oracle_check(wl, wl.steps - 1, b, heads=range(0, wl.Hq, 7))
    # the appended rows' codes are the oracle's
    L = wl.lens(wl.steps - 1)[0]
    for g in range(wl.Hkv):
        s, c0, e0 = orc.q8_fit(bits(wl.k[0, g, :L - wl.steps]))
        c1, e1 = orc.q8_append(bits(wl.k[0, g, L - wl.steps:L]), s, e0)
        np.testing.assert_array_equal(kc.codes[0, g, :L].cpu().numpy(), np.concatenate([c0, c1]))


def test_saturating_appends_stay_exact():
    """Appended keys 8x outside the fitted range saturate: the error bound
    grows (so does the shortlist) and the selection stays exact."""
    import top_retrieval_sparse_gb300 as tsa
    wl = make_decode("tiny", L0=8000, steps=1, K=200)
    L = wl.lens(0)[0]
    kv = _kv(tsa, wl, False)
    kc = tsa.KeyCodes(kv, B=1)
    tsa.quantize_keys(kv, kc, torch.tensor([L - 40], dtype=torch.int32, device=DEV), fit=True)
    wl.k[0, :, L - 40:L] = (wl.k[0, :, L - 40:L].float() * 8.0).to(torch.bfloat16)
    a, b = _decode_both(wl, 0, kc=kc, n_new=40)
    _same_selection(a, b, wl)
    _oracle_check(wl, 0, b)


def test_emission_key_far_off_takes_exact_fallback():
    """A q8 workspace carried across workloads whose logits differ 20x: the
    stored emission key is far too high (fewer than K positions kept: the
    finish rescans the head's bf16 keys) or far too low (many pairs)."""
    import top_retrieval_sparse_gb300 as tsa
    big = make_decode("tiny", L0=30_000, steps=1, K=300)
    small = make_decode("tiny", L0=30_000, steps=1, K=300)
    small.q_all[:] = (small.q_all.float() * 0.05).to(torch.bfloat16)
    n8 = tsa.decode_q8_workspace_size(1, big.Hq, big.Hkv, 128, big.lcap, big.K, big.n_init,
                                      big.n_recent)
    ws8 = torch.zeros((n8,), dtype=torch.uint8, device=DEV)
    for wl in (big, big, small, big, small, small):
        a, b = _decode_both(wl, 0, ws8=ws8)
        _same_selection(a, b, wl)
        _oracle_check(wl, 0, b)


def test_zero_scale_channels_and_constant_keys():
    """Channels that are zero in every key (scale 0) and keys that all tie."""
    wl = make_decode("tiny", L0=3000, steps=1, K=100)
    wl.k[:, :, :, ::3] = 0
    a, b = _decode_both(wl, 0)
    _same_selection(a, b, wl)
    _oracle_check(wl, 0, b)
    wl.k[:] = wl.k[:, :, :1, :]
    a, b = _decode_both(wl, 0)
    _same_selection(a, b, wl)


@pytest.mark.slow
def test_full_llama128k_sampled_heads():
    """The benchmark's workload (128K, K = 2048, 32 heads) at full size."""
    wl = make_decode("llama128k", steps=2)
    for t in range(2):
        a, b = _decode_both(wl, t)
        _same_selection(a, b, wl)
    _oracle_check(wl, 1, b, heads=(0, 13, 31))
