"""Shared test helpers: run the CUDA path through the binding and compare it
with the fp64 oracle under the checking rules.

Rules (stated for this path): top-K sets are bit-exact, except where the fp64
K-th and (K+1)-th logits differ by less than 1e-6 relative, in which case every
chosen position must score at least z_(K) - 1e-6|z_(K)|; outputs are within
max-abs 2e-3 of the fp64 oracle evaluated on the returned set.
"""
from __future__ import annotations

import numpy as np
import torch

import oracle as orc
from workloads.gen import bits

OUT_TOL = 2e-3      # max-abs on the attention output
LSE_TOL = 2e-3      # abs on the log-sum-exp
TIE_REL = 1e-6      # near-tie margin for top-K sets


def gpu_decode(wl, step, device="cuda", paged=None, K=None):
    import top_retrieval_sparse_gb300 as tsa
    K = wl.K if K is None else K
    use_pages = (wl.page_table is not None) if paged is None else paged
    if use_pages:
        kv = tsa.kv_paged(wl.k_pages.to(device), wl.v_pages.to(device),
                          wl.page_table.to(device))
    else:
        kv = tsa.kv_contiguous(wl.k.to(device), wl.v.to(device))
    q = wl.q(step).to(device).contiguous()
    lens = torch.tensor(wl.lens(step), dtype=torch.int32, device=device)
    B, Hq, d = q.shape
    lse = torch.empty((B, Hq), dtype=torch.float32, device=device)
    idx = torch.empty((B, Hq, max(K, 1)), dtype=torch.int32, device=device)
    sc = torch.empty((B, Hq, max(K, 1)), dtype=torch.float32, device=device)
    out, _, _, _ = tsa.sparse_attn_decode(q, kv, lens, K, wl.n_init, wl.n_recent, wl.scale,
                                          lse_out=lse, topk_idx=idx if K else None,
                                          topk_score=sc if K else None)
    torch.cuda.synchronize()
    return out.cpu().numpy(), lse.cpu().numpy(), idx.cpu().numpy()[..., :K], sc.cpu().numpy()[..., :K]


def check_head(wl, step, b, h, g_out, g_lse, g_idx, g_sc=None, K=None):
    """Compare one (sequence, head) of a GPU decode step with the oracle.
    Returns a dict of diagnostics; raises AssertionError on a rule violation."""
    K = wl.K if K is None else K
    G = wl.Hq // wl.Hkv
    L = wl.lens(step)[b]
    kb = bits(wl.k[b, h // G, :L])
    vb = bits(wl.v[b, h // G, :L])
    qb = bits(wl.q(step)[b, h])
    r = orc.decode_head(qb, kb, vb, K, wl.n_init, wl.n_recent, wl.scale)
    z = r["z"]
    pool = np.array([i for i in range(L) if not (i < wl.n_init or i >= L - wl.n_recent)],
                    np.int64)
    got = g_idx[g_idx >= 0].astype(np.int64)
    assert np.all(g_idx[len(got):] == -1), "padding must follow the selected positions"
    verdict = orc.topk_check(z, pool, K, got, TIE_REL)
    assert verdict in (1, 2), f"b={b} h={h}: top-K set rejected (|got|={len(got)})"
    if verdict == 1:
        ref_out, ref_lse = r["out"], r["lse"]
    else:
        ref_out, ref_lse = orc.decode_eval_set(z, vb, wl.n_init, wl.n_recent, got)
    err = float(np.max(np.abs(g_out - ref_out))) if len(ref_out) else 0.0
    assert err <= OUT_TOL, f"b={b} h={h}: out max-abs err {err}"
    if np.isfinite(ref_lse):
        assert abs(g_lse - ref_lse) <= LSE_TOL, f"b={b} h={h}: lse {g_lse} vs {ref_lse}"
    else:
        assert g_lse == -np.inf
    zerr = 0.0
    if g_sc is not None and len(got):
        zerr = float(np.max(np.abs(g_sc[: len(got)] - z[got]) / np.maximum(np.abs(z[got]), 1e-30)))
    return {"verdict": verdict, "err": err, "zrel": zerr}
