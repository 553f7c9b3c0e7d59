"""Seeded synthetic KV caches and query streams for decode-step top-K attention.

The pages measure on real models and datasets (infinity-Bench, RULER,
needle-in-a-haystack, PG19, LongBench); these synthetic inputs stand in for
them with the head geometries the pages use (Llama-3-8B 32/8, Yi-9B 32/4,
Qwen2.5-7B 28/4, head dim 128) and a built-in query/key distribution gap
(RetrievalAttention, section 2 "Why conventional ANNS fails": queries and
keys come from different projections; Figure 3b).

Recipe (every draw from a torch.Generator seeded per component):
  mu              fixed N(0, I) draw rescaled to norm 3 (the key offset)
  ordinary key    k = mu + sigma * xi, xi ~ N(0, I); sigma = 1 ("iid"
                  family) or per-channel sigma_j ~ U[0.5, 2] ("proj", "walk")
  value           v ~ N(0, I)
  head direction  u_h ~ N(0, I) ("iid") or u_h = P x_h with P a fixed
                  128x128 N(0, 1/d) matrix and x_h ~ N(0, I) ("proj")
  step query      q = u_h + 0.3 xi ("iid") or u_h + 0.3 P xi ("proj")
  planted key     k = 0.5 u_h + N(0, 0.1^2 I) at positions drawn uniformly
                  without replacement from [0, L0) for query head h, written
                  into KV head h // G; a later head overwrites an earlier one
  walk query      ("walk", the ReTopK stream) per head a normalised AR(1)
                  walk qbar' = normalise(0.97 qbar + sqrt(1-0.97^2) xi/sqrt(d))
                  scaled to norm sqrt(d); the C walk steps before decode are
                  the prefill queries
  decode steps    every step appends one ordinary token before attending,
                  so step t sees L0 + t + 1 keys; all appended rows are drawn
                  up front (rows past the current length are never read)

Tensors are produced in float32 and rounded to bf16 last.
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field
from typing import Optional

import torch

CONFIGS = {
    # 1: tiny exact top-K decode
    "tiny": dict(B=1, Hq=4, Hkv=1, d=128, L0=4096, steps=8, K=64, n_init=4,
                 n_recent=64, family="iid", plant=16, seed=0),
    # 2: Llama-3-8B layer, 128K context
    "llama128k": dict(B=1, Hq=32, Hkv=8, d=128, L0=131072, steps=64, K=2048,
                      n_init=128, n_recent=512, family="proj", plant_frac=0.01,
                      seed=0),
    # 3: ReTopK reuse path, Qwen2.5-7B geometry
    "retopk64k": dict(B=1, Hq=28, Hkv=4, d=128, L0=65536, steps=512, K=512,
                      C=32, R=4, W=32, tau=0.85, T_r=128, family="walk", seed=0),
    # 3b: the same ReTopK recipe at 1M context with K = 1024 (the pages' long-
    # context setting for the reuse path)
    "retopk1m": dict(B=1, Hq=28, Hkv=4, d=128, L0=1 << 20, steps=512, K=1024,
                     C=32, R=4, W=32, tau=0.85, T_r=128, family="walk", seed=0),
    # ReTopK at 4M context (the 1M-5M cross-model setting, K = 1024)
    "retopk4m": dict(B=1, Hq=28, Hkv=4, d=128, L0=1 << 22, steps=512, K=1024,
                     C=32, R=4, W=32, tau=0.85, T_r=128, family="walk", seed=0),
    # 4: batched paged decode, Yi-9B geometry
    "yi_paged": dict(B=16, Hq=32, Hkv=4, d=128, Lmin=8192, Lmax=131072,
                     steps=32, K=1024, n_init=64, n_recent=256, family="iid",
                     plant=16, page_size=16, seed=0),
    # 5: 1M-token single sequence, Llama-3-8B geometry
    "llama1m": dict(B=1, Hq=32, Hkv=8, d=128, L0=1 << 20, steps=16, K=4096,
                    n_init=128, n_recent=1024, family="proj", plant_frac=0.005,
                    seed=0),
}


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _randn(shape, seed, device):
    return torch.randn(shape, generator=_gen(seed, device), device=device,
                       dtype=torch.float32)


class _Stream:
    """Component seeds derived from one config seed."""

    def __init__(self, seed: int):
        self.base = 1_000_003 * (seed + 1)

    def __call__(self, tag: int, sub: int = 0) -> int:
        return (self.base + 7919 * tag + 104_729 * sub) % (2**62)


@dataclass
class DecodeWorkload:
    """Contiguous-layout decode workload (optionally also paged)."""

    name: str
    B: int
    Hq: int
    Hkv: int
    d: int
    K: int
    n_init: int
    n_recent: int
    steps: int
    L0: list            # prompt length per sequence
    lcap: int           # per-sequence capacity (max L0 + steps, rounded)
    k: torch.Tensor     # bf16 [B][Hkv][lcap][d]
    v: torch.Tensor     # bf16 [B][Hkv][lcap][d]
    q_all: torch.Tensor # bf16 [steps][B][Hq][d]
    scale: float = field(default=0.0)
    page_size: int = 0
    k_pages: Optional[torch.Tensor] = None   # bf16 [P][Hkv][page][d]
    v_pages: Optional[torch.Tensor] = None
    page_table: Optional[torch.Tensor] = None  # int32 [B][max_pages]

    def lens(self, step: int) -> list:
        return [l0 + step + 1 for l0 in self.L0]

    def q(self, step: int) -> torch.Tensor:
        return self.q_all[step]

    def to(self, device) -> "DecodeWorkload":
        kw = dict(self.__dict__)
        for n in ("k", "v", "q_all", "k_pages", "v_pages", "page_table"):
            if kw[n] is not None:
                kw[n] = kw[n].to(device)
        return DecodeWorkload(**kw)


@dataclass
class RetopkWorkload:
    name: str
    Hq: int
    Hkv: int
    d: int
    K: int
    C: int
    R: int
    W: int
    tau: float
    T_r: int
    steps: int
    L0: int
    lcap: int
    k: torch.Tensor           # bf16 [1][Hkv][lcap][d]
    v: torch.Tensor
    q_prefill: torch.Tensor   # bf16 [C][Hq][d]: walk steps -C .. -1
    q_all: torch.Tensor       # bf16 [steps][Hq][d]
    scale: float = 0.0

    def length(self, step: int) -> int:
        return self.L0 + step + 1

    def to(self, device) -> "RetopkWorkload":
        kw = dict(self.__dict__)
        for n in ("k", "v", "q_prefill", "q_all"):
            kw[n] = kw[n].to(device)
        return RetopkWorkload(**kw)


def _key_params(fam, d, s, device):
    mu = _randn((d,), s(1), device)
    mu = mu * (3.0 / mu.norm())
    if fam == "iid":
        sigma = torch.ones(d, device=device)
    else:
        g = _gen(s(2), device)
        sigma = 0.5 + 1.5 * torch.rand((d,), generator=g, device=device)
    return mu, sigma


def _fill_ordinary(dst_k, dst_v, mu, sigma, s, tag, device):
    """dst_*: bf16 [Hkv][n][d] views filled head by head (bounded temporaries)."""
    Hkv, n, d = dst_k.shape
    for g in range(Hkv):
        xi = _randn((n, d), s(tag, 2 * g), device)
        dst_k[g].copy_((mu + sigma * xi).to(torch.bfloat16))
        del xi
        vv = _randn((n, d), s(tag, 2 * g + 1), device)
        dst_v[g].copy_(vv.to(torch.bfloat16))
        del vv


def make_decode(name: str, device="cpu", L0: Optional[int] = None,
                steps: Optional[int] = None, B: Optional[int] = None,
                K: Optional[int] = None, paged: Optional[bool] = None,
                lcap_align: int = 64, **over) -> DecodeWorkload:
    """Build a decode workload.  Overrides shrink a config for quick parity
    runs (same recipe, smaller sizes)."""
    cfg = dict(CONFIGS[name])
    cfg.update({k: v for k, v in over.items() if v is not None})
    if steps is not None:
        cfg["steps"] = steps
    if B is not None:
        cfg["B"] = B
    if K is not None:
        cfg["K"] = K
    Bn, Hq, Hkv, d = cfg["B"], cfg["Hq"], cfg["Hkv"], cfg["d"]
    G = Hq // Hkv
    fam = cfg["family"]
    s = _Stream(cfg["seed"])
    nsteps = cfg["steps"]

    if "Lmin" in cfg and L0 is None:
        g = _gen(s(9), "cpu")
        L0s = torch.randint(cfg["Lmin"], cfg["Lmax"] + 1, (Bn,), generator=g).tolist()
    else:
        base = L0 if L0 is not None else cfg["L0"]
        if "Lmin" in cfg:  # downsized paged config keeps a spread of lengths
            g = _gen(s(9), "cpu")
            L0s = torch.randint(max(1, base // 16), base + 1, (Bn,), generator=g).tolist()
        else:
            L0s = [base] * Bn
    lmax = max(L0s) + nsteps
    lcap = ((lmax + lcap_align - 1) // lcap_align) * lcap_align

    mu, sigma = _key_params(fam, d, s, device)
    k = torch.zeros((Bn, Hkv, lcap, d), dtype=torch.bfloat16, device=device)
    v = torch.zeros((Bn, Hkv, lcap, d), dtype=torch.bfloat16, device=device)
    for b in range(Bn):
        _fill_ordinary(k[b], v[b], mu, sigma, s, 100 + b, device)

    # head directions (and the query projection for the "proj" family)
    if fam == "proj":
        P = _randn((d, d), s(3), device) / math.sqrt(d)
        x = _randn((Bn, Hq, d), s(4), device)
        u = x @ P.T
    else:
        P = None
        u = _randn((Bn, Hq, d), s(4), device)

    # planted keys near each query head's direction
    for b in range(Bn):
        n_plant = cfg.get("plant") or int(round(cfg["plant_frac"] * L0s[b]))
        n_plant = min(n_plant, L0s[b])
        for h in range(Hq):
            g = _gen(s(5, b * Hq + h), "cpu")
            pos = torch.randperm(L0s[b], generator=g)[:n_plant].to(device)
            noise = _randn((n_plant, d), s(6, b * Hq + h), device)
            kp = 0.5 * u[b, h] + 0.1 * noise
            k[b, h // G].index_copy_(0, pos, kp.to(torch.bfloat16))

    # step queries
    xi = _randn((nsteps, Bn, Hq, d), s(7), device)
    if P is not None:
        xi = xi @ P.T
    q_all = (u.unsqueeze(0) + 0.3 * xi).to(torch.bfloat16)

    wl = DecodeWorkload(name=name, B=Bn, Hq=Hq, Hkv=Hkv, d=d, K=cfg["K"],
                        n_init=cfg["n_init"], n_recent=cfg["n_recent"],
                        steps=nsteps, L0=L0s, lcap=lcap, k=k, v=v, q_all=q_all,
                        scale=1.0 / math.sqrt(d))
    use_pages = paged if paged is not None else ("page_size" in cfg)
    if use_pages:
        _paginate(wl, cfg.get("page_size", 16), s, device)
    return wl


def _paginate(wl: DecodeWorkload, ps: int, s: _Stream, device) -> None:
    """Scatter the per-sequence caches into a shared page pool with a random
    page table (every sequence owns ceil(lcap_b / ps) pages)."""
    Bn, Hkv, d = wl.B, wl.Hkv, wl.d
    need = [-(-(l0 + wl.steps) // ps) for l0 in wl.L0]
    total = sum(need)
    max_pages = max(need)
    g = _gen(s(8), "cpu")
    perm = torch.randperm(total, generator=g)
    kp = torch.zeros((total, Hkv, ps, d), dtype=torch.bfloat16, device=device)
    vp = torch.zeros((total, Hkv, ps, d), dtype=torch.bfloat16, device=device)
    table = torch.full((Bn, max_pages), -1, dtype=torch.int32)
    off = 0
    for b in range(Bn):
        ids = perm[off:off + need[b]]
        off += need[b]
        table[b, :need[b]] = ids.to(torch.int32)
        n = need[b] * ps
        src_k = torch.zeros((Hkv, n, d), dtype=torch.bfloat16, device=device)
        src_v = torch.zeros((Hkv, n, d), dtype=torch.bfloat16, device=device)
        m = min(n, wl.lcap)
        src_k[:, :m] = wl.k[b, :, :m]
        src_v[:, :m] = wl.v[b, :, :m]
        # [Hkv][pages][ps][d] -> [pages][Hkv][ps][d]
        kp[ids.to(device)] = src_k.view(Hkv, need[b], ps, d).transpose(0, 1)
        vp[ids.to(device)] = src_v.view(Hkv, need[b], ps, d).transpose(0, 1)
    wl.page_size = ps
    wl.k_pages, wl.v_pages = kp, vp
    wl.page_table = table.to(device)


def make_retopk(name: str = "retopk64k", device="cpu", L0: Optional[int] = None,
                steps: Optional[int] = None, **over) -> RetopkWorkload:
    cfg = dict(CONFIGS[name])
    cfg.update({k: v for k, v in over.items() if v is not None})
    if steps is not None:
        cfg["steps"] = steps
    if L0 is not None:
        cfg["L0"] = L0
    Hq, Hkv, d, Cn = cfg["Hq"], cfg["Hkv"], cfg["d"], cfg["C"]
    s = _Stream(cfg["seed"])
    nsteps, L0v = cfg["steps"], cfg["L0"]
    lcap = ((L0v + nsteps + 63) // 64) * 64
    mu, sigma = _key_params("walk", d, s, device)
    k = torch.zeros((1, Hkv, lcap, d), dtype=torch.bfloat16, device=device)
    v = torch.zeros((1, Hkv, lcap, d), dtype=torch.bfloat16, device=device)
    _fill_ordinary(k[0], v[0], mu, sigma, s, 100, device)

    rho = 0.97
    total = Cn + nsteps
    walk = torch.empty((total, Hq, d), dtype=torch.float32, device=device)
    qb = _randn((Hq, d), s(11), device)
    qb = qb / qb.norm(dim=-1, keepdim=True)
    noise = _randn((total, Hq, d), s(12), device) / math.sqrt(d)
    for t in range(total):
        if t > 0:
            qb = rho * qb + math.sqrt(1.0 - rho * rho) * noise[t]
            qb = qb / qb.norm(dim=-1, keepdim=True)
        walk[t] = qb * math.sqrt(d)
    qw = walk.to(torch.bfloat16)
    return RetopkWorkload(name=name, Hq=Hq, Hkv=Hkv, d=d, K=cfg["K"], C=Cn,
                          R=cfg["R"], W=cfg["W"], tau=cfg["tau"], T_r=cfg["T_r"],
                          steps=nsteps, L0=L0v, lcap=lcap, k=k, v=v,
                          q_prefill=qw[:Cn].contiguous(),
                          q_all=qw[Cn:].contiguous(), scale=1.0 / math.sqrt(d))


def bits(t: torch.Tensor):
    """bf16 tensor -> numpy uint16 bit patterns (CPU copy)."""
    import numpy as np
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy().view(np.uint16)
