"""sparse_attn_decode_noalloc: the decode step for callers that cannot
allocate device memory while they decode (an engine that reserved all memory
for its KV-cache pool up front, or a host where cudaMalloc is off limits in
the decode loop).  Its scratch is one fixed array that the library holds per
device, so it must give the same results as sparse_attn_decode with a caller
workspace, call after call, while the array keeps the previous call's
contents.

This file is collected last on purpose: the check also has to hold after
every other test has run in the same process."""
import ctypes as C

import numpy as np
import pytest
import torch

from helpers import LSE_TOL, OUT_TOL
from workloads.gen import make_decode


def test_rejects_problems_beyond_the_scratch_array():
    """A problem whose scratch exceeds the array is refused before any launch."""
    import top_retrieval_sparse_gb300 as tsa
    lib = tsa.lib()
    cap = tsa.noalloc_scratch_bytes()
    assert cap == 32 << 20
    fake = C.c_void_p(1 << 20)  # never dereferenced: the size check comes first
    kv = tsa._KvStruct(1 << 20, 1 << 21, None, 0, 0, 1 << 20)
    need = lib.tsa_decode_workspace_size(1, 32, 8, 128, 1 << 20, 2048, 128, 512)
    assert need > cap
    rc = lib.sparse_attn_decode_noalloc(fake, C.byref(kv), fake, 1, 32, 8, 128, 2048, 128, 512,
                                        0.1, fake, None, None, None, None)
    assert rc == -2
    msg = lib.tsa_last_error().decode()
    assert str(need) in msg and str(cap) in msg


def _run_both(wl, steps, dev="cuda"):
    import top_retrieval_sparse_gb300 as tsa
    kv = tsa.kv_contiguous(wl.k.to(dev), wl.v.to(dev))
    B, Hq, d, K = wl.B, wl.Hq, wl.d, wl.K
    n = tsa.decode_workspace_size(B, Hq, wl.Hkv, d, wl.lcap, K, wl.n_init, wl.n_recent)
    assert n <= tsa.noalloc_scratch_bytes()
    work = torch.zeros(n, dtype=torch.uint8, device=dev)

    def bufs():
        return (torch.empty((B, Hq, d), dtype=torch.float32, device=dev),
                torch.empty((B, Hq), dtype=torch.float32, device=dev),
                torch.empty((B, Hq, K), dtype=torch.int32, device=dev),
                torch.empty((B, Hq, K), dtype=torch.float32, device=dev))

    for t in steps:  # two calls in a row through each entry point
        q = wl.q(t).to(dev).contiguous()
        lens = torch.tensor(wl.lens(t), dtype=torch.int32, device=dev)
        a, b = bufs(), bufs()
        tsa.sparse_attn_decode(q, kv, lens, K, wl.n_init, wl.n_recent, wl.scale, out=a[0],
                               lse_out=a[1], topk_idx=a[2], topk_score=a[3], workspace=work)
        tsa.sparse_attn_decode_noalloc(q, kv, lens, K, wl.n_init, wl.n_recent, wl.scale,
                                       out=b[0], lse_out=b[1], topk_idx=b[2], topk_score=b[3])
        torch.cuda.synchronize()
        ref = [x.cpu().numpy() for x in a]
        got = [x.cpu().numpy() for x in b]
        assert np.max(np.abs(got[0] - ref[0])) <= OUT_TOL
        fin = np.isfinite(ref[1])
        assert np.array_equal(fin, np.isfinite(got[1]))
        assert np.max(np.abs(got[1][fin] - ref[1][fin]), initial=0.0) <= LSE_TOL
        for bb in range(B):
            for h in range(Hq):
                assert set(got[2][bb, h].tolist()) == set(ref[2][bb, h].tolist()), (t, bb, h)


@pytest.mark.gpu
def test_matches_workspace_entry_point_tiny():
    wl = make_decode("tiny", steps=2)  # 4 query heads on 1 KV head, 4K keys, K = 64
    _run_both(wl, [0, 1])


@pytest.mark.gpu
def test_matches_workspace_entry_point_many_tiles():
    """Two KV heads, ~100K keys (hundreds of scan tiles and a ragged tail)."""
    wl = make_decode("llama128k", L0=100_003, steps=2, B=1, K=256, Hq=8, Hkv=2,
                     n_init=16, n_recent=64, plant_frac=0.01)
    _run_both(wl, [0, 1])
