"""The C-ABI library builds, loads and exports every symbol include/tsa.h
declares; host-side validation rejects bad arguments without touching a device
(these checks never launch, so they run without a GPU)."""
import ctypes as C
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "tsa.h")).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^\s*(?:const\s+)?[\w\s\*]+?\b(\w+)\s*\(", text, flags=re.M)
    return sorted(set(n for n in names if n not in ("if", "sizeof")))


@pytest.fixture(scope="module")
def lib():
    import top_retrieval_sparse_gb300 as tsa
    return tsa.lib()


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert {"sparse_attn_decode", "lse_merge", "retopk_step", "retopk_create",
            "retopk_init", "tsa_decode_workspace_size"} <= set(names)
    for n in names:
        assert hasattr(lib, n), f"libtsa.so does not export {n}"


def test_library_is_in_tree(lib):
    import top_retrieval_sparse_gb300 as tsa
    assert tsa.library_path().startswith(ROOT)
    assert lib.tsa_version().decode().startswith("tsa")


FAKE = C.c_void_p(1 << 20)  # aligned, never dereferenced: validation fails first


def _kv(tsa, l_cap=1024, page_table=None, page_size=0, max_pages=0):
    return tsa._KvStruct(1 << 20, 1 << 21, page_table, page_size, max_pages, l_cap)


def _decode(lib, tsa, **kw):
    a = dict(q=FAKE, kv=_kv(tsa), lens=FAKE, B=1, Hq=8, Hkv=2, d=128, K=16, n_init=4,
             n_recent=8, scale=0.1, out=FAKE, lse=None, idx=None, sc=None, ws=FAKE,
             ws_bytes=1 << 40, stream=None)
    a.update(kw)
    return lib.sparse_attn_decode(a["q"], C.byref(a["kv"]), a["lens"], a["B"], a["Hq"],
                                  a["Hkv"], a["d"], a["K"], a["n_init"], a["n_recent"],
                                  a["scale"], a["out"], a["lse"], a["idx"], a["sc"], a["ws"],
                                  a["ws_bytes"], a["stream"])


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), -1),                        # only d = 128 is compiled
    (dict(Hq=6, Hkv=4), -1),                 # Hq % Hkv
    (dict(Hq=18, Hkv=2), -1),                # group size 9 > 8
    (dict(B=129, Hq=32, Hkv=4), -1),         # B * Hkv > 512
    (dict(K=-1), -1),
    (dict(n_init=-2), -1),
    (dict(q=None), -1),
    (dict(q=C.c_void_p((1 << 20) + 4)), -1),  # q not 16-byte aligned
    (dict(scale=float("nan")), -1),
    (dict(ws=None), -2),
    (dict(ws=C.c_void_p((1 << 20) + 64)), -2),  # workspace not 256-byte aligned
    (dict(ws_bytes=100), -2),                   # workspace too small
])
def test_decode_validation(lib, kw, code):
    import top_retrieval_sparse_gb300 as tsa
    assert _decode(lib, tsa, **kw) == code
    assert lib.tsa_last_error().decode() != ""


def test_decode_validation_paged(lib):
    import top_retrieval_sparse_gb300 as tsa
    assert _decode(lib, tsa, kv=_kv(tsa, 1024, 1 << 22, 24, 64)) == -1    # page size 24
    assert _decode(lib, tsa, kv=_kv(tsa, 1000, 1 << 22, 16, 64)) == -1    # l_cap mismatch
    assert _decode(lib, tsa, kv=_kv(tsa, 1024, 1 << 22, 16, 0)) == -1
    k = tsa._KvStruct(None, 1 << 21, None, 0, 0, 1024)
    assert _decode(lib, tsa, kv=k) == -1


def test_workspace_sizes(lib):
    small = lib.tsa_decode_workspace_size(1, 32, 8, 128, 131136, 2048, 128, 512)
    big = lib.tsa_decode_workspace_size(1, 32, 8, 128, 1 << 20, 4096, 128, 1024)
    assert 0 < small < big
    # scores + candidate positions dominate: 2 x 4 bytes per (head, position)
    assert big >= 32 * (1 << 20) * 8
    assert lib.tsa_decode_workspace_size(1, 32, 8, 128, 1000, -1, 0, 0) == 0


def test_lse_merge_validation(lib):
    assert lib.lse_merge(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 0, None) == -1
    assert lib.lse_merge(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 2048, None) == -1
    assert lib.lse_merge(None, FAKE, FAKE, FAKE, FAKE, FAKE, 4, 16, None) == -1
    assert lib.lse_merge(None, None, None, None, None, None, 0, 16, None) == 0


def test_retopk_host_state_machine(lib):
    """create / counters / destroy are host-only; step refuses before init."""
    n = lib.retopk_state_size(28, 128, 512, 32)
    assert n >= 28 * 32 * (128 + 512 + 1) * 4
    h = C.c_void_p()
    assert lib.retopk_create(C.byref(h), 28, 4, 128, 512, 32, 4, 32, 0.85, 128, 70000,
                             FAKE, n) == 0
    assert lib.retopk_workspace_size(h) > 28 * 70000 * 8
    t, head = C.c_int64(), C.c_int32()
    assert lib.retopk_get_counters(h, C.byref(t), C.byref(head)) == 0
    assert (t.value, head.value) == (0, 0)
    import top_retrieval_sparse_gb300 as tsa
    kv = _kv(tsa, 70000)
    rc = lib.retopk_step(h, FAKE, C.byref(kv), 100, 0.1, FAKE, None, None, None, None, None,
                         FAKE, 1 << 40, None)
    assert rc == -4  # not initialised
    assert lib.retopk_set_counters(h, 5, 40) == -1   # head outside [0, C)
    assert lib.retopk_set_counters(h, 5, 3) == 0
    rc = lib.retopk_step(h, FAKE, C.byref(kv), 70001, 0.1, FAKE, None, None, None, None, None,
                         FAKE, 1 << 40, None)
    assert rc == -1  # len beyond max_len
    rc = lib.retopk_step(h, FAKE, C.byref(kv), 100, 0.1, FAKE, None, None, None, None, None,
                         FAKE, 10, None)
    assert rc == -2  # workspace too small
    assert lib.retopk_destroy(h) == 0
    bad = C.c_void_p()
    assert lib.retopk_create(C.byref(bad), 28, 4, 128, 512, 32, 40, 32, 0.85, 128, 70000,
                             FAKE, n) == -1  # R > C
    assert lib.retopk_create(C.byref(bad), 28, 4, 128, 512, 32, 4, 32, 0.85, 0, 70000,
                             FAKE, n) == -1  # T_r < 1
    assert lib.retopk_create(C.byref(bad), 28, 4, 128, 512, 32, 4, 32, 0.85, 128, 70000,
                             FAKE, n - 1) == -1  # state too small
    # the selector's candidate bitmap: in one CTA's shared memory up to 1.5 M
    # positions, beyond that in the workspace (1 bit per position and query
    # head) with its second level (1 bit per word) in 192 KiB of shared
    # memory: 50331648 positions at most
    small = C.c_void_p()
    assert lib.retopk_create(C.byref(small), 28, 4, 128, 512, 32, 4, 32, 0.85, 128,
                             1_500_000, FAKE, n) == 0
    cap = 192 * 1024 * 8 * 32
    ok = C.c_void_p()
    assert lib.retopk_create(C.byref(ok), 28, 4, 128, 512, 32, 4, 32, 0.85, 128, cap,
                             FAKE, n) == 0
    # the long cache's bitmap is workspace: max_len / 8 bytes per query head more
    grow = lib.retopk_workspace_size(ok) - lib.retopk_workspace_size(small)
    dense = 28 * (cap - 1_500_000 - 64) * 16   # the pair list and spill area grow too
    assert grow >= dense + 28 * cap // 8
    assert lib.retopk_destroy(ok) == 0 and lib.retopk_destroy(small) == 0
    assert lib.retopk_create(C.byref(bad), 28, 4, 128, 512, 32, 4, 32, 0.85, 128, cap + 1,
                             FAKE, n) == -1  # max_len beyond the second level


def test_status_and_injection_validation(lib):
    """The status query refuses a bad workspace before any CUDA call; the
    injection hook checks its limit and launches nothing."""
    assert lib.tsa_workspace_status(None, 1, None) == -2
    assert lib.tsa_workspace_status(C.c_void_p((1 << 20) + 8), 1, None) == -2
    assert lib.tsa_inject_scan_stall(-1) == -1
    assert lib.tsa_inject_scan_stall(2_000_000_000) == -1
    n0 = lib.tsa_kernel_launches()
    assert lib.tsa_inject_scan_stall(1_000_000) == 0
    assert lib.tsa_inject_scan_stall(0) == 0   # cancel
    assert lib.tsa_kernel_launches() == n0


def _noalloc(lib, tsa, **kw):
    a = dict(q=FAKE, kv=_kv(tsa), lens=FAKE, B=1, Hq=8, Hkv=2, d=128, K=16, n_init=4,
             n_recent=8, scale=0.1, out=FAKE, lse=None, idx=None, sc=None, stream=None)
    a.update(kw)
    return lib.sparse_attn_decode_noalloc(a["q"], C.byref(a["kv"]), a["lens"], a["B"], a["Hq"],
                                          a["Hkv"], a["d"], a["K"], a["n_init"], a["n_recent"],
                                          a["scale"], a["out"], a["lse"], a["idx"], a["sc"],
                                          a["stream"])


@pytest.mark.parametrize("kw", [dict(d=64), dict(Hq=6, Hkv=4), dict(K=-1), dict(q=None),
                                dict(out=C.c_void_p((1 << 20) + 4)), dict(scale=float("inf")),
                                dict(lens=None)])
def test_noalloc_validates_before_touching_the_device(lib, kw):
    """Invalid arguments are refused with the decode entry point's own code
    before the scratch array or the stream is touched: without a GPU any CUDA
    call would fail with TSA_ERR_CUDA (-3), and no launch is counted."""
    import top_retrieval_sparse_gb300 as tsa
    n0 = lib.tsa_kernel_launches()
    assert _noalloc(lib, tsa, **kw) == -1
    assert lib.tsa_kernel_launches() == n0


def test_noalloc_size_limit_boundaries(lib):
    """The scratch need grows as B*Hq*16*(l_cap + 65536) bytes plus ~12 KiB per
    head: B*Hq = 4 fits up to about 458 K positions, B*Hq = 16 about 65 K, and
    B*Hq = 32 fits no cache at all; an oversize problem is refused (-2) before
    any CUDA call."""
    import top_retrieval_sparse_gb300 as tsa
    cap = lib.tsa_noalloc_scratch_bytes()
    assert cap == 32 << 20

    def need(B, Hq, Hkv, l_cap):
        return lib.tsa_decode_workspace_size(B, Hq, Hkv, 128, l_cap, 64, 4, 64)

    def largest_fit(B, Hq, Hkv):
        lo, hi = 0, 1 << 22
        if need(B, Hq, Hkv, 0) > cap:
            return -1
        while lo < hi:
            mid = (lo + hi + 1) // 2
            if need(B, Hq, Hkv, mid) <= cap:
                lo = mid
            else:
                hi = mid - 1
        return lo
    l4 = largest_fit(1, 4, 1)
    assert 450_000 < l4 < 460_000
    assert 60_000 < largest_fit(1, 16, 2) < 66_000
    assert largest_fit(1, 32, 8) == -1 and largest_fit(2, 16, 4) == -1
    assert _noalloc(lib, tsa, Hq=4, Hkv=1, kv=_kv(tsa, l4 + 64)) == -2
    assert "scratch" in lib.tsa_last_error().decode()


def test_prefill_supports_validation(lib):
    """retopk_prefill_supports checks its sizes, pointers and workspace on the
    host (no CUDA call: the codes are the validation ones, not -3)."""
    import top_retrieval_sparse_gb300 as tsa
    kv = _kv(tsa, 1024)
    n = lib.retopk_prefill_workspace_size(8, 28, 4, 128, 1024, 64)
    assert n > lib.tsa_decode_workspace_size(8, 28, 4, 128, 1024, 64, 0, 0)
    assert lib.retopk_prefill_workspace_size(0, 28, 4, 128, 1024, 64) == 0

    def call(**kw):
        a = dict(q=FAKE, L0=1000, C=8, Hq=28, Hkv=4, d=128, K=64, sup=FAKE, cnt=None, ws=FAKE,
                 nb=n, kv=kv)
        a.update(kw)
        return lib.retopk_prefill_supports(a["q"], C.byref(a["kv"]), a["L0"], a["C"], a["Hq"],
                                           a["Hkv"], a["d"], a["K"], 0.1, a["sup"], a["cnt"],
                                           a["ws"], a["nb"], None)
    assert call(C=0) == -1
    assert call(K=0) == -1
    assert call(L0=5) == -1         # fewer positions than queries
    assert call(L0=2000) == -1      # beyond l_cap
    assert call(sup=None) == -1
    assert call(d=64) == -1
    assert call(C=200) == -1        # C * Hkv > 512
    assert call(nb=n - 1) == -2
    assert call(ws=None) == -2


def test_retopk_batched_validation(lib):
    """retopk_step_batched checks its handles (count, initialised, equal
    shapes, no shared state), lengths and workspace on the host."""
    import top_retrieval_sparse_gb300 as tsa
    n = lib.retopk_state_size(28, 128, 512, 32)
    hs = []
    for j in range(3):
        h = C.c_void_p()
        assert lib.retopk_create(C.byref(h), 28, 4, 128, 512, 32, 4, 32, 0.85, 128, 70000,
                                 C.c_void_p((1 << 20) * (j + 1)), n) == 0
        assert lib.retopk_set_counters(h, 0, 0) == 0  # marks it initialised (host only)
        hs.append(h)
    other = C.c_void_p()
    assert lib.retopk_create(C.byref(other), 28, 4, 128, 256, 32, 4, 32, 0.85, 128, 70000,
                             C.c_void_p(1 << 26), n) == 0
    assert lib.retopk_set_counters(other, 0, 0) == 0
    w1 = lib.retopk_batched_workspace_size(hs[0], 1)
    w3 = lib.retopk_batched_workspace_size(hs[0], 3)
    assert w1 == lib.retopk_workspace_size(hs[0]) and w3 > 2 * w1
    assert lib.retopk_batched_workspace_size(hs[0], 65) == 0
    kv = tsa._KvStruct(1 << 20, 1 << 21, None, 0, 0, 70000)

    def call(handles, lens, nb=1 << 40):
        arr = (C.c_void_p * len(handles))(*[h.value for h in handles])
        ls = (C.c_int64 * len(lens))(*lens)
        return lib.retopk_step_batched(arr, len(handles), FAKE, C.byref(kv), ls, 0.1, FAKE,
                                       None, None, None, None, None, FAKE, nb, None)
    assert call([hs[0], other], [100, 200]) == -1          # different K
    assert call([hs[0], hs[0]], [100, 200]) == -1          # the same state twice
    assert call(hs, [100, 0, 50]) == -1                    # a length below 1
    assert call(hs, [100, 70001, 50]) == -1                # beyond max_len
    assert call(hs, [100, 200, 300], nb=w3 - 1) == -2      # workspace too small
    fresh = C.c_void_p()
    assert lib.retopk_create(C.byref(fresh), 28, 4, 128, 512, 32, 4, 32, 0.85, 128, 70000,
                             C.c_void_p(1 << 27), n) == 0
    assert call([hs[0], fresh], [100, 200]) == -4          # not initialised
    for h in hs + [other, fresh]:
        assert lib.retopk_destroy(h) == 0


def _kq(tsa, codes=1 << 20, scale=1 << 21, err=1 << 22):
    return tsa._Kq8Struct(codes, scale, err)


def _decode_q8(lib, tsa, **kw):
    a = dict(q=FAKE, kv=_kv(tsa), kq=_kq(tsa), n_new=1, lens=FAKE, B=1, Hq=8, Hkv=2, d=128,
             K=16, n_init=4, n_recent=8, scale=0.1, out=FAKE, ws=FAKE, ws_bytes=1 << 40)
    a.update(kw)
    kq = C.byref(a["kq"]) if a["kq"] is not None else None
    return lib.sparse_attn_decode_q8(a["q"], C.byref(a["kv"]), kq, a["n_new"], a["lens"],
                                     a["B"], a["Hq"], a["Hkv"], a["d"], a["K"], a["n_init"],
                                     a["n_recent"], a["scale"], a["out"], None, None, None,
                                     a["ws"], a["ws_bytes"], None)


@pytest.mark.parametrize("kw,code", [
    (dict(d=64), -1),
    (dict(Hq=18, Hkv=2), -1),
    (dict(K=-1), -1),
    (dict(kq=None), -1),
    (dict(n_new=-1), -1),
    (dict(scale=float("inf")), -1),
    (dict(lens=None), -1),
    (dict(ws=None), -2),
    (dict(ws_bytes=1000), -2),
])
def test_decode_q8_validation(lib, kw, code):
    import top_retrieval_sparse_gb300 as tsa
    if kw.get("kq", 0) is None:
        assert _decode_q8(lib, tsa, kq=None) == code
    else:
        assert _decode_q8(lib, tsa, **kw) == code
    assert lib.tsa_last_error().decode() != ""


def test_decode_q8_rejects_bad_codes(lib):
    import top_retrieval_sparse_gb300 as tsa
    assert _decode_q8(lib, tsa, kq=_kq(tsa, codes=(1 << 20) + 8)) == -1  # codes not 16-aligned
    assert _decode_q8(lib, tsa, kq=_kq(tsa, codes=0)) == -1
    assert _decode_q8(lib, tsa, kq=_kq(tsa, err=0)) == -1
    assert _decode_q8(lib, tsa, kq=_kq(tsa, scale=(1 << 21) + 2)) == -1  # scale not 4-aligned


def _quantize(lib, tsa, **kw):
    a = dict(kv=_kv(tsa), kq=_kq(tsa), lens=FAKE, B=1, Hkv=2, d=128, n_tail=1, fit=0)
    a.update(kw)
    kq = C.byref(a["kq"]) if a["kq"] is not None else None
    return lib.tsa_quantize_keys(C.byref(a["kv"]), kq, a["lens"], a["B"], a["Hkv"], a["d"],
                                 a["n_tail"], a["fit"], None)


def test_quantize_keys_validation(lib):
    import top_retrieval_sparse_gb300 as tsa
    assert _quantize(lib, tsa, d=64) == -1
    assert _quantize(lib, tsa, fit=2) == -1
    assert _quantize(lib, tsa, n_tail=-1) == -1
    assert _quantize(lib, tsa, kq=None) == -1
    assert _quantize(lib, tsa, lens=None) == -1
    assert _quantize(lib, tsa, Hkv=0) == -1
    assert _quantize(lib, tsa, kv=_kv(tsa, 1024, 1 << 22, 24, 64)) == -1  # page size 24
    assert _quantize(lib, tsa, B=0) == 0  # nothing to do: no launch


def test_q8_workspace_extends_the_decode_one(lib):
    args = (2, 32, 8, 128, 131136, 2048, 128, 512)
    plain = lib.tsa_decode_workspace_size(*args)
    q8 = lib.tsa_decode_q8_workspace_size(*args)
    # fp16 prepared queries, two floats per head, each region 256-byte aligned
    assert plain < q8 <= plain + 2 * 32 * (256 + 256 + 256) + 3 * 256
