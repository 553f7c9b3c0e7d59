"""Decode-step top-K sparse attention on GB300 (sm_103a).

Thin ctypes binding over ``libtsa.so`` (C ABI in ``include/tsa.h``).  The
functions keep the library's names (``sparse_attn_decode``, ``lse_merge``,
``retopk_*``) and only marshal arguments: every step of the computation runs
in the library's CUDA kernels.  PyTorch supplies device memory and streams.

Importing this package loads the library; if it is missing it is built with
nvcc, and if that fails the import raises -- there is no fallback path.
"""
from __future__ import annotations

import ctypes as C
import math
import os
import threading
from typing import Optional

import torch

from . import build as _build

__all__ = [
    "TsaError", "lib", "KV", "kv_contiguous", "kv_paged", "decode_workspace_size",
    "sparse_attn_decode", "lse_merge", "ReTopK", "library_path", "set_stage_events",
    "set_trace", "read_trace", "kernel_launches", "sparse_attn_decode_noalloc",
    "noalloc_scratch_bytes",
]

TSA_OK = 0
_ERRORS = {-1: "TSA_ERR_INVALID_ARG", -2: "TSA_ERR_WORKSPACE", -3: "TSA_ERR_CUDA",
           -4: "TSA_ERR_STATE", -5: "TSA_ERR_DEVICE_CHECK", -6: "TSA_ERR_TIMEOUT"}


class TsaError(RuntimeError):
    def __init__(self, code: int, msg: str):
        super().__init__(f"{_ERRORS.get(code, code)}: {msg}")
        self.code = code


class _KvStruct(C.Structure):
    _fields_ = [("k", C.c_void_p), ("v", C.c_void_p), ("page_table", C.c_void_p),
                ("page_size", C.c_int32), ("max_pages", C.c_int32), ("l_cap", C.c_int64)]


_lock = threading.Lock()
_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """Load libtsa.so (building it first if it is missing or stale)."""
    global _lib
    with _lock:
        if _lib is None:
            path = _build.build()
            L = C.CDLL(path)
            P, i32, i64, f32, sz = C.c_void_p, C.c_int, C.c_int64, C.c_float, C.c_size_t
            L.tsa_last_error.restype = C.c_char_p
            L.tsa_version.restype = C.c_char_p
            L.tsa_decode_workspace_size.argtypes = [i32, i32, i32, i32, i64, i32, i32, i32]
            L.tsa_decode_workspace_size.restype = sz
            L.sparse_attn_decode.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, i32, f32,
                                             P, P, P, P, P, sz, P]
            L.lse_merge.argtypes = [P, P, P, P, P, P, i32, i32, P]
            L.sparse_attn_decode_noalloc.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32,
                                                     i32, f32, P, P, P, P, P]
            L.tsa_noalloc_scratch_bytes.restype = sz
            L.retopk_state_size.argtypes = [i32, i32, i32, i32]
            L.retopk_state_size.restype = sz
            L.retopk_create.argtypes = [C.POINTER(P), i32, i32, i32, i32, i32, i32, i32, f32,
                                        i32, i64, P, sz]
            L.retopk_init.argtypes = [P, P, P, P, P]
            L.retopk_workspace_size.argtypes = [P]
            L.retopk_workspace_size.restype = sz
            L.retopk_step.argtypes = [P, P, P, i64, f32, P, P, P, P, P, P, P, sz, P]
            L.retopk_batched_workspace_size.argtypes = [P, i32]
            L.retopk_batched_workspace_size.restype = sz
            L.retopk_step_batched.argtypes = [P, i32, P, P, P, f32, P, P, P, P, P, P, P, sz, P]
            L.retopk_get_counters.argtypes = [P, C.POINTER(i64), C.POINTER(C.c_int32)]
            L.retopk_set_counters.argtypes = [P, i64, C.c_int32]
            L.retopk_destroy.argtypes = [P]
            L.tsa_set_stage_events.argtypes = [C.POINTER(P), i32]
            L.tsa_set_trace.argtypes = [P, sz]
            L.tsa_kernel_launches.restype = C.c_ulonglong
            L.tsa_workspace_status.argtypes = [P, i32, P]
            L.sparse_attn_decode_shard.argtypes = [P, P, i64, i64, i64, i32, i32, i32, i32, i32,
                                                   i32, f32, P, P, P, P, P, sz, P]
            L.tsa_attend_set_workspace_size.argtypes = [i32, i32, i32]
            L.tsa_attend_set_workspace_size.restype = sz
            L.attend_set.argtypes = [P, P, i32, i32, i32, i32, P, P, i32, f32, P, P, P, sz, P]
            L.retopk_prefill_workspace_size.argtypes = [i32, i32, i32, i32, i64, i32]
            L.retopk_prefill_workspace_size.restype = sz
            L.retopk_prefill_supports.argtypes = [P, P, i64, i32, i32, i32, i32, i32, f32, P, P,
                                                  P, sz, P]
            L.tsa_inject_scan_stall.argtypes = [C.c_longlong]
            L.tsa_quantize_keys.argtypes = [P, P, P, i32, i32, i32, i64, i32, P]
            L.tsa_decode_q8_workspace_size.argtypes = [i32, i32, i32, i32, i64, i32, i32, i32]
            L.tsa_decode_q8_workspace_size.restype = sz
            L.sparse_attn_decode_q8.argtypes = [P, P, P, i32, P, i32, i32, i32, i32, i32, i32,
                                                i32, f32, P, P, P, P, P, sz, P]
            _lib = L
    return _lib


def _check(rc: int) -> None:
    if rc != TSA_OK:
        raise TsaError(rc, lib().tsa_last_error().decode())


def _p(t: Optional[torch.Tensor]):
    return None if t is None else C.c_void_p(t.data_ptr())


def _stream(stream) -> C.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return C.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def _want(t: torch.Tensor, dtype, name: str):
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def kernel_launches() -> int:
    """Kernels the library has launched in this process so far."""
    return int(lib().tsa_kernel_launches())


def set_stage_events(events) -> None:
    """Per-stage timing: a list of 4 torch.cuda.Event(enable_timing=True) (or None).

    Later calls on this thread record them before the first launch and after
    the scan, the selection and the attention kernel, on the call's stream."""
    if not events:
        _check(lib().tsa_set_stage_events(None, 0))
        return
    arr = (C.c_void_p * len(events))(*[C.c_void_p(e.cuda_event) for e in events])
    _check(lib().tsa_set_stage_events(arr, len(events)))


def set_trace(buf: Optional[torch.Tensor]) -> None:
    """Per-CTA kernel timeline into a uint8 device tensor (see include/tsa.h);
    the first 4 bytes count records and must be zeroed by the caller."""
    if buf is None:
        _check(lib().tsa_set_trace(None, 0))
    else:
        _check(lib().tsa_set_trace(_p(buf), buf.numel()))


def read_trace(buf: torch.Tensor):
    """Decode a trace buffer into a list of dicts (kernel, cta, sm, t0..t3)."""
    import numpy as np
    raw = buf.cpu().numpy()
    n = int(raw[:4].view(np.uint32)[0])
    cap = (raw.size - 64) // 48
    rec = raw[64:64 + 48 * min(n, cap)].view(np.uint32).reshape(-1, 12)
    out = []
    for r in rec:
        t = r[4:12].view(np.uint64)
        out.append({"kernel": int(r[0]), "cta": int(r[1]), "sm": int(r[2]),
                    "info": int(r[3]), "t": [int(x) for x in t]})
    return out


class KV:
    """A layer's KV cache as the library sees it (keeps the tensors alive)."""

    def __init__(self, k, v, page_table=None, page_size=0):
        _want(k, torch.bfloat16, "k")
        _want(v, torch.bfloat16, "v")
        self.k, self.v, self.page_table = k, v, page_table
        if page_table is None:
            if k.dim() != 4:
                raise ValueError("contiguous k must be [B][Hkv][l_cap][d]")
            self.B, self.Hkv, self.l_cap, self.d = k.shape
            self.struct = _KvStruct(k.data_ptr(), v.data_ptr(), None, 0, 0, self.l_cap)
        else:
            _want(page_table, torch.int32, "page_table")
            if k.dim() != 4:
                raise ValueError("paged k must be [pages][Hkv][page_size][d]")
            _, self.Hkv, ps, self.d = k.shape
            self.B, max_pages = page_table.shape
            self.l_cap = max_pages * ps
            self.struct = _KvStruct(k.data_ptr(), v.data_ptr(), page_table.data_ptr(), ps,
                                    max_pages, self.l_cap)


def kv_contiguous(k: torch.Tensor, v: torch.Tensor) -> KV:
    return KV(k, v)


def kv_paged(k_pages: torch.Tensor, v_pages: torch.Tensor, page_table: torch.Tensor) -> KV:
    return KV(k_pages, v_pages, page_table)


def decode_workspace_size(B, Hq, Hkv, d, l_cap, K, n_init, n_recent) -> int:
    return int(lib().tsa_decode_workspace_size(B, Hq, Hkv, d, l_cap, K, n_init, n_recent))


def sparse_attn_decode(q: torch.Tensor, kv: KV, lens: torch.Tensor, K: int, n_init: int,
                       n_recent: int, scale: Optional[float] = None,
                       out: Optional[torch.Tensor] = None,
                       lse_out: Optional[torch.Tensor] = None,
                       topk_idx: Optional[torch.Tensor] = None,
                       topk_score: Optional[torch.Tensor] = None,
                       workspace: Optional[torch.Tensor] = None, stream=None):
    """One decode step over every sequence and query head (see include/tsa.h).

    q: bf16 [B][Hq][d] on the device; lens: int32 [B] on the device.
    workspace: uint8, zero-filled before its first use and then reused as
    is (each call leaves it ready for the next); None allocates a fresh one.
    Returns (out, lse_out, topk_idx, topk_score) (the optional ones may be None).
    """
    _want(q, torch.bfloat16, "q")
    _want(lens, torch.int32, "lens")
    B, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        nb = decode_workspace_size(B, Hq, kv.Hkv, d, kv.l_cap, K, n_init, n_recent)
        workspace = torch.zeros(max(nb, 256), dtype=torch.uint8, device=q.device)
    _check(lib().sparse_attn_decode(
        _p(q), C.byref(kv.struct), _p(lens), B, Hq, kv.Hkv, d, K, n_init, n_recent,
        float(scale), _p(out), _p(lse_out), _p(topk_idx), _p(topk_score), _p(workspace),
        workspace.numel() * workspace.element_size(), _stream(stream)))
    return out, lse_out, topk_idx, topk_score


class _Kq8Struct(C.Structure):
    _fields_ = [("codes", C.c_void_p), ("scale", C.c_void_p), ("err", C.c_void_p)]


class KeyCodes:
    """The int8 copy of a cache's keys (see tsa_kq8 in include/tsa.h): codes
    with the row geometry of kv.k (one byte per element, offset binary),
    per-(sequence, KV head, channel) scales and error bounds."""

    def __init__(self, kv: "KV", B: Optional[int] = None):
        dev = kv.k.device
        self.B = kv.B if B is None else B
        self.codes = torch.empty(kv.k.shape, dtype=torch.uint8, device=dev)
        self.scale = torch.zeros((self.B, kv.Hkv, kv.d), dtype=torch.float32, device=dev)
        self.err = torch.zeros((self.B, kv.Hkv, kv.d), dtype=torch.float32, device=dev)
        self.struct = _Kq8Struct(self.codes.data_ptr(), self.scale.data_ptr(),
                                 self.err.data_ptr())


def quantize_keys(kv: "KV", codes: KeyCodes, lens: torch.Tensor, fit: bool = True,
                  n_tail: int = 0, stream=None) -> KeyCodes:
    """Fit scales and code rows [0, lens[b]) (fit), or code the last n_tail
    rows of each sequence with the stored scales."""
    _want(lens, torch.int32, "lens")
    _check(lib().tsa_quantize_keys(C.byref(kv.struct), C.byref(codes.struct), _p(lens),
                                   codes.B, kv.Hkv, kv.d, int(n_tail), 1 if fit else 0,
                                   _stream(stream)))
    return codes


def decode_q8_workspace_size(B, Hq, Hkv, d, l_cap, K, n_init, n_recent) -> int:
    return int(lib().tsa_decode_q8_workspace_size(B, Hq, Hkv, d, l_cap, K, n_init, n_recent))


def sparse_attn_decode_q8(q: torch.Tensor, kv: KV, codes: KeyCodes, lens: torch.Tensor, K: int,
                          n_init: int, n_recent: int, n_new: int = 0,
                          scale: Optional[float] = None, out: Optional[torch.Tensor] = None,
                          lse_out: Optional[torch.Tensor] = None,
                          topk_idx: Optional[torch.Tensor] = None,
                          topk_score: Optional[torch.Tensor] = None,
                          workspace: Optional[torch.Tensor] = None, stream=None):
    """sparse_attn_decode through the key codes (same results; the last n_new
    rows of each sequence are coded first).  The workspace is a q8 one."""
    _want(q, torch.bfloat16, "q")
    _want(lens, torch.int32, "lens")
    B, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        nb = decode_q8_workspace_size(B, Hq, kv.Hkv, d, kv.l_cap, K, n_init, n_recent)
        workspace = torch.zeros(max(nb, 256), dtype=torch.uint8, device=q.device)
    _check(lib().sparse_attn_decode_q8(
        _p(q), C.byref(kv.struct), C.byref(codes.struct), int(n_new), _p(lens), B, Hq, kv.Hkv,
        d, K, n_init, n_recent, float(scale), _p(out), _p(lse_out), _p(topk_idx),
        _p(topk_score), _p(workspace), workspace.numel() * workspace.element_size(),
        _stream(stream)))
    return out, lse_out, topk_idx, topk_score


def sparse_attn_decode_noalloc(q: torch.Tensor, kv: KV, lens: torch.Tensor, K: int,
                               n_init: int, n_recent: int, scale: Optional[float] = None,
                               out: Optional[torch.Tensor] = None,
                               lse_out: Optional[torch.Tensor] = None,
                               topk_idx: Optional[torch.Tensor] = None,
                               topk_score: Optional[torch.Tensor] = None, stream=None):
    """sparse_attn_decode with the library's own fixed scratch array instead
    of a workspace (for callers that cannot allocate while decoding; limits
    and concurrency rules in include/tsa.h).  The output buffers are the
    caller's: pass them to allocate nothing here either."""
    _want(q, torch.bfloat16, "q")
    _want(lens, torch.int32, "lens")
    B, Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    _check(lib().sparse_attn_decode_noalloc(
        _p(q), C.byref(kv.struct), _p(lens), B, Hq, kv.Hkv, d, K, n_init, n_recent,
        float(scale), _p(out), _p(lse_out), _p(topk_idx), _p(topk_score), _stream(stream)))
    return out, lse_out, topk_idx, topk_score


def noalloc_scratch_bytes() -> int:
    return int(lib().tsa_noalloc_scratch_bytes())


def decode_shard(q: torch.Tensor, kv: "KV", shard_len: int, pos_offset: int, global_len: int,
                 K: int, n_init: int, n_recent: int, scale=None, out=None, lse_out=None,
                 topk_idx=None, topk_score=None, workspace=None, stream=None):
    """One shard [pos_offset, pos_offset + shard_len) of a sequence of
    global_len positions (q bf16 [Hq][128]): local top-K (local row indices)
    and attention over the shard's window rows and that top-K."""
    _want(q, torch.bfloat16, "q")
    Hq, d = q.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((Hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = decode_workspace_size(1, Hq, kv.Hkv, d, kv.l_cap, K, n_init, n_recent)
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    _check(lib().sparse_attn_decode_shard(_p(q), C.byref(kv.struct), int(shard_len),
                                          int(pos_offset), int(global_len), Hq, kv.Hkv, d, K,
                                          n_init, n_recent, float(scale), _p(out), _p(lse_out),
                                          _p(topk_idx), _p(topk_score), _p(workspace),
                                          workspace.numel(), _stream(stream)))
    return out


def attend_set(q: torch.Tensor, kv: "KV", positions: torch.Tensor, counts: torch.Tensor,
               scale=None, out=None, lse_out=None, workspace=None, stream=None):
    """Attention over given rows: q bf16 [B][Hq][128], positions int32
    [B][Hq][M], counts int32 [B][Hq]; returns out fp32 [B][Hq][128]."""
    _want(q, torch.bfloat16, "q")
    _want(positions, torch.int32, "positions")
    _want(counts, torch.int32, "counts")
    B, Hq, d = q.shape
    M = positions.shape[-1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty((B, Hq, d), dtype=torch.float32, device=q.device)
    if workspace is None:
        n = int(lib().tsa_attend_set_workspace_size(B, Hq, M))
        workspace = torch.zeros(n, dtype=torch.uint8, device=q.device)
    _check(lib().attend_set(_p(q), C.byref(kv.struct), B, Hq, kv.Hkv, d, _p(positions),
                            _p(counts), M, float(scale), _p(out), _p(lse_out), _p(workspace),
                            workspace.numel(), _stream(stream)))
    return out


def prefill_workspace_size(C, Hq, Hkv, d, l_cap, K) -> int:
    return int(lib().retopk_prefill_workspace_size(C, Hq, Hkv, d, l_cap, K))


def prefill_supports(q_prefill: torch.Tensor, kv: "KV", L0: int, K: int, scale=None,
                     supports=None, counts=None, workspace=None, stream=None):
    """Exact causal top-K of the last C prefill queries (q_prefill bf16
    [C][Hq][128], query c at position L0 - C + c) over their prefixes, in one
    call: returns (supports int32 [C][Hq][K] padded with -1, counts int32
    [C][Hq])."""
    _want(q_prefill, torch.bfloat16, "q_prefill")
    Cn, Hq, d = q_prefill.shape
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dev = q_prefill.device
    if supports is None:
        supports = torch.empty((Cn, Hq, K), dtype=torch.int32, device=dev)
    if counts is None:
        counts = torch.empty((Cn, Hq), dtype=torch.int32, device=dev)
    if workspace is None:
        n = prefill_workspace_size(Cn, Hq, kv.Hkv, d, kv.l_cap, K)
        workspace = torch.zeros(n, dtype=torch.uint8, device=dev)
    _check(lib().retopk_prefill_supports(_p(q_prefill), C.byref(kv.struct), int(L0), Cn, Hq,
                                         kv.Hkv, d, K, float(scale), _p(supports), _p(counts),
                                         _p(workspace), workspace.numel(), _stream(stream)))
    return supports, counts


def workspace_status(workspace: torch.Tensor, clear: bool = True, stream=None) -> int:
    """Device-side status of a decode or ReTopK workspace (synchronises the
    stream): 0, TSA_ERR_TIMEOUT (-6) or TSA_ERR_DEVICE_CHECK (-5)."""
    return int(lib().tsa_workspace_status(_p(workspace), 1 if clear else 0, _stream(stream)))


def inject_scan_stall(wait_limit_ns: int) -> None:
    """Fault injection for tests: the next call's key scan gives up a wait
    after wait_limit_ns (its first CTA withholds a tile copy)."""
    _check(lib().tsa_inject_scan_stall(int(wait_limit_ns)))


def lse_merge(o_a, lse_a, o_b, lse_b, o_out=None, lse_out=None, stream=None):
    """Eq. 4-5 merge of two (o, lse) partials: o fp32 [rows][d], lse fp32 [rows]."""
    rows, d = o_a.shape
    if o_out is None:
        o_out = torch.empty_like(o_a)
    if lse_out is None:
        lse_out = torch.empty_like(lse_a)
    for t, n in ((o_a, "o_a"), (o_b, "o_b"), (o_out, "o_out"), (lse_a, "lse_a"),
                 (lse_b, "lse_b"), (lse_out, "lse_out")):
        _want(t, torch.float32, n)
    _check(lib().lse_merge(_p(o_a), _p(lse_a), _p(o_b), _p(lse_b), _p(o_out), _p(lse_out),
                           rows, d, _stream(stream)))
    return o_out, lse_out


class ReTopK:
    """ReTopK per-layer state (query-support FIFO per head) on the device."""

    def __init__(self, Hq, Hkv, d, K, C_, R, W, tau, T_r, max_len, device="cuda"):
        n = int(lib().retopk_state_size(Hq, d, K, C_))
        if n == 0:
            raise TsaError(-1, "invalid ReTopK sizes")
        self.state = torch.zeros(n, dtype=torch.uint8, device=device)
        self.handle = C.c_void_p()
        _check(lib().retopk_create(C.byref(self.handle), Hq, Hkv, d, K, C_, R, W, float(tau),
                                   T_r, max_len, _p(self.state), n))
        self.Hq, self.Hkv, self.d, self.K, self.C, self.R, self.W = Hq, Hkv, d, K, C_, R, W
        self.cand_cap = R * K + W
        self.workspace = torch.zeros(int(lib().retopk_workspace_size(self.handle)),
                                     dtype=torch.uint8, device=device)

    def __del__(self):
        try:
            if self.handle:
                lib().retopk_destroy(self.handle)
                self.handle = C.c_void_p()
        except Exception:
            pass

    def init(self, prefill_q, prefill_supports, prefill_counts, stream=None):
        _want(prefill_q, torch.bfloat16, "prefill_q")
        _want(prefill_supports, torch.int32, "prefill_supports")
        _want(prefill_counts, torch.int32, "prefill_counts")
        _check(lib().retopk_init(self.handle, _p(prefill_q), _p(prefill_supports),
                                 _p(prefill_counts), _stream(stream)))

    def step(self, q, kv: KV, length: int, scale=None, out=None, support_out=None,
             path_out=None, mcand_out=None, cand_out=None, lse_out=None, stream=None):
        _want(q, torch.bfloat16, "q")
        if scale is None:
            scale = 1.0 / math.sqrt(self.d)
        if out is None:
            out = torch.empty((self.Hq, self.d), dtype=torch.float32, device=q.device)
        _check(lib().retopk_step(self.handle, _p(q), C.byref(kv.struct), int(length),
                                 float(scale), _p(out), _p(support_out), _p(path_out),
                                 _p(mcand_out), _p(cand_out), _p(lse_out), _p(self.workspace),
                                 self.workspace.numel(), _stream(stream)))
        return out

    @staticmethod
    def batched_workspace_size(proto: "ReTopK", n_max: int) -> int:
        return int(lib().retopk_batched_workspace_size(proto.handle, n_max))

    @staticmethod
    def step_batched(handles, q, kv: KV, lens, scale=None, out=None, support_out=None,
                     path_out=None, mcand_out=None, cand_out=None, lse_out=None,
                     workspace=None, stream=None):
        """One step of len(handles) sequences, each with its own state: q bf16
        [n][Hq][128], kv with the n sequences in call order, lens (host ints)."""
        _want(q, torch.bfloat16, "q")
        n = len(handles)
        Hq, d = handles[0].Hq, handles[0].d
        if scale is None:
            scale = 1.0 / math.sqrt(d)
        if out is None:
            out = torch.empty((n, Hq, d), dtype=torch.float32, device=q.device)
        if workspace is None:
            workspace = torch.zeros(ReTopK.batched_workspace_size(handles[0], n),
                                    dtype=torch.uint8, device=q.device)
        hs = (C.c_void_p * n)(*[h.handle.value for h in handles])
        ls = (C.c_int64 * n)(*[int(x) for x in lens])
        _check(lib().retopk_step_batched(hs, n, _p(q), C.byref(kv.struct), ls, float(scale),
                                         _p(out), _p(support_out), _p(path_out), _p(mcand_out),
                                         _p(cand_out), _p(lse_out), _p(workspace),
                                         workspace.numel(), _stream(stream)))
        return out

    def counters(self):
        t, h = C.c_int64(), C.c_int32()
        _check(lib().retopk_get_counters(self.handle, C.byref(t), C.byref(h)))
        return t.value, h.value

    def set_counters(self, t: int, fifo_head: int) -> None:
        _check(lib().retopk_set_counters(self.handle, t, fifo_head))
