"""fp64 CPU oracle for decode-step top-K sparse attention.

TEST INFRASTRUCTURE ONLY.  This package wraps ``oracle.c`` (plain,
single-threaded C in IEEE double) through ctypes.  Only the tests, the smoke
check and the benchmark's CPU-baseline leg may import it; the CUDA library
never does, and the two share no code.

Every function takes bf16 data as numpy ``uint16`` bit patterns (widened
exactly inside the C code) and returns float64 / int64 numpy arrays.

Sources: "RetrievalAttention: Accelerating Long-Context LLM Inference via
Vector Retrieval" (Eq. 1-5, the Flat baseline, the static pattern W) and
"Recall Before You Rank: Similarity-Guided Top-K Reuse for Efficient
Long-Context Attention" (ReTopK method sections 1-5).
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_DIR = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_DIR, "oracle.c")
_SO = os.path.join(_DIR, "_build", "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile oracle.c into _build/liboracle.so with gcc (IEEE, no FMA contraction)."""
    os.makedirs(os.path.dirname(_SO), exist_ok=True)
    if force or not os.path.exists(_SO) or os.path.getmtime(_SO) < max(
        os.path.getmtime(_SRC), os.path.getmtime(os.path.join(_DIR, "oracle.h"))
    ):
        tmp = _SO + f".tmp{os.getpid()}"
        subprocess.check_call(
            ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
             "-fPIC", "-shared", _SRC, "-o", tmp, "-lm"]
        )
        os.replace(tmp, _SO)
    return _SO


class _RetopkState(C.Structure):
    _fields_ = [
        ("Hq", C.c_int), ("d", C.c_int), ("K", C.c_int64), ("C", C.c_int),
        ("R", C.c_int), ("W", C.c_int64), ("tau", C.c_double),
        ("T_r", C.c_int64), ("t", C.c_int64), ("stamp", C.c_int64),
        ("qbar", C.POINTER(C.c_double)), ("sup", C.POINTER(C.c_int64)),
        ("sup_n", C.POINTER(C.c_int64)), ("age", C.POINTER(C.c_int64)),
    ]


class _Margins(C.Structure):
    _fields_ = [("path_abs", C.c_double), ("rho_abs", C.c_double),
                ("topk_rel", C.c_double)]


class _Result(C.Structure):
    _fields_ = [
        ("path", C.c_int), ("own_path", C.c_int), ("max_rho", C.c_double),
        ("adopt_path", C.c_int), ("adopt_cand", C.c_int), ("cand_ok", C.c_int),
        ("sup_ok", C.c_int), ("n_cand", C.c_int64), ("n_sup", C.c_int64),
        ("lse", C.c_double),
    ]


_P = C.c_void_p


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_SO)
            i64, f64, i32 = C.c_int64, C.c_double, C.c_int
            L.orc_bf16_to_f64.argtypes = [C.c_uint16]
            L.orc_bf16_to_f64.restype = f64
            L.orc_in_window.argtypes = [i64, i64, i64, i64]
            L.orc_in_window.restype = i32
            L.orc_scores.argtypes = [_P, _P, i64, i32, i64, f64, _P]
            L.orc_topk.argtypes = [_P, _P, i64, i64, _P]
            L.orc_topk.restype = i64
            L.orc_topk_check.argtypes = [_P, _P, i64, i64, _P, i64, f64]
            L.orc_topk_check.restype = i32
            L.orc_partial.argtypes = [_P, _P, i64, _P, i32, i64, _P, _P, _P, _P]
            L.orc_merge.argtypes = [_P, f64, f64, _P, f64, f64, i32, _P, _P]
            L.orc_decode_head.argtypes = [_P, _P, _P, i64, i32, i64, f64, i64,
                                          i64, i64, _P, _P, _P, _P, _P]
            L.orc_decode_eval_set.argtypes = [_P, _P, i64, i32, i64, i64, i64,
                                              _P, i64, _P, _P]
            L.orc_retopk_create.argtypes = [_P, i32, i32, i64, i32, i32, i64,
                                            f64, i64]
            L.orc_retopk_create.restype = i32
            L.orc_retopk_destroy.argtypes = [_P]
            L.orc_retopk_set_slot.argtypes = [_P, i32, i32, _P, _P, i64]
            L.orc_retopk_step_head.argtypes = [_P, i32, _P, _P, _P, i64, i64,
                                               f64, _P, i32, _P, i64, _P, i64,
                                               _P, _P, _P, _P]
            L.orc_retopk_advance.argtypes = [_P]
            L.orc_q8_fit.argtypes = [_P, i64, i32, i64, _P, _P, _P]
            L.orc_q8_append.argtypes = [_P, i64, i32, i64, _P, _P, _P]
            L.orc_q8_bound.argtypes = [_P, i32, f64, _P]
            L.orc_q8_bound.restype = f64
            _lib = L
    return _lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(C.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError(f"bf16 data must be passed as uint16 bit patterns, got {a.dtype}")
    return a


def _i64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.int64))


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def bf16_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (vectorised, same rule as the C code)."""
    b = np.asarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)


def in_window(i: int, L: int, n_init: int, n_recent: int) -> bool:
    return bool(lib().orc_in_window(i, L, n_init, n_recent))


def scores(q: np.ndarray, k: np.ndarray, scale: float) -> np.ndarray:
    """z_i = scale * q . k_i for the L rows of k ([L][d] uint16)."""
    q, k = _u16(q), _u16(k)
    L, d = k.shape
    z = np.empty(L, np.float64)
    lib().orc_scores(_ptr(q), _ptr(k), L, d, d, scale, _ptr(z))
    return z


def topk(z: np.ndarray, pool, K: int) -> np.ndarray:
    z, pool = _f64(z), _i64(pool)
    out = np.empty(max(K, 1), np.int64)
    n = lib().orc_topk(_ptr(z), _ptr(pool), len(pool), K, _ptr(out))
    return out[:n].copy()


def topk_check(z: np.ndarray, pool, K: int, got, rel: float = 1e-6) -> int:
    z, pool, got = _f64(z), _i64(pool), _i64(got)
    return int(lib().orc_topk_check(_ptr(z), _ptr(pool), len(pool), K,
                                    _ptr(got), len(got), rel))


def partial(z: np.ndarray, idx, v: np.ndarray):
    """(o, m, l, lse) of softmax-weighted V over positions idx."""
    z, idx, v = _f64(z), _i64(idx), _u16(v)
    d = v.shape[1]
    o = np.empty(d, np.float64)
    m, l, lse = C.c_double(), C.c_double(), C.c_double()
    lib().orc_partial(_ptr(z), _ptr(idx), len(idx), _ptr(v), d, d, _ptr(o),
                      C.byref(m), C.byref(l), C.byref(lse))
    return o, m.value, l.value, lse.value


def merge(o1, m1, l1, o2, m2, l2):
    """Eq. 4-5 rescale merge of two disjoint partials given as (o, m, l)."""
    o1, o2 = _f64(o1), _f64(o2)
    o = np.empty_like(o1)
    lse = C.c_double()
    lib().orc_merge(_ptr(o1), m1, l1, _ptr(o2), m2, l2, len(o1), _ptr(o), C.byref(lse))
    return o, lse.value


def decode_head(q, k, v, K: int, n_init: int, n_recent: int, scale: float):
    """One query head of the decode step.  Returns dict(out, lse, sel, z)."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    L, d = k.shape
    out = np.empty(d, np.float64)
    lse = C.c_double()
    sel = np.empty(max(K, 1), np.int64)
    n_sel = C.c_int64()
    z = np.empty(max(L, 1), np.float64)
    lib().orc_decode_head(_ptr(q), _ptr(k), _ptr(v), L, d, d, scale, K, n_init,
                          n_recent, _ptr(out), C.byref(lse), _ptr(sel),
                          C.byref(n_sel), _ptr(z))
    return {"out": out, "lse": lse.value, "sel": sel[: n_sel.value].copy(),
            "z": z[:L].copy()}


def decode_eval_set(z, v, n_init: int, n_recent: int, given):
    """Attention over W_t u given (given disjoint from W_t), from logits z."""
    z, v, given = _f64(z), _u16(v), _i64(given)
    L, d = v.shape
    out = np.empty(d, np.float64)
    lse = C.c_double()
    lib().orc_decode_eval_set(_ptr(z), _ptr(v), L, d, d, n_init, n_recent,
                              _ptr(given), len(given), _ptr(out), C.byref(lse))
    return out, lse.value


def window_positions(L: int, n_init: int, n_recent: int) -> np.ndarray:
    return np.array([i for i in range(L) if in_window(i, L, n_init, n_recent)], np.int64)


class ReTopK:
    """Per-layer ReTopK state of the oracle (query-support FIFO per head)."""

    def __init__(self, Hq, d, K, C_, R, W, tau, T_r,
                 path_abs=1e-6, rho_abs=1e-6, topk_rel=1e-6):
        self._st = _RetopkState()
        rc = lib().orc_retopk_create(C.byref(self._st), Hq, d, K, C_, R, W, tau, T_r)
        if rc != 0:
            raise ValueError("invalid ReTopK parameters")
        self.Hq, self.d, self.K, self.C, self.R, self.W = Hq, d, K, C_, R, W
        self.margins = _Margins(path_abs, rho_abs, topk_rel)

    def __del__(self):
        try:
            lib().orc_retopk_destroy(C.byref(self._st))
        except Exception:
            pass

    @property
    def t(self) -> int:
        return self._st.t

    def set_slot(self, h: int, c: int, q: np.ndarray, support) -> None:
        q, support = _u16(q), _i64(support)
        lib().orc_retopk_set_slot(C.byref(self._st), h, c, _ptr(q), _ptr(support),
                                  len(support))

    def step_head(self, h, q, k, v, scale, other_path=-1, other_cand=None,
                  other_sup=None):
        q, k, v = _u16(q), _u16(k), _u16(v)
        L, d = k.shape
        cand = np.empty(self.R * self.K + self.W + 1, np.int64)
        sup = np.empty(max(self.K, 1), np.int64)
        out = np.empty(d, np.float64)
        res = _Result()
        oc = _i64(other_cand) if other_cand is not None else None
        os_ = _i64(other_sup) if other_sup is not None else None
        lib().orc_retopk_step_head(
            C.byref(self._st), h, _ptr(q), _ptr(k), _ptr(v), L, d, scale,
            C.byref(self.margins), int(other_path),
            _ptr(oc) if oc is not None else None, 0 if oc is None else len(oc),
            _ptr(os_) if os_ is not None else None, 0 if os_ is None else len(os_),
            _ptr(cand), _ptr(sup), _ptr(out), C.byref(res))
        r = {f: getattr(res, f) for f, _ in _Result._fields_}
        r["cand"] = cand[: res.n_cand].copy() if not res.path else None
        r["sup"] = sup[: res.n_sup].copy()
        r["out"] = out
        return r

    def advance(self) -> None:
        lib().orc_retopk_advance(C.byref(self._st))

    # read-only views of the FIFO (for invariant checks)
    def slot_support(self, h: int, c: int) -> np.ndarray:
        hc = h * self.C + c
        n = self._st.sup_n[hc]
        return np.array([self._st.sup[hc * self.K + s] for s in range(n)], np.int64)

    def slot_age(self, h: int, c: int) -> int:
        return int(self._st.age[h * self.C + c])

    def slot_qbar(self, h: int, c: int) -> np.ndarray:
        base = (h * self.C + c) * self.d
        return np.array([self._st.qbar[base + j] for j in range(self.d)])


# ---------------------------------------------------------------------------
# f4. Scalar int8 key quantisation (RetrievalAttention review, Appendix C
# "CPU memory minimization"; per-channel symmetric is the reading of the
# scheme the pages leave open).  Definitions in oracle.h.

def q8_fit(k: np.ndarray):
    """k: [L, d] bf16 bits.  Returns (scale float32[d], codes uint8[L, d]
    offset binary, err float64[d])."""
    k = _u16(k)
    L, d = k.shape
    scale = np.zeros(d, np.float32)
    codes = np.zeros((L, d), np.uint8)
    err = np.zeros(d, np.float64)
    lib().orc_q8_fit(_ptr(k), L, d, d, _ptr(scale), _ptr(codes), _ptr(err))
    return scale, codes, err


def q8_append(k: np.ndarray, scale: np.ndarray, err: np.ndarray):
    """Codes of more rows k [n, d] with fitted scales; returns (codes,
    err updated as a running maximum; the input is not modified)."""
    k = _u16(k)
    n, d = k.shape
    scale = np.ascontiguousarray(scale, np.float32)
    err = _f64(err).copy()
    codes = np.zeros((n, d), np.uint8)
    lib().orc_q8_append(_ptr(k), n, d, d, _ptr(scale), _ptr(codes), _ptr(err))
    return codes, err


def q8_bound(q: np.ndarray, scale: float, err: np.ndarray) -> float:
    """scale * sum_j |q_j| e_j: the bound on a logit's quantisation error."""
    q = _u16(q)
    err = _f64(err)
    return float(lib().orc_q8_bound(_ptr(q), len(q), scale, _ptr(err)))
