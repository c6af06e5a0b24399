"""Float64 CPU oracle for the exact attention forward pass (TEST INFRASTRUCTURE).

Only the tests, the smoke check and the benchmark's CPU-baseline leg may import
this package. It is the plain definition that the CUDA library is checked
against and shares no code with it. The arithmetic lives in ``fa_oracle.cpp``
(C++, IEEE double, no fast-math); this module only builds and marshals.

Every function here is pinned by ``tests/test_oracle_pins.py`` against values
the pages print, closed forms, invariants and independent library routines.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "fa_oracle.cpp")
_LIB = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile fa_oracle.cpp into liboracle.so (portable flags: no -march, no fast-math)."""
    if force or not os.path.exists(_LIB) or os.path.getmtime(_LIB) < os.path.getmtime(_SRC):
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["g++", "-O2", "-std=c++17", "-fPIC", "-shared", "-pthread",
               "-fno-fast-math", "-ffp-contract=off", _SRC, "-o", tmp]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    if _lib is None:
        build()
        lib = ctypes.CDLL(_LIB)
        dp = ctypes.POINTER(ctypes.c_double)
        i64p = ctypes.POINTER(ctypes.c_int64)
        lib.fa_oracle_hw_threads.restype = ctypes.c_int
        lib.fa_oracle_attention.restype = ctypes.c_int
        lib.fa_oracle_attention.argtypes = [dp, dp, dp] + [ctypes.c_int] * 5 + [
            ctypes.c_double, ctypes.c_int, dp, dp, ctypes.c_int]
        lib.fa_oracle_attention_rows.restype = ctypes.c_int
        lib.fa_oracle_attention_rows.argtypes = [dp, dp, dp] + [ctypes.c_int] * 5 + [
            ctypes.c_double, ctypes.c_int, i64p, ctypes.c_int64, dp, dp, ctypes.c_int]
        lib.fa_oracle_probs.restype = None
        lib.fa_oracle_probs.argtypes = [dp, dp, ctypes.c_int, ctypes.c_int, ctypes.c_int,
                                        ctypes.c_double, ctypes.c_int, dp]
        lib.fa_oracle_online_softmax.restype = ctypes.c_int
        lib.fa_oracle_online_softmax.argtypes = [dp, ctypes.c_int, ctypes.c_int, dp, dp, dp, dp]
        lib.fa_oracle_merge.restype = None
        lib.fa_oracle_merge.argtypes = [ctypes.c_double, ctypes.c_double, dp,
                                        ctypes.c_double, ctypes.c_double, dp, ctypes.c_int,
                                        dp, dp, dp]
        lib.fa_oracle_block_state.restype = None
        lib.fa_oracle_block_state.argtypes = [dp, dp, dp, ctypes.c_int, ctypes.c_int64,
                                              ctypes.c_int, ctypes.c_int, ctypes.c_double,
                                              ctypes.c_int, dp, dp, dp]
        lib.fa_oracle_attention_bwd.restype = ctypes.c_int
        lib.fa_oracle_attention_bwd.argtypes = [dp, dp, dp, dp] + [ctypes.c_int] * 5 + [
            ctypes.c_double, ctypes.c_int, dp, dp, dp, ctypes.c_int]
        _declare_dropout(lib)
        _lib = lib
    return _lib


def _declare_dropout(lib):
    dp = ctypes.POINTER(ctypes.c_double)
    i64p = ctypes.POINTER(ctypes.c_int64)
    u32p = ctypes.POINTER(ctypes.c_uint32)
    u64, u32 = ctypes.c_uint64, ctypes.c_uint32
    lib.fa_oracle_philox4x32_10.restype = None
    lib.fa_oracle_philox4x32_10.argtypes = [u32p, u32p, u32p]
    lib.fa_oracle_dropout_threshold.restype = ctypes.c_int
    lib.fa_oracle_dropout_threshold.argtypes = [ctypes.c_double]
    lib.fa_oracle_dropout_keep.restype = ctypes.c_int
    lib.fa_oracle_dropout_keep.argtypes = [ctypes.c_int] * 4 + [ctypes.c_double, u64, u32,
                                                                ctypes.POINTER(ctypes.c_uint8)]
    lib.fa_oracle_attention_dropout.restype = ctypes.c_int
    lib.fa_oracle_attention_dropout.argtypes = [dp, dp, dp] + [ctypes.c_int] * 5 + [
        ctypes.c_double, ctypes.c_int, ctypes.c_double, u64, u32, dp, dp, ctypes.c_int]
    lib.fa_oracle_attention_dropout_rows.restype = ctypes.c_int
    lib.fa_oracle_attention_dropout_rows.argtypes = [dp, dp, dp] + [ctypes.c_int] * 5 + [
        ctypes.c_double, ctypes.c_int, ctypes.c_double, u64, u32, i64p, ctypes.c_int64, dp, dp,
        ctypes.c_int]
    lib.fa_oracle_attention_bwd_dropout.restype = ctypes.c_int
    lib.fa_oracle_attention_bwd_dropout.argtypes = [dp, dp, dp, dp] + [ctypes.c_int] * 5 + [
        ctypes.c_double, ctypes.c_int, ctypes.c_double, u64, u32, dp, dp, dp, ctypes.c_int]


_EXPORTS = ("fa_oracle_hw_threads", "fa_oracle_attention", "fa_oracle_attention_rows",
            "fa_oracle_probs", "fa_oracle_online_softmax", "fa_oracle_merge",
            "fa_oracle_block_state", "fa_oracle_attention_bwd", "fa_oracle_philox4x32_10",
            "fa_oracle_dropout_threshold", "fa_oracle_dropout_keep",
            "fa_oracle_attention_dropout", "fa_oracle_attention_dropout_rows",
            "fa_oracle_attention_bwd_dropout")


class using_library:
    """Context manager: run the wrappers of this module against another build of the
    oracle (the mutation tests load deliberately broken copies this way)."""

    def __init__(self, path: str):
        self.path = path

    def __enter__(self):
        global _lib
        _load()
        self._saved = _lib
        lib = ctypes.CDLL(self.path)
        for name in _EXPORTS:
            f, g = getattr(lib, name), getattr(self._saved, name)
            f.restype, f.argtypes = g.restype, g.argtypes
        _lib = lib
        return self

    def __exit__(self, *exc):
        global _lib
        _lib = self._saved
        return False


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(np.asarray(a, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.POINTER(ctypes.c_double))


def hw_threads() -> int:
    return int(_load().fa_oracle_hw_threads())


def attention(Q, K, V, scale: float, causal: bool, nthreads: int = 0):
    """O [B,H,Nq,d], L [B,H,Nq] by the plain definition. Q: [B,H,Nq,d]; K, V: [B,H,Nk,d]."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    assert K.shape == (B, H, Nk, d) and V.shape == (B, H, Nk, d)
    O = np.empty((B, H, Nq, d), np.float64)
    L = np.empty((B, H, Nq), np.float64)
    _load().fa_oracle_attention(_ptr(Q), _ptr(K), _ptr(V), B, H, Nq, Nk, d, float(scale),
                                int(bool(causal)), _ptr(O), _ptr(L), int(nthreads))
    return O, L


def attention_rows(Q, K, V, scale: float, causal: bool, rows, nthreads: int = 0):
    """The definition on selected flat rows r = (b*H + h)*Nq + i. Returns O [n,d], L [n]."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert rows.ndim == 1 and (rows.size == 0 or (rows.min() >= 0 and rows.max() < B * H * Nq))
    n = rows.size
    O = np.empty((n, d), np.float64)
    L = np.empty((n,), np.float64)
    _load().fa_oracle_attention_rows(_ptr(Q), _ptr(K), _ptr(V), B, H, Nq, Nk, d, float(scale),
                                     int(bool(causal)),
                                     rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n,
                                     _ptr(O), _ptr(L), int(nthreads))
    return O, L


def probs(Q, K, scale: float, causal: bool):
    """P [Nq, Nk] of one head. Q: [Nq,d], K: [Nk,d]."""
    Q, K = _f64(Q), _f64(K)
    Nq, d = Q.shape
    Nk = K.shape[0]
    P = np.empty((Nq, Nk), np.float64)
    _load().fa_oracle_probs(_ptr(Q), _ptr(K), Nq, Nk, d, float(scale), int(bool(causal)), _ptr(P))
    return P


def online_softmax(x, block: int):
    """(m, l, m_trace, l_trace) of the online softmax recurrence over chunks of `block`."""
    x = _f64(x).ravel()
    n = x.size
    nchunks = (n + block - 1) // block
    mt = np.empty(max(nchunks, 1), np.float64)
    lt = np.empty(max(nchunks, 1), np.float64)
    m = ctypes.c_double()
    l = ctypes.c_double()
    c = _load().fa_oracle_online_softmax(_ptr(x), n, int(block), ctypes.byref(m), ctypes.byref(l),
                                         _ptr(mt), _ptr(lt))
    return m.value, l.value, mt[:c].copy(), lt[:c].copy()


def merge(a, b):
    """Merge two states (m, d, o) -> (m, d, o); o may be None for the (m, d) pair."""
    ma, da, oa = a
    mb, db, ob = b
    if oa is None:
        oa = np.zeros(0)
        ob = np.zeros(0)
    oa, ob = _f64(oa).ravel(), _f64(ob).ravel()
    assert oa.size == ob.size
    out = np.empty(oa.size, np.float64)
    m = ctypes.c_double()
    d = ctypes.c_double()
    _load().fa_oracle_merge(float(ma), float(da), _ptr(oa), float(mb), float(db), _ptr(ob),
                            oa.size, ctypes.byref(m), ctypes.byref(d), _ptr(out))
    return m.value, d.value, out


def block_state(q, K, V, i: int, j0: int, j1: int, scale: float, causal: bool):
    """The (m, d, o~) state of keys [j0, j1) for query row i (q: [d], K, V: [Nk, d])."""
    q, K, V = _f64(q).ravel(), _f64(K), _f64(V)
    d = q.size
    out = np.empty(d, np.float64)
    m = ctypes.c_double()
    den = ctypes.c_double()
    _load().fa_oracle_block_state(_ptr(q), _ptr(K), _ptr(V), d, int(i), int(j0), int(j1),
                                  float(scale), int(bool(causal)), ctypes.byref(m),
                                  ctypes.byref(den), _ptr(out))
    return m.value, den.value, out


def attention_bwd(Q, K, V, dO, scale: float, causal: bool, nthreads: int = 0):
    """(dQ, dK, dV) of the attention forward for the upstream gradient dO (float64)."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    assert K.shape == V.shape == (B, H, Nk, d) and dO.shape == Q.shape
    dQ = np.empty_like(Q)
    dK = np.empty_like(K)
    dV = np.empty_like(V)
    _load().fa_oracle_attention_bwd(_ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, H, Nq, Nk, d,
                                    float(scale), int(bool(causal)), _ptr(dQ), _ptr(dK), _ptr(dV),
                                    int(nthreads))
    return dQ, dK, dV


def philox4x32_10(ctr, key):
    """The four 32-bit output words of Philox-4x32-10 for one counter and key."""
    c = np.ascontiguousarray(np.asarray(ctr, dtype=np.uint32))
    k = np.ascontiguousarray(np.asarray(key, dtype=np.uint32))
    assert c.shape == (4,) and k.shape == (2,)
    out = np.zeros(4, np.uint32)
    u32p = ctypes.POINTER(ctypes.c_uint32)
    _load().fa_oracle_philox4x32_10(c.ctypes.data_as(u32p), k.ctypes.data_as(u32p),
                                    out.ctypes.data_as(u32p))
    return out


def dropout_threshold(p_drop: float) -> int:
    """The 8-bit threshold t of p_drop, or -1 when p_drop is out of range."""
    return int(_load().fa_oracle_dropout_threshold(float(p_drop)))


def dropout_keep(B: int, H: int, Nq: int, Nk: int, p_drop: float, seed: int, offset: int):
    """The keep mask [B,H,Nq,Nk] (uint8, 1 = kept) of the dropout definition."""
    keep = np.zeros((B, H, Nq, Nk), np.uint8)
    rc = _load().fa_oracle_dropout_keep(int(B), int(H), int(Nq), int(Nk), float(p_drop),
                                        int(seed), int(offset),
                                        keep.ctypes.data_as(ctypes.POINTER(ctypes.c_uint8)))
    if rc != 0:
        raise ValueError(f"invalid dropout probability {p_drop}")
    return keep


def attention_dropout(Q, K, V, scale: float, causal: bool, p_drop: float, seed: int,
                      offset: int, nthreads: int = 0):
    """O [B,H,Nq,d], L [B,H,Nq] of attention with dropout (the mask of seed/offset)."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    assert K.shape == (B, H, Nk, d) and V.shape == (B, H, Nk, d)
    O = np.empty((B, H, Nq, d), np.float64)
    L = np.empty((B, H, Nq), np.float64)
    rc = _load().fa_oracle_attention_dropout(_ptr(Q), _ptr(K), _ptr(V), B, H, Nq, Nk, d,
                                             float(scale), int(bool(causal)), float(p_drop),
                                             int(seed), int(offset), _ptr(O), _ptr(L),
                                             int(nthreads))
    if rc < 0:
        raise ValueError(f"invalid dropout probability {p_drop}")
    return O, L


def attention_dropout_rows(Q, K, V, scale: float, causal: bool, p_drop: float, seed: int,
                           offset: int, rows, nthreads: int = 0):
    """attention_dropout on selected flat rows r = (b*H + h)*Nq + i: O [n,d], L [n]."""
    Q, K, V = _f64(Q), _f64(K), _f64(V)
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64))
    assert rows.ndim == 1 and (rows.size == 0 or (rows.min() >= 0 and rows.max() < B * H * Nq))
    n = rows.size
    O = np.empty((n, d), np.float64)
    L = np.empty((n,), np.float64)
    rc = _load().fa_oracle_attention_dropout_rows(
        _ptr(Q), _ptr(K), _ptr(V), B, H, Nq, Nk, d, float(scale), int(bool(causal)),
        float(p_drop), int(seed), int(offset),
        rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)), n, _ptr(O), _ptr(L), int(nthreads))
    if rc < 0:
        raise ValueError(f"invalid dropout probability {p_drop}")
    return O, L


def attention_bwd_dropout(Q, K, V, dO, scale: float, causal: bool, p_drop: float, seed: int,
                          offset: int, nthreads: int = 0):
    """(dQ, dK, dV) of the dropout forward (mask of seed/offset) for upstream gradient dO."""
    Q, K, V, dO = _f64(Q), _f64(K), _f64(V), _f64(dO)
    B, H, Nq, d = Q.shape
    Nk = K.shape[2]
    assert K.shape == V.shape == (B, H, Nk, d) and dO.shape == Q.shape
    dQ = np.empty_like(Q)
    dK = np.empty_like(K)
    dV = np.empty_like(V)
    rc = _load().fa_oracle_attention_bwd_dropout(
        _ptr(Q), _ptr(K), _ptr(V), _ptr(dO), B, H, Nq, Nk, d, float(scale), int(bool(causal)),
        float(p_drop), int(seed), int(offset), _ptr(dQ), _ptr(dK), _ptr(dV), int(nthreads))
    if rc < 0:
        raise ValueError(f"invalid dropout probability {p_drop}")
    return dQ, dK, dV
