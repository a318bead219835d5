"""fp64 CPU oracle for the attention kernels (test infrastructure only).

Only the tests, the package smoke check and the benchmark's CPU-baseline leg
may import this package.  The library itself never does; it shares no code
with it.  The arithmetic lives in ``attn_oracle.c`` (plain C loops in double,
OpenMP over output rows); this module compiles it with gcc on first use and
marshals numpy arrays into it.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, brute-force library softmax, mask enumeration, layout
equivalences, the pages' own parameter arithmetic in ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
# the mutation tests point these at a deliberately broken copy of the source
_SRC = os.environ.get("ATTN_ORACLE_SRC") or os.path.join(_HERE, "attn_oracle.c")
_OUT_DIR = os.environ.get("ATTN_ORACLE_BUILD") or os.path.join(_HERE, "_build")
_LIB = os.path.join(_OUT_DIR, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle into ``oracle/_build/liboracle.so`` (gcc, OpenMP)."""
    os.makedirs(_OUT_DIR, exist_ok=True)
    if (not force and os.path.exists(_LIB)
            and os.path.getmtime(_LIB) >= os.path.getmtime(_SRC)):
        return _LIB
    tmp = _LIB + ".tmp.%d" % os.getpid()
    cmd = ["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-fopenmp", "-fno-fast-math",
           "-ffp-contract=off", _SRC, "-o", tmp, "-lm"]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB)
    return _LIB


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i32, i64, f64 = ctypes.c_int, ctypes.c_long, ctypes.c_double
            lib.oracle_f16_to_double.argtypes = [ctypes.c_uint16]
            lib.oracle_f16_to_double.restype = f64
            lib.oracle_decode.argtypes = [P, i32, P, P, i32, P, P, P, P, i32, i32, i64, i64,
                                          i32, i32, i32, i32, i32, f64, f64,
                                          i32, P, P, P, P, i32, i32]
            lib.oracle_decode.restype = i32
            lib.oracle_prefill.argtypes = [P, P, P, i32, i32, i32, i32, i32, i32, f64, f64,
                                           i32, P, P, P, P, i32]
            lib.oracle_prefill.restype = i32
            lib.oracle_prefill_paged.argtypes = [P, P, P, P, P, P, i32, i32, i64, i32, i32, i32, i32,
                                                 i32, f64, f64, i32, P, P, P, P, i32]
            lib.oracle_prefill_paged.restype = i32
            lib.oracle_decode_tiered.argtypes = [P, i32, P, P, i32, P, P, P, P, i32, i32, i64, i64,
                                                 P, P, P, P, i64,
                                                 i32, i32, i32, i32, i32, f64, f64,
                                                 i32, P, P, P, P, i32]
            lib.oracle_decode_tiered.restype = i32
            lib.oracle_max_threads.restype = i32
            _lib = lib
    return _lib


def _np(x):
    """torch tensor (any device) or array -> contiguous numpy array."""
    if x is None:
        return None
    if hasattr(x, "detach"):
        x = x.detach().cpu().contiguous().numpy()
    return np.ascontiguousarray(x)


def _ptr(a):
    return None if a is None else a.ctypes.data_as(ctypes.c_void_p)


def _f16_bits(a):
    a = _np(a)
    if a.dtype == np.float16:
        return a.view(np.uint16)
    assert a.dtype == np.uint16, a.dtype
    return a


def _q_arg(q):
    """(array, q_f32): f16 queries as their bits, f32 queries as binary32 values."""
    a = _np(q)
    if a.dtype == np.float32:
        return a, 1
    return _f16_bits(a), 0


def f16_to_double(bits: int) -> float:
    return float(_load().oracle_f16_to_double(int(bits) & 0xFFFF))


def max_threads() -> int:
    return int(_load().oracle_max_threads())


def decode(case, rows=None, n_threads: int = 0):
    """Oracle decode for a DecodeCase-like object.

    rows: None for every (b, h) in row-major order, or a list of (b, h) pairs.
    Returns (out float64 [n, D], lse float64 [n]) with lse in natural-log units.
    """
    lib = _load()
    q, q_f32 = _q_arg(case.q)
    if case.int8:
        k = _np(case.k).astype(np.int8, copy=False)
        v = _np(case.v).astype(np.int8, copy=False)
        ks, vs = _f16_bits(case.k_scales), _f16_bits(case.v_scales)
    else:
        k, v = _f16_bits(case.k), _f16_bits(case.v)
        ks = vs = None
    kv_len = _np(case.kv_len).astype(np.int32, copy=False)
    pt = None if case.page_table is None else _np(case.page_table).astype(np.int32, copy=False)
    if rows is None:
        n_rows, rb, rh = -1, None, None
        n = case.batch * case.n_heads
    else:
        rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
        n_rows = n = rows.shape[0]
        rb, rh = np.ascontiguousarray(rows[:, 0]), np.ascontiguousarray(rows[:, 1])
    out = np.zeros((n, case.head_dim), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    n_pages = int(case.k.shape[0]) if pt is not None else 0
    rc = lib.oracle_decode(_ptr(q), q_f32, _ptr(k), _ptr(v), int(bool(case.int8)), _ptr(ks), _ptr(vs),
                           _ptr(kv_len), _ptr(pt), int(case.page_size or 0),
                           int(case.max_pages or 0), int(case.cap), n_pages,
                           case.batch, case.n_heads, case.n_kv_heads, case.head_dim,
                           int(case.window), float(case.softcap), float(case.scale),
                           n_rows, _ptr(rb), _ptr(rh), _ptr(out), _ptr(lse), int(n_threads),
                           int(getattr(case, "ring", 0) or 0))
    if rc != 0:
        raise ValueError("oracle_decode rejected its arguments")
    return out, lse


def prefill(case, rows=None, n_threads: int = 0):
    """Oracle prefill / vision attention for a PrefillCase-like object.

    rows: None for every (i, h) in row-major order, or a list of (i, h) pairs.
    Returns (out float64 [n, D], lse float64 [n]).
    """
    lib = _load()
    q, k, v = _f16_bits(case.q), _f16_bits(case.k), _f16_bits(case.v)
    if rows is None:
        n_rows, ri, rh = -1, None, None
        n = case.seq_len * case.n_heads
    else:
        rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
        n_rows = n = rows.shape[0]
        ri, rh = np.ascontiguousarray(rows[:, 0]), np.ascontiguousarray(rows[:, 1])
    out = np.zeros((n, case.head_dim), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.oracle_prefill(_ptr(q), _ptr(k), _ptr(v), case.seq_len, case.n_heads,
                            case.n_kv_heads, case.head_dim, int(bool(case.causal)),
                            int(case.window), float(case.softcap), float(case.scale),
                            n_rows, _ptr(ri), _ptr(rh), _ptr(out), _ptr(lse), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_prefill rejected its arguments")
    return out, lse


def prefill_paged(case, rows=None, n_threads: int = 0):
    """Oracle chunked prefill / multi-token decode for a ChunkCase-like object.

    rows: None for every (packed query row, head) in row-major order, or a list
    of (row, head) pairs.  Returns (out float64 [n, D], lse float64 [n]).
    """
    lib = _load()
    q, k, v = _f16_bits(case.q), _f16_bits(case.k), _f16_bits(case.v)
    q_start = _np(case.q_start).astype(np.int32, copy=False)
    kv_len = _np(case.kv_len).astype(np.int32, copy=False)
    pt = _np(case.page_table).astype(np.int32, copy=False)
    total_q = int(q_start[-1])
    if rows is None:
        n_rows, rr, rh = -1, None, None
        n = total_q * case.n_heads
    else:
        rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
        n_rows = n = rows.shape[0]
        rr, rh = np.ascontiguousarray(rows[:, 0]), np.ascontiguousarray(rows[:, 1])
    out = np.zeros((n, case.head_dim), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    rc = lib.oracle_prefill_paged(_ptr(q), _ptr(k), _ptr(v), _ptr(q_start), _ptr(kv_len), _ptr(pt),
                                  int(case.page_size), int(case.max_pages), int(case.k.shape[0]),
                                  case.batch, case.n_heads, case.n_kv_heads, case.head_dim,
                                  int(case.window), float(case.softcap), float(case.scale),
                                  n_rows, _ptr(rr), _ptr(rh), _ptr(out), _ptr(lse), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_prefill_paged rejected its arguments")
    return out, lse


def decode_tiered(case, rows=None, n_threads: int = 0):
    """Oracle tiered decode for a TieredCase-like object (cold cache + f16 hot ring).

    rows: None for every (b, h) in row-major order, or a list of (b, h) pairs.
    Returns (out float64 [n, D], lse float64 [n]) with lse in natural-log units.
    """
    lib = _load()
    q, q_f32 = _q_arg(case.q)
    if case.int8:
        ck = _np(case.k).astype(np.int8, copy=False)
        cv = _np(case.v).astype(np.int8, copy=False)
        cks, cvs = _f16_bits(case.k_scales), _f16_bits(case.v_scales)
    else:
        ck, cv = _f16_bits(case.k), _f16_bits(case.v)
        cks = cvs = None
    cold_len = _np(case.kv_len).astype(np.int32, copy=False)
    pt = None if case.page_table is None else _np(case.page_table).astype(np.int32, copy=False)
    hk, hv = _f16_bits(case.hot_k), _f16_bits(case.hot_v)
    hot_len = _np(case.hot_len).astype(np.int32, copy=False)
    hot_start = _np(case.hot_start).astype(np.int32, copy=False)
    if rows is None:
        n_rows, rb, rh = -1, None, None
        n = case.batch * case.n_heads
    else:
        rows = np.asarray(rows, dtype=np.int32).reshape(-1, 2)
        n_rows = n = rows.shape[0]
        rb, rh = np.ascontiguousarray(rows[:, 0]), np.ascontiguousarray(rows[:, 1])
    out = np.zeros((n, case.head_dim), dtype=np.float64)
    lse = np.zeros((n,), dtype=np.float64)
    n_pages = int(case.k.shape[0]) if case.page_table is not None else 0
    rc = lib.oracle_decode_tiered(_ptr(q), q_f32, _ptr(ck), _ptr(cv), int(case.int8), _ptr(cks), _ptr(cvs),
                                  _ptr(cold_len), _ptr(pt), int(case.page_size), int(case.max_pages or 0),
                                  int(case.cap), n_pages, _ptr(hk), _ptr(hv), _ptr(hot_len), _ptr(hot_start),
                                  int(case.hot_ring), case.batch, case.n_heads, case.n_kv_heads, case.head_dim,
                                  int(case.window), float(case.softcap), float(case.scale),
                                  n_rows, _ptr(rb), _ptr(rh), _ptr(out), _ptr(lse), int(n_threads))
    if rc != 0:
        raise ValueError("oracle_decode_tiered rejected its arguments")
    return out, lse
