"""CPU oracle for the DSA layer -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the benchmark's CPU-baseline
leg import this package.  The product library never loads it, and it shares
no code with the CUDA path.  The arithmetic lives in ``oracle.c`` (plain C,
fp64 accumulation, OpenMP over independent query rows); this module only
compiles it with gcc and marshals numpy arrays.

bf16 arrays are passed as numpy uint16 arrays of raw bit patterns.

Parity pins: every function here is checked in ``tests/test_oracle_pins.py``
against something other than itself (exact integer identities, a textbook
library routine for dense causal attention and its autograd gradient,
brute-force subset enumeration for the top-k, finite differences, and the
hand-worked fixtures under ``tests/golden/``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None


class OracleError(RuntimeError):
    pass


def build(force: bool = False) -> str:
    """Compile liboracle.so next to oracle.c (gcc, OpenMP, no FMA contraction)."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["gcc", "-O2", "-fopenmp", "-ffp-contract=off", "-fPIC", "-shared",
                               "-o", tmp, _SRC, "-lm"])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            i64, vp, dbl = ctypes.c_int64, ctypes.c_void_p, ctypes.c_double
            lib.oracle_num_threads.argtypes = []
            lib.oracle_pool_keys.argtypes = [vp, i64, i64, vp]
            lib.oracle_index_scores.argtypes = [vp, vp, vp, i64, i64, i64, vp, i64, i64, vp]
            lib.oracle_topk.argtypes = [vp, i64, i64, vp, vp]
            lib.oracle_index_topk.argtypes = [vp, vp, vp, i64, i64, i64, i64, vp, i64, vp, vp]
            lib.oracle_attn_fwd.argtypes = [vp, vp, vp, vp, i64, i64, i64, i64, dbl, vp, i64, vp, vp]
            lib.oracle_attn_bwd_dq.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, dbl, vp, i64, vp]
            lib.oracle_attn_bwd_dkdv.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, dbl, vp, i64, vp, vp]
            lib.oracle_attn_bwd_rows.argtypes = [vp, vp, vp, vp, vp, i64, i64, i64, i64, dbl, vp, i64, vp, vp, vp]
            for name in ("oracle_attn_bwd_rows", "oracle_num_threads", "oracle_pool_keys", "oracle_index_scores", "oracle_topk",
                         "oracle_index_topk", "oracle_attn_fwd", "oracle_attn_bwd_dq", "oracle_attn_bwd_dkdv"):
                getattr(lib, name).restype = ctypes.c_int
            _lib = lib
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _check(rc):
    if rc != 0:
        raise OracleError({-1: "bad argument", -2: "malformed pool_idx row", -3: "out of memory"}.get(rc, rc))


def num_threads() -> int:
    return _load().oracle_num_threads()


def _rows(rows, S):
    return _c(np.arange(S) if rows is None else rows, np.int64)


def pool_keys(k_idx: np.ndarray) -> np.ndarray:
    """Khat [S//4, Di] fp32 from k_idx [S, Di] (bf16 bits)."""
    k_idx = _c(k_idx, np.uint16)
    S, Di = k_idx.shape
    out = np.empty((S // 4, Di), np.float32)
    _check(_load().oracle_pool_keys(k_idx.ctypes.data, S, Di, out.ctypes.data))
    return out


def index_scores(q_idx, k_idx, w, rows=None) -> np.ndarray:
    """Scores [len(rows), max(rows)//4] (double); entries p >= row//4 are NaN."""
    q_idx, k_idx, w = _c(q_idx, np.uint16), _c(k_idx, np.uint16), _c(w, np.float32)
    S, Hi, Di = q_idx.shape
    rows = _rows(rows, S)
    stride = max(1, int(rows.max()) // 4 if rows.size else 1)
    out = np.full((rows.size, stride), np.nan, np.float64)
    _check(_load().oracle_index_scores(q_idx.ctypes.data, k_idx.ctypes.data, w.ctypes.data, S, Hi, Di,
                                       rows.ctypes.data, rows.size, stride, out.ctypes.data))
    return out


def topk(scores: np.ndarray, k: int):
    """Top-k of one score row (double) -> (pool_idx [k] int32, kth fp32)."""
    scores = _c(scores, np.float64)
    out = np.empty(k, np.int32)
    kth = np.empty(1, np.float32)
    _check(_load().oracle_topk(scores.ctypes.data, scores.size, k, out.ctypes.data, kth.ctypes.data))
    return out, float(kth[0])


def index_topk(q_idx, k_idx, w, topk_: int, rows=None):
    """Indexer + top-k -> (pool_idx [len(rows), topk] int32, kth [len(rows)] fp32)."""
    q_idx, k_idx, w = _c(q_idx, np.uint16), _c(k_idx, np.uint16), _c(w, np.float32)
    S, Hi, Di = q_idx.shape
    rows = _rows(rows, S)
    out = np.empty((rows.size, topk_), np.int32)
    kth = np.empty(rows.size, np.float32)
    _check(_load().oracle_index_topk(q_idx.ctypes.data, k_idx.ctypes.data, w.ctypes.data, S, Hi, Di, topk_,
                                     rows.ctypes.data, rows.size, out.ctypes.data, kth.ctypes.data))
    return out, kth


def attn_fwd(q, k, v, pool_idx, scale=0.0, rows=None):
    """Sparse attention forward -> (o [n, Hq, D] double, lse [n, Hq] double)."""
    q, k, v, pool_idx = _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16), _c(pool_idx, np.int32)
    S, Hq, D = q.shape
    topk_ = pool_idx.shape[1]
    rows = _rows(rows, S)
    o = np.empty((rows.size, Hq, D), np.float64)
    lse = np.empty((rows.size, Hq), np.float64)
    _check(_load().oracle_attn_fwd(q.ctypes.data, k.ctypes.data, v.ctypes.data, pool_idx.ctypes.data, S, Hq, D,
                                   topk_, float(scale), rows.ctypes.data, rows.size, o.ctypes.data, lse.ctypes.data))
    return o, lse


def attn_bwd_dq(dO, q, k, v, pool_idx, scale=0.0, rows=None):
    """dq [n, Hq, D] (double) for the listed query rows."""
    dO, q, k, v = _c(dO, np.uint16), _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    pool_idx = _c(pool_idx, np.int32)
    S, Hq, D = q.shape
    rows = _rows(rows, S)
    dq = np.empty((rows.size, Hq, D), np.float64)
    _check(_load().oracle_attn_bwd_dq(dO.ctypes.data, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                      pool_idx.ctypes.data, S, Hq, D, pool_idx.shape[1], float(scale),
                                      rows.ctypes.data, rows.size, dq.ctypes.data))
    return dq


def attn_bwd_dkdv(dO, q, k, v, pool_idx, scale=0.0, key_rows=None):
    """(dk, dv) [n, D] (double) for the listed key rows."""
    dO, q, k, v = _c(dO, np.uint16), _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    pool_idx = _c(pool_idx, np.int32)
    S, Hq, D = q.shape
    key_rows = _rows(key_rows, S)
    dk = np.empty((key_rows.size, D), np.float64)
    dv = np.empty((key_rows.size, D), np.float64)
    _check(_load().oracle_attn_bwd_dkdv(dO.ctypes.data, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                        pool_idx.ctypes.data, S, Hq, D, pool_idx.shape[1], float(scale),
                                        key_rows.ctypes.data, key_rows.size, dk.ctypes.data, dv.ctypes.data))
    return dk, dv


def attn_bwd_rows(dO, q, k, v, pool_idx, scale=0.0, rows=None):
    """Backward of the listed query rows -> (dq [n, Hq, D], dk [S, D], dv [S, D]) in double;
    dk/dv hold only those rows' contributions (all rows: the whole backward)."""
    dO, q, k, v = _c(dO, np.uint16), _c(q, np.uint16), _c(k, np.uint16), _c(v, np.uint16)
    pool_idx = _c(pool_idx, np.int32)
    S, Hq, D = q.shape
    rows = _rows(rows, S)
    dq = np.empty((rows.size, Hq, D), np.float64)
    dk = np.zeros((S, D), np.float64)
    dv = np.zeros((S, D), np.float64)
    _check(_load().oracle_attn_bwd_rows(dO.ctypes.data, q.ctypes.data, k.ctypes.data, v.ctypes.data,
                                        pool_idx.ctypes.data, S, Hq, D, pool_idx.shape[1], float(scale),
                                        rows.ctypes.data, rows.size, dq.ctypes.data, dk.ctypes.data, dv.ctypes.data))
    return dq, dk, dv
