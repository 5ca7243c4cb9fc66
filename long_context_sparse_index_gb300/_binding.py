"""ctypes binding of libdsa (argument marshalling only).

Every function here checks tensor dtypes, shapes and devices, allocates
outputs and workspace with torch when the caller does not pass them, and
calls the C entry point of the same name on the current CUDA stream.  All
arithmetic runs in libdsa's CUDA kernels; there is no other code path, and a
missing library raises instead of falling back.
"""
from __future__ import annotations

import ctypes
import os
import threading

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libdsa.so")

DSA_OK, DSA_ERR_INVALID_ARG, DSA_ERR_UNSUPPORTED, DSA_ERR_WORKSPACE = 0, 1, 2, 3
DSA_ERR_CUDA, DSA_ERR_TIMEOUT, DSA_ERR_INTERNAL = 4, 5, 6
STATUS_NAMES = {0: "DSA_OK", 1: "DSA_ERR_INVALID_ARG", 2: "DSA_ERR_UNSUPPORTED", 3: "DSA_ERR_WORKSPACE",
                4: "DSA_ERR_CUDA", 5: "DSA_ERR_TIMEOUT", 6: "DSA_ERR_INTERNAL"}

# every symbol the C header declares
EXPORTED = ("dsa_index_topk_workspace", "dsa_index_topk", "dsa_sparse_attn_fwd", "dsa_sparse_attn_bwd_workspace",
            "dsa_sparse_attn_bwd", "dsa_sync_status", "dsa_clear_status", "dsa_last_error", "dsa_version",
            "dsa_profile_enable", "dsa_profile_read", "dsa_launch_count", "dsa_launch_count_reset",
            "dsa_index_topk_noalloc", "dsa_sparse_attn_fwd_range", "dsa_sparse_attn_bwd_range",
            "dsa_zigzag_ranges", "dsa_index_topk_varlen_workspace", "dsa_index_topk_varlen",
            "dsa_sparse_attn_fwd_varlen", "dsa_sparse_attn_bwd_varlen_workspace", "dsa_sparse_attn_bwd_varlen",
            "dsa_sparse_attn_bwd_deterministic_workspace", "dsa_sparse_attn_bwd_deterministic",
            "dsa_index_topk_stats", "dsa_measure_l2", "dsa_index_topk_workspace_slots", "dsa_trace_configure",
            "dsa_last_kernel_config", "dsa_sparse_attn_fwd_tc", "dsa_measure_umma",
            "dsa_fwd_tc_profile", "dsa_measure_fold")

_lock = threading.Lock()
_lib = None


class DsaError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


def _configure(lib):
    """Declares the argument and result types of every C ABI entry point."""
    i64, i32, vp, sz, f32 = ctypes.c_int64, ctypes.c_int, ctypes.c_void_p, ctypes.c_size_t, ctypes.c_float
    lib.dsa_index_topk_workspace.argtypes = [i64, i32, i32, i32, i32]
    lib.dsa_index_topk_workspace.restype = sz
    lib.dsa_index_topk_workspace_slots.argtypes = [i64, i32, i32, i32, i32, i32]
    lib.dsa_index_topk_workspace_slots.restype = sz
    lib.dsa_index_topk.argtypes = [vp, vp, vp, i64, i32, i32, i32, i32, i64, i64, vp, vp, sz, vp]
    lib.dsa_sparse_attn_fwd.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, f32, vp, vp, vp]
    lib.dsa_sparse_attn_fwd_tc.argtypes = [vp, vp, vp, vp, i64, i32, i32, i32, f32, vp, vp, vp]
    lib.dsa_sparse_attn_bwd_workspace.argtypes = [i64, i32, i32]
    lib.dsa_sparse_attn_bwd_workspace.restype = sz
    lib.dsa_sparse_attn_bwd.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, f32, vp, vp, vp, vp,
                                        sz, vp]
    lib.dsa_sparse_attn_fwd_range.argtypes = [vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, f32, vp, vp, vp]
    lib.dsa_sparse_attn_bwd_range.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i64, i64, i32, i32, i32, f32,
                                              vp, vp, vp, vp, sz, vp]
    lib.dsa_zigzag_ranges.argtypes = [i64, i32, i32, ctypes.POINTER(ctypes.c_int64)]
    for f in (lib.dsa_sparse_attn_fwd_range, lib.dsa_sparse_attn_bwd_range, lib.dsa_zigzag_ranges):
        f.restype = ctypes.c_int
    pi64 = ctypes.POINTER(ctypes.c_int64)
    lib.dsa_index_topk_varlen_workspace.argtypes = [pi64, i32, i32, i32, i32, i32]
    lib.dsa_index_topk_varlen_workspace.restype = sz
    lib.dsa_index_topk_varlen.argtypes = [vp, vp, vp, pi64, i32, i32, i32, i32, i32, vp, vp, sz, vp]
    lib.dsa_sparse_attn_fwd_varlen.argtypes = [vp, vp, vp, vp, pi64, i32, i32, i32, i32, f32, vp, vp, vp]
    lib.dsa_sparse_attn_bwd_varlen_workspace.argtypes = [pi64, i32, i32, i32]
    lib.dsa_sparse_attn_bwd_varlen_workspace.restype = sz
    lib.dsa_sparse_attn_bwd_varlen.argtypes = [vp, vp, vp, vp, vp, vp, vp, pi64, i32, i32, i32, i32, f32, vp,
                                               vp, vp, vp, sz, vp]
    for f in (lib.dsa_index_topk_varlen, lib.dsa_sparse_attn_fwd_varlen, lib.dsa_sparse_attn_bwd_varlen):
        f.restype = ctypes.c_int
    lib.dsa_sparse_attn_bwd_deterministic_workspace.argtypes = [i64, i32, i32, i32]
    lib.dsa_sparse_attn_bwd_deterministic_workspace.restype = sz
    lib.dsa_sparse_attn_bwd_deterministic.argtypes = [vp, vp, vp, vp, vp, vp, vp, i64, i32, i32, i32, f32, vp,
                                                      vp, vp, vp, sz, vp]
    lib.dsa_sparse_attn_bwd_deterministic.restype = ctypes.c_int
    lib.dsa_sync_status.argtypes = [vp]
    lib.dsa_clear_status.argtypes = []
    for f in (lib.dsa_index_topk, lib.dsa_sparse_attn_fwd, lib.dsa_sparse_attn_fwd_tc, lib.dsa_sparse_attn_bwd,
              lib.dsa_sync_status,
              lib.dsa_clear_status):
        f.restype = ctypes.c_int
    lib.dsa_last_error.argtypes = []
    lib.dsa_last_error.restype = ctypes.c_char_p
    lib.dsa_version.argtypes = []
    lib.dsa_version.restype = ctypes.c_char_p
    lib.dsa_profile_enable.argtypes = [ctypes.c_int]
    lib.dsa_profile_enable.restype = None
    lib.dsa_profile_read.argtypes = [ctypes.c_char_p, ctypes.c_int, ctypes.POINTER(ctypes.c_double),
                                     ctypes.POINTER(ctypes.c_int64), ctypes.c_int]
    lib.dsa_profile_read.restype = ctypes.c_int
    lib.dsa_launch_count.argtypes = []
    lib.dsa_launch_count.restype = ctypes.c_int64
    lib.dsa_index_topk_noalloc.argtypes = [vp, vp, vp, i64, i32, i32, i32, i32, i64, i64, vp, vp]
    lib.dsa_index_topk_noalloc.restype = ctypes.c_int
    lib.dsa_launch_count_reset.argtypes = []
    lib.dsa_launch_count_reset.restype = None
    lib.dsa_index_topk_stats.argtypes = [vp, sz, ctypes.POINTER(ctypes.c_int64), ctypes.c_int, vp]
    lib.dsa_index_topk_stats.restype = ctypes.c_int
    lib.dsa_measure_l2.argtypes = [ctypes.c_int, vp, sz, ctypes.c_int, vp]
    lib.dsa_measure_l2.restype = ctypes.c_double
    lib.dsa_measure_umma.argtypes = [ctypes.c_int, ctypes.c_int, ctypes.c_int, vp]
    lib.dsa_measure_umma.restype = ctypes.c_double
    lib.dsa_measure_fold.argtypes = [ctypes.c_int, ctypes.c_int, vp]
    lib.dsa_measure_fold.restype = ctypes.c_double
    lib.dsa_last_kernel_config.argtypes = [ctypes.c_char_p, sz]
    lib.dsa_last_kernel_config.restype = ctypes.c_int
    return lib


def load():
    """Loads libdsa.so (built by __graft_entry__.build()); raises if it is missing."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise DsaError(DSA_ERR_CUDA, f"{LIB_PATH} is not built; run __graft_entry__.build()")
            _lib = _configure(ctypes.CDLL(LIB_PATH))
    return _lib


def load_library(path: str):
    """A configured handle on another build of the library at `path` (the
    debug build's range checks, the trace build's counters), for calling its
    C ABI directly."""
    return _configure(ctypes.CDLL(path))


def _check(rc: int):
    if rc != DSA_OK:
        raise DsaError(rc, load().dsa_last_error().decode())


def _stream_handle(stream) -> int:
    s = torch.cuda.current_stream() if stream is None else stream
    return int(s.cuda_stream)


def _need(t: torch.Tensor, name: str, dtype, ndim: int):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if t.device.index != torch.cuda.current_device():
        raise ValueError(f"{name} is on {t.device}, but the kernels run on the current device "
                         f"cuda:{torch.cuda.current_device()}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if t.dim() != ndim or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous {ndim}-d tensor (got shape {tuple(t.shape)})")


def index_topk_workspace_size(S: int, Hi: int, Di: int, chunk: int, topk: int, slots: int | None = None) -> int:
    """Recommended index workspace bytes, or the bytes for exactly `slots` chunk slots."""
    if slots is None:
        return int(load().dsa_index_topk_workspace(S, Hi, Di, chunk, topk))
    return int(load().dsa_index_topk_workspace_slots(S, Hi, Di, chunk, topk, slots))


def sparse_attn_bwd_workspace_size(S: int, Hq: int, D: int) -> int:
    return int(load().dsa_sparse_attn_bwd_workspace(S, Hq, D))


def _workspace(nbytes: int, device, given):
    """A caller's workspace must be a contiguous CUDA tensor on the current
    device (the library checks its size); None allocates one."""
    if given is not None:
        _need(given, "workspace", given.dtype, given.dim())
        return given
    return torch.empty(max(nbytes, 256), dtype=torch.uint8, device=device)


def _shape(t: torch.Tensor, name: str, shape):
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)} (got {tuple(t.shape)})")


def _attn_shapes(q, k, v, pool_idx, o=None, lse=None, dO=None):
    """q, o, dO [nq, Hq, D]; lse [nq, Hq]; pool_idx [nq, topk]; k, v [S, D]:
    the kernels index every one of them by these extents."""
    nq, Hq, D = q.shape
    S = k.shape[0]
    _shape(k, "k", (S, D))
    _shape(v, "v", (S, D))
    if pool_idx.shape[0] != nq:
        raise ValueError(f"pool_idx must have {nq} rows (got {pool_idx.shape[0]})")
    for t, name in ((o, "o"), (dO, "dO")):
        if t is not None:
            _shape(t, name, (nq, Hq, D))
    if lse is not None:
        _shape(lse, "lse", (nq, Hq))
    return nq, Hq, D, S


def _out(given, name: str, shape, dtype, device):
    """A caller-supplied output must be a contiguous CUDA tensor of the given
    dtype and shape on the current device (the kernels write through its
    pointer); None allocates one."""
    if given is None:
        return torch.empty(shape, dtype=dtype, device=device)
    _need(given, name, dtype, len(shape))
    if tuple(given.shape) != tuple(shape):
        raise ValueError(f"{name} must have shape {tuple(shape)} (got {tuple(given.shape)})")
    return given


def dsa_index_topk(q_idx, k_idx, w, chunk: int, topk: int, q_begin: int = 0, q_end: int | None = None,
                   pool_idx=None, workspace=None, stream=None):
    """pool_idx [q_end - q_begin, topk] int32 of the selected pools (ascending, -1 padded)."""
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    _need(k_idx, "k_idx", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    S, Hi, Di = q_idx.shape
    if k_idx.shape != (S, Di) or w.shape != (S, Hi):
        raise ValueError("k_idx must be [S, Di] and w [S, Hi]")
    q_end = S if q_end is None else q_end
    pool_idx = _out(pool_idx, "pool_idx", (max(q_end - q_begin, 0), topk), torch.int32, q_idx.device)
    lib = load()
    ws = _workspace(lib.dsa_index_topk_workspace(S, Hi, Di, chunk, topk), q_idx.device, workspace)
    _check(lib.dsa_index_topk(q_idx.data_ptr(), k_idx.data_ptr(), w.data_ptr(), S, Hi, Di, chunk, topk, q_begin,
                              q_end, pool_idx.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(),
                              _stream_handle(stream)))
    return pool_idx


def dsa_index_topk_noalloc(q_idx, k_idx, w, chunk: int, topk: int, q_begin: int = 0, q_end: int | None = None,
                           pool_idx=None, stream=None):
    """dsa_index_topk without a workspace, for callers that must not allocate
    device scratch: the library's fixed built-in buffer is used instead (S up
    to 32768 with chunk up to 256).  `pool_idx` should be passed preallocated
    by such callers; if omitted it is allocated here for convenience."""
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    _need(k_idx, "k_idx", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    S, Hi, Di = q_idx.shape
    if k_idx.shape != (S, Di) or w.shape != (S, Hi):
        raise ValueError("k_idx must be [S, Di] and w [S, Hi]")
    q_end = S if q_end is None else q_end
    pool_idx = _out(pool_idx, "pool_idx", (max(q_end - q_begin, 0), topk), torch.int32, q_idx.device)
    _check(load().dsa_index_topk_noalloc(q_idx.data_ptr(), k_idx.data_ptr(), w.data_ptr(), S, Hi, Di, chunk, topk,
                                         q_begin, q_end, pool_idx.data_ptr(), _stream_handle(stream)))
    return pool_idx


def dsa_sparse_attn_fwd(q, k, v, pool_idx, scale: float = 0.0, o=None, lse=None, stream=None, q_begin: int = 0):
    """(o [nq, Hq, D] bf16, lse [nq, Hq] fp32) for queries q_begin .. q_begin + nq - 1.

    q, pool_idx, o and lse hold those queries' rows (nq = q.shape[0]); k and v
    hold the whole sequence [S, D].  With q_begin = 0 and nq = S this is the
    unsharded forward."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 2)
    _need(v, "v", torch.bfloat16, 2)
    _need(pool_idx, "pool_idx", torch.int32, 2)
    nq, Hq, D, S = _attn_shapes(q, k, v, pool_idx)
    o = _out(o, "o", q.shape, torch.bfloat16, q.device)
    lse = _out(lse, "lse", (nq, Hq), torch.float32, q.device)
    _check(load().dsa_sparse_attn_fwd_range(q.data_ptr(), k.data_ptr(), v.data_ptr(), pool_idx.data_ptr(), S,
                                            q_begin, q_begin + nq, Hq, D, pool_idx.shape[1], float(scale),
                                            o.data_ptr(), lse.data_ptr(), _stream_handle(stream)))
    return o, lse


def dsa_sparse_attn_fwd_tc(q, k, v, pool_idx, scale: float = 0.0, o=None, lse=None, stream=None):
    """The whole-sequence forward on the tcgen05 tensor cores (the measured
    tensor-core alternative to dsa_sparse_attn_fwd): (o [S, Hq, D] bf16,
    lse [S, Hq] fp32)."""
    _need(q, "q", torch.bfloat16, 3)
    _need(k, "k", torch.bfloat16, 2)
    _need(v, "v", torch.bfloat16, 2)
    _need(pool_idx, "pool_idx", torch.int32, 2)
    nq, Hq, D, S = _attn_shapes(q, k, v, pool_idx)
    if nq != S:
        raise ValueError("dsa_sparse_attn_fwd_tc: q must hold every query of the sequence")
    o = _out(o, "o", q.shape, torch.bfloat16, q.device)
    lse = _out(lse, "lse", (nq, Hq), torch.float32, q.device)
    _check(load().dsa_sparse_attn_fwd_tc(q.data_ptr(), k.data_ptr(), v.data_ptr(), pool_idx.data_ptr(), S, Hq, D,
                                         pool_idx.shape[1], float(scale), o.data_ptr(), lse.data_ptr(),
                                         _stream_handle(stream)))
    return o, lse


def dsa_sparse_attn_bwd(dO, q, k, v, o, lse, pool_idx, scale: float = 0.0, dq=None, dk=None, dv=None,
                        workspace=None, stream=None, q_begin: int = 0):
    """(dq [nq, Hq, D], dk [S, D], dv [S, D]) in bf16 for queries q_begin .. q_begin + nq - 1.

    dO, q, o, lse, pool_idx and dq hold those queries' rows; k, v, dk and dv
    the whole sequence.  dk and dv are this range's contribution (the full
    gradient when the range is the whole sequence)."""
    for t, n, nd in ((dO, "dO", 3), (q, "q", 3), (o, "o", 3), (k, "k", 2), (v, "v", 2)):
        _need(t, n, torch.bfloat16, nd)
    _need(lse, "lse", torch.float32, 2)
    _need(pool_idx, "pool_idx", torch.int32, 2)
    nq, Hq, D, S = _attn_shapes(q, k, v, pool_idx, o=o, lse=lse, dO=dO)
    dq = _out(dq, "dq", q.shape, torch.bfloat16, q.device)
    dk = _out(dk, "dk", k.shape, torch.bfloat16, q.device)
    dv = _out(dv, "dv", v.shape, torch.bfloat16, q.device)
    lib = load()
    ws = _workspace(lib.dsa_sparse_attn_bwd_workspace(S, Hq, D), q.device, workspace)
    _check(lib.dsa_sparse_attn_bwd_range(dO.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                         lse.data_ptr(), pool_idx.data_ptr(), S, q_begin, q_begin + nq, Hq, D,
                                         pool_idx.shape[1], float(scale), dq.data_ptr(), dk.data_ptr(),
                                         dv.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(),
                                         _stream_handle(stream)))
    return dq, dk, dv


def sparse_attn_bwd_deterministic_workspace_size(S: int, Hq: int, D: int, topk: int) -> int:
    return int(load().dsa_sparse_attn_bwd_deterministic_workspace(S, Hq, D, topk))


def dsa_sparse_attn_bwd_deterministic(dO, q, k, v, o, lse, pool_idx, scale: float = 0.0, dq=None, dk=None,
                                      dv=None, workspace=None, stream=None):
    """(dq [S, Hq, D], dk [S, D], dv [S, D]) in bf16 for the whole sequence,
    with dk and dv summed in a fixed order (the same bits on every run)."""
    for t, n, nd in ((dO, "dO", 3), (q, "q", 3), (o, "o", 3), (k, "k", 2), (v, "v", 2)):
        _need(t, n, torch.bfloat16, nd)
    _need(lse, "lse", torch.float32, 2)
    _need(pool_idx, "pool_idx", torch.int32, 2)
    S, Hq, D, _ = _attn_shapes(q, k, v, pool_idx, o=o, lse=lse, dO=dO)
    if k.shape[0] != S:
        raise ValueError("the deterministic backward takes the whole sequence: q and k need the same rows")
    topk = pool_idx.shape[1]
    dq = _out(dq, "dq", q.shape, torch.bfloat16, q.device)
    dk = _out(dk, "dk", k.shape, torch.bfloat16, q.device)
    dv = _out(dv, "dv", v.shape, torch.bfloat16, q.device)
    lib = load()
    need = lib.dsa_sparse_attn_bwd_deterministic_workspace(S, Hq, D, topk)
    ws = _workspace(int(need), q.device, workspace)
    _check(lib.dsa_sparse_attn_bwd_deterministic(dO.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(),
                                                 o.data_ptr(), lse.data_ptr(), pool_idx.data_ptr(), S, Hq, D, topk,
                                                 float(scale), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(),
                                                 ws.data_ptr(), ws.numel() * ws.element_size(),
                                                 _stream_handle(stream)))
    return dq, dk, dv


def _cu(cu_seqlens):
    vals = [int(x) for x in cu_seqlens]
    return (ctypes.c_int64 * len(vals))(*vals), len(vals) - 1


def dsa_index_topk_varlen(q_idx, k_idx, w, cu_seqlens, chunk: int, topk: int, pool_idx=None, workspace=None,
                          stream=None):
    """Packed batch: pool_idx [T, topk] with each sequence's pool indices
    counted from its own first token (cu_seqlens: nseq + 1 host offsets)."""
    _need(q_idx, "q_idx", torch.bfloat16, 3)
    _need(k_idx, "k_idx", torch.bfloat16, 2)
    _need(w, "w", torch.float32, 2)
    T, Hi, Di = q_idx.shape
    _shape(k_idx, "k_idx", (T, Di))
    _shape(w, "w", (T, Hi))
    cu, nseq = _cu(cu_seqlens)
    if nseq < 1 or cu[nseq] != T:
        raise ValueError("cu_seqlens must end at the packed length")
    pool_idx = _out(pool_idx, "pool_idx", (T, topk), torch.int32, q_idx.device)
    lib = load()
    ws = _workspace(lib.dsa_index_topk_varlen_workspace(cu, nseq, Hi, Di, chunk, topk), q_idx.device, workspace)
    _check(lib.dsa_index_topk_varlen(q_idx.data_ptr(), k_idx.data_ptr(), w.data_ptr(), cu, nseq, Hi, Di, chunk, topk,
                                     pool_idx.data_ptr(), ws.data_ptr(), ws.numel() * ws.element_size(),
                                     _stream_handle(stream)))
    return pool_idx


def dsa_sparse_attn_fwd_varlen(q, k, v, pool_idx, cu_seqlens, scale: float = 0.0, o=None, lse=None, stream=None):
    """Packed batch forward: (o [T, Hq, D], lse [T, Hq]), each sequence attending within itself."""
    for t, n, nd in ((q, "q", 3), (k, "k", 2), (v, "v", 2)):
        _need(t, n, torch.bfloat16, nd)
    _need(pool_idx, "pool_idx", torch.int32, 2)
    T, Hq, D, _ = _attn_shapes(q, k, v, pool_idx)
    _shape(k, "k", (T, D))
    cu, nseq = _cu(cu_seqlens)
    o = _out(o, "o", q.shape, torch.bfloat16, q.device)
    lse = _out(lse, "lse", (T, Hq), torch.float32, q.device)
    _check(load().dsa_sparse_attn_fwd_varlen(q.data_ptr(), k.data_ptr(), v.data_ptr(), pool_idx.data_ptr(), cu, nseq,
                                             Hq, D, pool_idx.shape[1], float(scale), o.data_ptr(), lse.data_ptr(),
                                             _stream_handle(stream)))
    return o, lse


def dsa_sparse_attn_bwd_varlen(dO, q, k, v, o, lse, pool_idx, cu_seqlens, scale: float = 0.0, dq=None, dk=None,
                               dv=None, workspace=None, stream=None):
    """Packed batch backward: (dq [T, Hq, D], dk [T, D], dv [T, D])."""
    for t, n, nd in ((dO, "dO", 3), (q, "q", 3), (o, "o", 3), (k, "k", 2), (v, "v", 2)):
        _need(t, n, torch.bfloat16, nd)
    _need(lse, "lse", torch.float32, 2)
    _need(pool_idx, "pool_idx", torch.int32, 2)
    T, Hq, D, _ = _attn_shapes(q, k, v, pool_idx, o=o, lse=lse, dO=dO)
    _shape(k, "k", (T, D))
    cu, nseq = _cu(cu_seqlens)
    dq = _out(dq, "dq", q.shape, torch.bfloat16, q.device)
    dk = _out(dk, "dk", k.shape, torch.bfloat16, q.device)
    dv = _out(dv, "dv", v.shape, torch.bfloat16, q.device)
    lib = load()
    ws = _workspace(lib.dsa_sparse_attn_bwd_varlen_workspace(cu, nseq, Hq, D), q.device, workspace)
    _check(lib.dsa_sparse_attn_bwd_varlen(dO.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                          lse.data_ptr(), pool_idx.data_ptr(), cu, nseq, Hq, D, pool_idx.shape[1],
                                          float(scale), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), ws.data_ptr(),
                                          ws.numel() * ws.element_size(), _stream_handle(stream)))
    return dq, dk, dv


def zigzag_ranges(S: int, world: int, rank: int):
    """[(b0, e0), (b1, e1)]: the two query ranges of `rank` under zig-zag sharding (host only)."""
    out = (ctypes.c_int64 * 4)()
    _check(load().dsa_zigzag_ranges(S, world, rank, out))
    return [(int(out[0]), int(out[1])), (int(out[2]), int(out[3]))]


def dsa_sync_status(stream=None):
    """Synchronises the stream; raises DsaError if a kernel recorded a failed bounded wait or check."""
    _check(load().dsa_sync_status(_stream_handle(stream)))


def dsa_clear_status():
    _check(load().dsa_clear_status())


def profile_enable(on: bool = True):
    """Record a CUDA event pair around every kernel launch (measurement only)."""
    load().dsa_profile_enable(1 if on else 0)


def profile_read() -> dict:
    """{kernel name: (total device ms, launches)} since the last read; synchronises."""
    lib = load()
    n, name_len = 64, 64
    names = ctypes.create_string_buffer(n * name_len)
    ms = (ctypes.c_double * n)()
    cnt = (ctypes.c_int64 * n)()
    k = lib.dsa_profile_read(names, name_len, ms, cnt, n)
    if k < 0:
        raise DsaError(DSA_ERR_CUDA, lib.dsa_last_error().decode())
    raw = names.raw
    out = {}
    for j in range(k):
        nm = raw[j * name_len:(j + 1) * name_len].split(b"\0", 1)[0].decode()
        out[nm] = (float(ms[j]), int(cnt[j]))
    return out


def index_topk_stats(workspace: torch.Tensor, stream=None) -> dict:
    """Counters of the last dsa_index_topk call on `workspace` (synchronises)."""
    lib = load()
    out = (ctypes.c_int64 * 8)()
    n = lib.dsa_index_topk_stats(workspace.data_ptr(), workspace.numel() * workspace.element_size(), out, 8,
                                 _stream_handle(stream))
    if n < 0:
        raise DsaError(DSA_ERR_CUDA, lib.dsa_last_error().decode())
    names = ("fallback_rows",)
    return {names[j]: int(out[j]) for j in range(min(n, len(names)))}


def last_kernel_config() -> dict:
    """What the last dsa_* call made on this host thread ran: its entry point,
    variant, kernels (name, launches) in launch order and plan parameters."""
    import json
    lib = load()
    n = lib.dsa_last_kernel_config(None, 0)
    buf = ctypes.create_string_buffer(n + 1)
    lib.dsa_last_kernel_config(buf, n + 1)
    return json.loads(buf.value.decode())


def measure_l2(kind: int, buf: torch.Tensor, iters: int = 20, stream=None) -> float:
    """GB/s of an L2 probe kernel on `buf` (kind 0 stream read, 1 1-KB gather, 2 red.v4 reductions of
    4 rows x 128 B, 3 / 4 bulk reductions of 2 KB / 512 B, 5 / 6 / 7 red.v4 of 2 x 256 B / 8 x 64 B /
    16 x 32 B, 8 kinds 2 and 3 at once)."""
    lib = load()
    r = lib.dsa_measure_l2(kind, buf.data_ptr(), buf.numel() * buf.element_size(), iters, _stream_handle(stream))
    if r < 0:
        raise DsaError(DSA_ERR_CUDA, lib.dsa_last_error().decode())
    return float(r)


def measure_umma(n: int, issuers: int = 1, groups: int = 2000, stream=None) -> float:
    """Clock cycles per tcgen05.mma (M 128, N n, K 16, bf16) as seen by its
    issuing thread, with `issuers` issuing CTAs on every SM."""
    lib = load()
    r = lib.dsa_measure_umma(n, issuers, groups, _stream_handle(stream))
    if r < 0:
        raise DsaError(DSA_ERR_CUDA, lib.dsa_last_error().decode())
    return float(r)


def measure_fold(mode: int, heads: int = 2000, stream=None) -> float:
    """Clock cycles per head of the indexer's accumulator handoff in isolation
    (mode 0 loads only, 1 loads and fold), or per 32-column tensor-memory load
    (mode 2)."""
    lib = load()
    r = lib.dsa_measure_fold(mode, heads, _stream_handle(stream))
    if r < 0:
        raise DsaError(DSA_ERR_CUDA, lib.dsa_last_error().decode())
    return float(r)


def launch_count() -> int:
    return int(load().dsa_launch_count())


def launch_count_reset():
    load().dsa_launch_count_reset()


def version() -> str:
    return load().dsa_version().decode()
