"""Seeded synthetic inputs for the DSA layer workloads (input data only).

Both the CPU oracle tests and the GPU path take their inputs from here; this
module holds none of the layer's arithmetic.  The generator itself lives in
``synth.c`` (counter-based SplitMix64, Box-Muller normals, bf16 round-to-
nearest-even) and is compiled on first use with gcc.

bf16 tensors are returned as ``numpy.uint16`` arrays holding the raw bf16 bit
patterns; ``bf16_to_f32`` widens them exactly.

The workloads follow the sizes and value distributions of the GLM-5.3-Flash
DeepSeek-Sparse-Attention layer discussed in "SkyRL 将 GLM-5.3-Flash 训练上下文
扩至 100 万 token" (§1 DSA 真稀疏: 4-token pools, ~2048 selected keys per query,
query-chunked indexer) and "How Lila Sciences and Anyscale Scaled
GLM-5.3-Flash Training" (lessons: random-token inputs suffice for speed and
memory measurements).  No public dataset is involved.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "synth.c")
_LIB_PATH = os.path.join(_HERE, "libsynth.so")
_lock = threading.Lock()
_lib = None

# tensor ids: each input tensor draws from its own stream
TID_Q_IDX, TID_K_IDX, TID_W, TID_Q, TID_K, TID_V, TID_DO, TID_POOLSEL, TID_ZIPF = 1, 2, 3, 4, 5, 6, 7, 8, 9


def build(force: bool = False) -> str:
    """Compile libsynth.so next to synth.c (gcc, OpenMP)."""
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
            u64, i64, dbl, vp = ctypes.c_uint64, ctypes.c_int64, ctypes.c_double, ctypes.c_void_p
            lib.synth_normal_bf16.argtypes = [u64, u64, u64, dbl, vp]
            lib.synth_uniform_f32.argtypes = [u64, u64, u64, vp]
            lib.synth_int_bf16.argtypes = [u64, u64, u64, i64, i64, vp]
            lib.synth_int_f32.argtypes = [u64, u64, u64, i64, i64, vp]
            lib.synth_cluster_keys_bf16.argtypes = [u64, u64, i64, i64, i64, i64, dbl, dbl, vp]
            lib.synth_zipf_pool_magnitudes.argtypes = [u64, u64, i64, dbl, dbl, vp, vp]
            lib.synth_scale_pools_bf16.argtypes = [i64, i64, vp, vp]
            lib.synth_pool_selection.argtypes = [u64, u64, i64, i64, vp, i64, vp]
            for f in (lib.synth_normal_bf16, lib.synth_uniform_f32, lib.synth_int_bf16, lib.synth_int_f32,
                      lib.synth_cluster_keys_bf16, lib.synth_zipf_pool_magnitudes, lib.synth_scale_pools_bf16,
                      lib.synth_pool_selection):
                f.restype = None
            _lib = lib
    return _lib


def _ptr(a: np.ndarray) -> int:
    assert a.flags.c_contiguous
    return a.ctypes.data


def bf16_to_f32(bits: np.ndarray) -> np.ndarray:
    """Widen raw bf16 bit patterns to float32 (exact)."""
    return (bits.astype(np.uint32) << 16).view(np.float32)


def normal_bf16(seed, tid, shape, scale=1.0, out=None) -> np.ndarray:
    a = np.empty(shape, np.uint16) if out is None else out
    _load().synth_normal_bf16(seed, tid, a.size, float(scale), _ptr(a))
    return a


def uniform_f32(seed, tid, shape) -> np.ndarray:
    a = np.empty(shape, np.float32)
    _load().synth_uniform_f32(seed, tid, a.size, _ptr(a))
    return a


def int_bf16(seed, tid, shape, lo, hi) -> np.ndarray:
    a = np.empty(shape, np.uint16)
    _load().synth_int_bf16(seed, tid, a.size, lo, hi, _ptr(a))
    return a


def int_f32(seed, tid, shape, lo, hi) -> np.ndarray:
    a = np.empty(shape, np.float32)
    _load().synth_int_f32(seed, tid, a.size, lo, hi, _ptr(a))
    return a


def cluster_keys_bf16(seed, tid, S, Di, n_clusters=8, plant_every=16, centroid_norm=8.0, noise=0.5):
    a = np.empty((S, Di), np.uint16)
    _load().synth_cluster_keys_bf16(seed, tid, S, Di, n_clusters, plant_every, centroid_norm, noise, _ptr(a))
    return a


def zipf_pool_magnitudes(seed, tid, P, s=1.1, amax=64.0):
    mag = np.empty(P, np.float32)
    rank = np.empty(P, np.int64)
    _load().synth_zipf_pool_magnitudes(seed, tid, P, s, amax, _ptr(mag), _ptr(rank))
    return mag, rank


def pool_selection(seed, tid, S, topk, hot=None) -> np.ndarray:
    """A valid stand-in pool selection [S, topk] int32 (ascending, -1 padded)."""
    out = np.empty((S, topk), np.int32)
    hot = np.zeros(0, np.int64) if hot is None else np.ascontiguousarray(hot, dtype=np.int64)
    _load().synth_pool_selection(seed, tid, S, topk, _ptr(hot) if hot.size else None, hot.size, _ptr(out))
    return out


@dataclasses.dataclass(frozen=True)
class Workload:
    """One synthetic DSA-layer configuration (batch 1)."""
    name: str
    S: int
    Hi: int = 32        # indexer heads
    Di: int = 64        # indexer head dim
    topk: int = 512     # pools kept per query
    chunk: int = 256    # indexer query chunk
    Hq: int = 16        # attention query heads (sharing one KV head)
    D: int = 128        # attention head dim
    values: str = "normal"   # "int" | "normal" | "cluster" | "zipf"
    q_idx_scale: float = 1.0
    seed: int = 0
    backward: bool = False

    @property
    def pools(self) -> int:
        return self.S // 4

    @property
    def scale(self) -> float:
        return 1.0 / float(np.sqrt(self.D))


WORKLOADS = {
    # exactness case: integer-valued inputs, every product and sum exact
    "tiny_int_s2048": Workload("tiny_int_s2048", 2048, Hi=8, topk=64, chunk=256, values="int", seed=0,
                               backward=True),
    "s16k": Workload("s16k", 16384, values="normal", seed=1),
    "s32k": Workload("s32k", 32768, values="normal", q_idx_scale=0.125, seed=5, backward=True),
    "s128k": Workload("s128k", 131072, values="normal", q_idx_scale=0.125, seed=2, backward=True),
    "s256k_cluster": Workload("s256k_cluster", 262144, chunk=512, values="cluster", seed=3),
    "s1m_cluster": Workload("s1m_cluster", 1048576, chunk=512, values="cluster", seed=3),
    # the same inputs with the attention backward (the layer's whole step at 1M)
    "s1m_cluster_bwd": Workload("s1m_cluster_bwd", 1048576, chunk=512, values="cluster", seed=3, backward=True),
    "s64k_zipf": Workload("s64k_zipf", 65536, values="zipf", seed=4, backward=True),
}


def indexer_inputs(wl: Workload):
    """q_idx [S,Hi,Di] bf16, k_idx [S,Di] bf16, w [S,Hi] fp32."""
    S, Hi, Di, s = wl.S, wl.Hi, wl.Di, wl.seed
    if wl.values == "int":
        q_idx = int_bf16(s, TID_Q_IDX, (S, Hi, Di), -3, 3)
        k_idx = int_bf16(s, TID_K_IDX, (S, Di), -3, 3)
        w = int_f32(s, TID_W, (S, Hi), 0, 3)
        return q_idx, k_idx, w
    q_idx = normal_bf16(s, TID_Q_IDX, (S, Hi, Di), wl.q_idx_scale)
    if wl.values == "cluster":
        k_idx = cluster_keys_bf16(s, TID_K_IDX, S, Di)
    else:
        k_idx = normal_bf16(s, TID_K_IDX, (S, Di))
    if wl.values == "zipf":
        mag, _ = zipf_pool_magnitudes(s, TID_ZIPF, (S + 3) // 4)
        _load().synth_scale_pools_bf16(S, Di, _ptr(mag), _ptr(k_idx))
    w = uniform_f32(s, TID_W, (S, Hi))
    return q_idx, k_idx, w


def attention_inputs(wl: Workload):
    """q [S,Hq,D], k [S,D], v [S,D] (bf16 bits)."""
    S, Hq, D, s = wl.S, wl.Hq, wl.D, wl.seed
    if wl.values == "int":
        return (int_bf16(s, TID_Q, (S, Hq, D), -2, 2), int_bf16(s, TID_K, (S, D), -2, 2),
                int_bf16(s, TID_V, (S, D), -2, 2))
    return normal_bf16(s, TID_Q, (S, Hq, D)), normal_bf16(s, TID_K, (S, D)), normal_bf16(s, TID_V, (S, D))


def grad_output(wl: Workload):
    """dO [S,Hq,D] bf16 bits (upstream gradient)."""
    if wl.values == "int":
        return int_bf16(wl.seed, TID_DO, (wl.S, wl.Hq, wl.D), -2, 2)
    return normal_bf16(wl.seed, TID_DO, (wl.S, wl.Hq, wl.D))


def hot_pools(wl: Workload, n_hot: int = 64) -> np.ndarray:
    """Pools with the largest Zipf magnitudes (popular pools), for the zipf workload."""
    if wl.values != "zipf":
        return np.zeros(0, np.int64)
    _, rank = zipf_pool_magnitudes(wl.seed, TID_ZIPF, (wl.S + 3) // 4)
    return np.argsort(rank, kind="stable")[:n_hot].astype(np.int64)


def stand_in_selection(wl: Workload, S: int | None = None) -> np.ndarray:
    """Valid pool_idx for testing attention on its own (see synth_pool_selection)."""
    return pool_selection(wl.seed, TID_POOLSEL, wl.S if S is None else S, wl.topk, hot_pools(wl))
