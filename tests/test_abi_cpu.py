"""Host-side checks of the C ABI that need no GPU: the library loads, exports
every entry point include/dsa.h declares, and rejects bad arguments with the
documented status codes before touching the device."""
import ctypes
import math
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "dsa.h")


@pytest.fixture(scope="module")
def lib():
    from long_context_sparse_index_gb300 import build as b
    b.build()
    import long_context_sparse_index_gb300 as dsa
    return dsa.load()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_the_three_calls_and_helpers():
    names = declared_functions()
    for n in ("dsa_index_topk", "dsa_sparse_attn_fwd", "dsa_sparse_attn_bwd", "dsa_index_topk_workspace",
              "dsa_sparse_attn_bwd_workspace", "dsa_sync_status", "dsa_last_error"):
        assert n in names


def test_library_exports_every_declared_symbol(lib):
    import long_context_sparse_index_gb300 as dsa
    for name in declared_functions():
        assert hasattr(lib, name), name
        assert name in dsa.EXPORTED or name in ("dsa_index_topk_workspace",)


def test_version(lib):
    assert lib.dsa_version().startswith(b"libdsa")


def _pow2_ceil(x):
    p = 1
    while p < x:
        p <<= 1
    return p


def _pow2_floor(x):
    p = 1
    while 2 * p <= x:
        p <<= 1
    return p


def _index_ws(S, chunk, topk, nbuf):
    """The index workspace as the header describes it, each part rounded up to 256 B."""
    r = lambda x: (x + 255) // 256 * 256
    P = S // 4
    P1 = max(P, 1)
    Ppad = r(P) if P else 256
    sigma = max(_pow2_floor(max(1, topk // 16)), _pow2_ceil((P + 4095) // 4096))
    c = (2 * math.sqrt(sigma) + math.sqrt(4 * sigma + topk)) ** 2
    cap = max(4096, _pow2_ceil(math.ceil(c + 4 * math.sqrt(sigma * c))))
    G = (P + sigma - 1) // sigma
    samp_ld = r(G) if G else 256
    rows = min(chunk, S)
    thr_ld = (rows + 127) // 128 * 128
    return (512 + 2 * r(P1 * 256) + r(S * 4) + r(64 * Ppad * 4) + r(nbuf * rows * samp_ld * 4) + r(nbuf * thr_ld * 8)
            + r(nbuf * thr_ld * 4) + r(nbuf * rows * cap * 8))


def test_workspace_sizes(lib):
    S, chunk = 131072, 256
    assert lib.dsa_index_topk_workspace(S, 32, 64, chunk, 512) == _index_ws(S, chunk, 512, 8)
    # the slot's candidate lists: 4096 per row for topk 512, sampled every 32nd pool
    assert _index_ws(S, chunk, 512, 8) - _index_ws(S, chunk, 512, 7) == 256 * 1024 * 4 + 256 * 12 + 256 * 4096 * 8
    assert lib.dsa_index_topk_workspace(1048576, 32, 64, 512, 512) == _index_ws(1048576, 512, 512, 8)
    assert lib.dsa_index_topk_workspace(1024, 8, 64, 512, 64) == _index_ws(1024, 512, 64, 2)
    assert lib.dsa_index_topk_workspace(1024, 8, 64, 100, 2048) == _index_ws(1024, 100, 2048, 8)
    assert lib.dsa_index_topk_workspace(0, 32, 64, chunk, 512) == 0
    # one chunk covering the whole sequence needs one slot of S rows
    assert lib.dsa_index_topk_workspace(1000, 8, 64, 4096, 64) == lib.dsa_index_topk_workspace(1000, 8, 64, 1000, 64)
    assert lib.dsa_index_topk_workspace(1024, 8, 64, 1024, 64) == _index_ws(1024, 1024, 64, 1)
    # the built-in no-alloc buffer holds the two-slot minimum for S <= 32768 with chunk <= 256, topk <= 512
    need = max(_index_ws(S_, c_, k_, min(2, (S_ + c_ - 1) // c_)) for S_ in (4097, 16388, 20000, 32768)
               for c_ in (1, 64, 256) for k_ in (1, 8, 64, 255, 512))
    assert need <= 32 << 20
    assert lib.dsa_sparse_attn_bwd_workspace(S, 16, 128) == 2 * S * 128 * 4 + S * 16 * 4


FAKE = 0x10000  # 16-byte aligned dummy address; calls below fail validation before any device access


def _idx(lib, **kw):
    a = dict(q=FAKE, k=FAKE, w=FAKE, S=1024, Hi=8, Di=64, chunk=128, topk=64, b=0, e=1024, out=FAKE, ws=FAKE,
             wsb=1 << 30, stream=None)
    a.update(kw)
    return lib.dsa_index_topk(a["q"], a["k"], a["w"], a["S"], a["Hi"], a["Di"], a["chunk"], a["topk"], a["b"], a["e"],
                              a["out"], a["ws"], a["wsb"], a["stream"])


def test_index_topk_rejects_bad_arguments(lib):
    import long_context_sparse_index_gb300 as dsa
    assert _idx(lib, q=None) == dsa.DSA_ERR_INVALID_ARG
    assert _idx(lib, w=FAKE + 2) == dsa.DSA_ERR_INVALID_ARG
    assert _idx(lib, q=FAKE + 4) == dsa.DSA_ERR_INVALID_ARG
    assert _idx(lib, S=0) == dsa.DSA_ERR_INVALID_ARG
    assert _idx(lib, chunk=0) == dsa.DSA_ERR_INVALID_ARG
    assert _idx(lib, topk=0) == dsa.DSA_ERR_INVALID_ARG
    assert _idx(lib, b=10, e=10) == dsa.DSA_ERR_INVALID_ARG
    assert _idx(lib, e=1025) == dsa.DSA_ERR_INVALID_ARG
    assert _idx(lib, Di=128) == dsa.DSA_ERR_UNSUPPORTED
    assert _idx(lib, Hi=65) == dsa.DSA_ERR_UNSUPPORTED
    assert _idx(lib, topk=4096) == dsa.DSA_ERR_UNSUPPORTED
    assert _idx(lib, wsb=100) == dsa.DSA_ERR_WORKSPACE
    # the two-slot minimum passes the argument checks (and then needs a GPU); one byte less does not
    S, chunk = 1024, 128
    minimum = _index_ws(S, chunk, 64, 2)
    assert _idx(lib, S=S, e=S, chunk=chunk, wsb=minimum - 1) == dsa.DSA_ERR_WORKSPACE
    assert _idx(lib, S=S, e=S, chunk=chunk, wsb=minimum) != dsa.DSA_ERR_WORKSPACE
    assert _idx(lib, ws=None) == dsa.DSA_ERR_WORKSPACE
    assert _idx(lib, ws=FAKE + 16) == dsa.DSA_ERR_INVALID_ARG
    assert b"workspace" in lib.dsa_last_error()


def test_attention_rejects_bad_arguments(lib):
    import long_context_sparse_index_gb300 as dsa
    f = lib.dsa_sparse_attn_fwd
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 16, 128, 8, 0.0, FAKE, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 8, 128, 8, 0.0, FAKE, FAKE, None) == dsa.DSA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 16, 64, 8, 0.0, FAKE, FAKE, None) == dsa.DSA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, 0, 16, 128, 8, 0.0, FAKE, FAKE, None) == dsa.DSA_ERR_INVALID_ARG
    b = lib.dsa_sparse_attn_bwd
    args = [FAKE] * 7 + [64, 16, 128, 8, 0.0] + [FAKE] * 3
    assert b(*args, FAKE, 16, None) == dsa.DSA_ERR_WORKSPACE
    assert b(*args, None, 1 << 30, None) == dsa.DSA_ERR_WORKSPACE
    assert b(*args[:7], 64, 16, 128, 4096, 0.0, *args[12:], FAKE, 1 << 30, None) == dsa.DSA_ERR_UNSUPPORTED


def test_tcgen05_forward_and_probes_reject_bad_arguments(lib):
    """The tcgen05 forward takes the default forward's checks; the tensor-core
    probe and the profile reader refuse bad arguments (and the profile reader
    answers -1 in the default build, which has no counters) without touching
    the device."""
    import long_context_sparse_index_gb300 as dsa
    f = lib.dsa_sparse_attn_fwd_tc
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 16, 128, 8, 0.0, FAKE, None, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 8, 128, 8, 0.0, FAKE, FAKE, None) == dsa.DSA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 16, 64, 8, 0.0, FAKE, FAKE, None) == dsa.DSA_ERR_UNSUPPORTED
    assert f(FAKE, FAKE, FAKE, FAKE, 0, 16, 128, 8, 0.0, FAKE, FAKE, None) == dsa.DSA_ERR_INVALID_ARG
    assert f(FAKE + 8, FAKE, FAKE, FAKE, 64, 16, 128, 8, 0.0, FAKE, FAKE, None) == dsa.DSA_ERR_INVALID_ARG
    assert b"16-byte aligned" in lib.dsa_last_error()
    m = lib.dsa_measure_umma
    for n, issuers, groups in ((8, 1, 10), (48, 1, 10), (16, 0, 10), (16, 4, 10), (256, 3, 10), (16, 1, 0)):
        assert m(n, issuers, groups, None) == -1.0
    assert b"dsa_measure_umma" in lib.dsa_last_error()
    fo = lib.dsa_measure_fold
    for mode, heads in ((-1, 100), (3, 100), (1, 1)):
        assert fo(mode, heads, None) == -1.0
    assert b"dsa_measure_fold" in lib.dsa_last_error()
    p = lib.dsa_fwd_tc_profile
    p.argtypes = [ctypes.c_void_p, ctypes.c_int]
    assert p(None, 4) == -1
    buf = (ctypes.c_uint64 * (32 * 4))()
    assert p(ctypes.addressof(buf), 0) == -1
    assert p(ctypes.addressof(buf), 4) == -1
    assert b"without DSA_FWD_PROFILE" in lib.dsa_last_error()


def test_attention_ranges_are_checked(lib):
    """The range forms reject a query range outside [0, S) before any device access."""
    import long_context_sparse_index_gb300 as dsa
    f = lib.dsa_sparse_attn_fwd_range
    for qb, qe in ((0, 0), (-1, 10), (10, 65), (40, 30)):
        assert f(FAKE, FAKE, FAKE, FAKE, 64, qb, qe, 16, 128, 8, 0.0, FAKE, FAKE, None) == dsa.DSA_ERR_INVALID_ARG
        assert b"query range" in lib.dsa_last_error()
    b = lib.dsa_sparse_attn_bwd_range
    args = [FAKE] * 7 + [64, 70, 80, 16, 128, 8, 0.0] + [FAKE] * 3 + [FAKE, 1 << 30, None]
    assert b(*args) == dsa.DSA_ERR_INVALID_ARG


def test_last_kernel_config_reports_the_outermost_call(lib):
    """dsa_last_kernel_config describes the last entry point this thread
    called: a call rejected before any launch lists no kernels; an entry point
    that forwards to another (dsa_sparse_attn_fwd -> _range) reports as
    itself; the output is truncated to the buffer with snprintf semantics."""
    import json
    import long_context_sparse_index_gb300 as dsa
    assert _idx(lib, S=0) == dsa.DSA_ERR_INVALID_ARG
    cfg = dsa.last_kernel_config()
    assert cfg["entry"] == "dsa_index_topk" and cfg["kernels"] == []
    f = lib.dsa_sparse_attn_fwd
    assert f(FAKE, FAKE, FAKE, FAKE, 64, 16, 128, 8, 0.0, FAKE, None, None) == dsa.DSA_ERR_INVALID_ARG
    cfg = dsa.last_kernel_config()
    assert cfg["entry"] == "dsa_sparse_attn_fwd" and cfg["kernels"] == [] and cfg["params"] == {}
    n = lib.dsa_last_kernel_config(None, 0)
    full = ctypes.create_string_buffer(n + 1)
    assert lib.dsa_last_kernel_config(full, n + 1) == n
    assert json.loads(full.value.decode())["entry"] == "dsa_sparse_attn_fwd"
    short = ctypes.create_string_buffer(8)
    assert lib.dsa_last_kernel_config(short, 8) == n
    assert short.value == full.value[:7]


def test_deterministic_backward_workspace_and_checks(lib):
    """The deterministic backward's workspace holds at least its fp32 dK/dV
    accumulators, Delta and the per-pool query lists (S x topk int32), plus
    the (pool, 1024-query block) counters (S/4 x S/1024 x 4 B, capped at
    256 MiB) and a little padding; shapes it cannot index with 32-bit list
    positions give 0 and DSA_ERR_UNSUPPORTED, before any device access."""
    import long_context_sparse_index_gb300 as dsa
    ws = lib.dsa_sparse_attn_bwd_deterministic_workspace
    S, topk = 131072, 512
    need = ws(S, 16, 128, topk)
    floor = 2 * S * 128 * 4 + S * 16 * 4 + S * topk * 4 + (S // 4) * (S // 1024) * 4
    assert floor <= need <= floor + 4 * S + (1 << 20)
    assert ws(1, 16, 128, 1) > 0 and ws(5, 16, 128, 3) > 0
    assert ws(S, 8, 128, topk) == 0 and ws(S, 16, 64, topk) == 0 and ws(S, 16, 128, 4096) == 0
    assert ws(0, 16, 128, topk) == 0
    assert ws((1 << 31) // 2048, 16, 128, 2048) == 0 and ws((1 << 31) // 2048 - 1, 16, 128, 2048) > 0
    # more pools than the counter scan holds, even in one counting block (topk = 1 keeps S x topk legal)
    assert ws(4 * (1 << 26) + 4, 16, 128, 1) == 0 and ws(4 * (1 << 26), 16, 128, 1) > 0
    b = lib.dsa_sparse_attn_bwd_deterministic
    args = [FAKE] * 7 + [64, 16, 128, 8, 0.0] + [FAKE] * 3
    assert b(*args, FAKE, 16, None) == dsa.DSA_ERR_WORKSPACE
    assert b(*args, None, 1 << 30, None) == dsa.DSA_ERR_WORKSPACE
    assert b(*args, FAKE + 16, 1 << 30, None) == dsa.DSA_ERR_INVALID_ARG  # workspace not 256-byte aligned
    assert b(*args[:7], 1 << 21, 16, 128, 1024, 0.0, *args[12:], FAKE, 1 << 40, None) == dsa.DSA_ERR_UNSUPPORTED
    assert b(None, *args[1:], FAKE, 1 << 30, None) == dsa.DSA_ERR_INVALID_ARG


def test_varlen_checks_cu_seqlens_and_workspace(lib):
    """Packed batches: cu_seqlens must start at 0 and increase strictly; the
    indexer's workspace is one slice (the longest sequence's) per sequence
    indexed at once -- the long sequences with fewer than 304 indexer tiles,
    up to 4 of them -- the backward's that of the packed length (its fp32
    dK/dV accumulators span the batch); errors come back before any sequence
    runs."""
    import ctypes
    import long_context_sparse_index_gb300 as dsa
    def cu(*v):
        return (ctypes.c_int64 * len(v))(*v)
    good = cu(0, 5, 1029, 1030)
    assert lib.dsa_index_topk_varlen_workspace(good, 3, 8, 64, 256, 64) == lib.dsa_index_topk_workspace(1024, 8, 64,
                                                                                                         256, 64)
    assert lib.dsa_sparse_attn_bwd_varlen_workspace(good, 3, 16, 128) == lib.dsa_sparse_attn_bwd_workspace(1030, 16,
                                                                                                           128)
    # topk 64: sequences of more than 260 tokens run the indexer; 1000 tokens
    # make 8 tiles (each may run alongside others), 20000 tokens ~1500 (alone)
    one = lib.dsa_index_topk_workspace(1000, 8, 64, 256, 64)
    assert lib.dsa_index_topk_varlen_workspace(cu(0, 1000, 2000, 3000, 4000, 5000), 5, 8, 64, 256, 64) == 4 * one
    assert lib.dsa_index_topk_varlen_workspace(cu(0, 1000, 1100, 2100), 3, 8, 64, 256, 64) == 2 * one
    assert lib.dsa_index_topk_varlen_workspace(cu(0, 20000, 21000), 2, 8, 64, 256, 64) == \
        lib.dsa_index_topk_workspace(20000, 8, 64, 256, 64)
    for bad, n in ((cu(1, 5), 1), (cu(0, 5, 5), 2), (cu(0, 7, 3), 2), (cu(0), 0)):
        assert lib.dsa_index_topk_varlen_workspace(bad, n, 8, 64, 256, 64) == 0
        assert lib.dsa_index_topk_varlen(FAKE, FAKE, FAKE, bad, n, 8, 64, 256, 64, FAKE, FAKE, 1 << 30,
                                         None) == dsa.DSA_ERR_INVALID_ARG
        assert lib.dsa_sparse_attn_fwd_varlen(FAKE, FAKE, FAKE, FAKE, bad, n, 16, 128, 8, 0.0, FAKE, FAKE,
                                              None) == dsa.DSA_ERR_INVALID_ARG
    assert lib.dsa_index_topk_varlen(FAKE, FAKE, FAKE, good, 3, 8, 64, 256, 64, FAKE, FAKE, 1000,
                                     None) == dsa.DSA_ERR_WORKSPACE
    args = [FAKE] * 7 + [good, 3, 16, 128, 8, 0.0] + [FAKE] * 3
    assert lib.dsa_sparse_attn_bwd_varlen(*args, FAKE, 1000, None) == dsa.DSA_ERR_WORKSPACE


def test_no_device_reports_cuda_error_not_crash(lib):
    """With valid arguments but no usable GPU the call fails with DSA_ERR_CUDA
    (or runs, on a GPU host) -- it never falls back to another path."""
    import long_context_sparse_index_gb300 as dsa
    import torch
    if torch.cuda.is_available():
        pytest.skip("GPU present")
    assert _idx(lib) == dsa.DSA_ERR_CUDA


def test_binding_refuses_cpu_tensors():
    import torch
    import long_context_sparse_index_gb300 as dsa
    q = torch.zeros(8, 2, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        dsa.dsa_index_topk(q, torch.zeros(8, 64, dtype=torch.bfloat16), torch.zeros(8, 2), chunk=4, topk=1)


def test_profile_summaries_match_the_kernel_sources():
    """Each committed ncu summary under profiles/ names the hash of the
    kernel sources it was captured on; the bench reports a kernel's DRAM
    traffic only while that hash still matches.  A kernel edited without a new
    capture fails here instead of dropping its traffic from the bench line."""
    import importlib.util
    import sys
    spec = importlib.util.spec_from_file_location("bench_for_profiles", os.path.join(ROOT, "bench.py"))
    bench = importlib.util.module_from_spec(spec)
    argv = sys.argv
    try:
        sys.argv = ["bench.py"]
        spec.loader.exec_module(bench)
    finally:
        sys.argv = argv
    for kernel in bench.KERNEL_SOURCE:
        traffic, source = bench.profiled_traffic(kernel, 131072)
        assert traffic is not None and traffic > 0, f"{kernel}: {source}"
