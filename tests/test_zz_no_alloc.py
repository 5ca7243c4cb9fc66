"""The allocation-free indexer entry point, dsa_index_topk_noalloc.

It serves callers that cannot allocate device memory where they call the
indexer (a runtime with a fixed device-memory budget, or a path that must not
wait on the device allocator): its scratch is a fixed buffer built into the
library.  These tests call it through the C ABI and require exactly the
pool indices of dsa_index_topk (which takes a caller workspace) on two calls
in a row.  The file is named to be collected last.
"""
import ctypes

import numpy as np
import pytest

import synth

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def lib():
    from long_context_sparse_index_gb300 import build as b
    b.build()
    import long_context_sparse_index_gb300 as dsa
    return dsa.load()


def _bf16(bits):
    return torch.from_numpy(np.ascontiguousarray(bits).view(np.int16)).view(torch.bfloat16).cuda()


def _regular(lib, q, k, w, S, Hi, chunk, topk):
    out = torch.full((S, topk), -7, dtype=torch.int32, device="cuda")
    ws = torch.empty(lib.dsa_index_topk_workspace(S, Hi, 64, chunk, topk), dtype=torch.uint8, device="cuda")
    rc = lib.dsa_index_topk(q.data_ptr(), k.data_ptr(), w.data_ptr(), S, Hi, 64, chunk, topk, 0, S, out.data_ptr(),
                            ws.data_ptr(), ws.numel(), None)
    assert rc == 0, lib.dsa_last_error()
    return out


def _noalloc(lib, q, k, w, S, Hi, chunk, topk):
    out = torch.full((S, topk), -7, dtype=torch.int32, device="cuda")
    rc = lib.dsa_index_topk_noalloc(q.data_ptr(), k.data_ptr(), w.data_ptr(), S, Hi, 64, chunk, topk, 0, S,
                                    out.data_ptr(), None)
    assert rc == 0, lib.dsa_last_error()
    return out


@pytest.mark.gpu
@pytest.mark.parametrize("name", ["tiny_int_s2048", "s16k"])
def test_noalloc_matches_workspace_entry_point_twice(lib, name):
    wl = synth.WORKLOADS[name]
    q_idx, k_idx, w = synth.indexer_inputs(wl)
    q, k, wt = _bf16(q_idx), _bf16(k_idx), torch.from_numpy(w).cuda()
    ref = _regular(lib, q, k, wt, wl.S, wl.Hi, wl.chunk, wl.topk)
    first = _noalloc(lib, q, k, wt, wl.S, wl.Hi, wl.chunk, wl.topk)
    second = _noalloc(lib, q, k, wt, wl.S, wl.Hi, wl.chunk, wl.topk)
    torch.cuda.synchronize()
    assert lib.dsa_sync_status(None) == 0, lib.dsa_last_error()
    # pool indices are integers: compared bit for bit, like every other index test
    assert torch.equal(first, ref)
    assert torch.equal(second, ref)


@pytest.mark.gpu
def test_noalloc_matches_oracle_on_integer_inputs(lib):
    """On the integer workload every score is exact, so the selection is
    unique: the built-in-buffer call must give the oracle's pool indices bit
    for bit, on two calls in a row."""
    import oracle
    wl = synth.WORKLOADS["tiny_int_s2048"]
    q_idx, k_idx, w = synth.indexer_inputs(wl)
    ref, _ = oracle.index_topk(q_idx, k_idx, w, wl.topk)
    q, k, wt = _bf16(q_idx), _bf16(k_idx), torch.from_numpy(w).cuda()
    for _ in range(2):
        got = _noalloc(lib, q, k, wt, wl.S, wl.Hi, wl.chunk, wl.topk)
        torch.cuda.synchronize()
        assert lib.dsa_sync_status(None) == 0, lib.dsa_last_error()
        assert np.array_equal(got.cpu().numpy(), ref)


@pytest.mark.gpu
def test_noalloc_rejects_sizes_beyond_its_buffer(lib):
    import long_context_sparse_index_gb300 as dsa
    S, Hi = 65536, 8
    q = torch.zeros((S, Hi, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.zeros((S, 64), dtype=torch.bfloat16, device="cuda")
    w = torch.zeros((S, Hi), dtype=torch.float32, device="cuda")
    out = torch.full((S, 64), -7, dtype=torch.int32, device="cuda")
    rc = lib.dsa_index_topk_noalloc(q.data_ptr(), k.data_ptr(), w.data_ptr(), S, Hi, 64, 256, 64, 0, S,
                                    out.data_ptr(), None)
    assert rc == dsa.DSA_ERR_WORKSPACE
    assert b"built-in buffer" in lib.dsa_last_error()
    torch.cuda.synchronize()
    assert int((out != -7).sum()) == 0  # nothing ran
