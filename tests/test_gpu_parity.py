"""GPU parity: the CUDA path through the C ABI against the CPU oracle on the same seeded inputs."""
import ctypes
import os

import numpy as np
import pytest

import oracle
import synth
from tests._util import (assert_close, bits_to_torch, check_selection_scores, check_selection_valid,
                         torch_bf16_to_f64)

torch = pytest.importorskip("torch")
pytestmark = pytest.mark.gpu

if torch.cuda.is_available():
    import long_context_sparse_index_gb300 as dsa
DEV = "cuda"


def _indexer_to_gpu(q_idx, k_idx, w):
    return bits_to_torch(q_idx, DEV), bits_to_torch(k_idx, DEV), torch.from_numpy(w).to(DEV)


def _attn_to_gpu(*arrs):
    return [bits_to_torch(a, DEV) for a in arrs]


# --------------------------------------------------------------------------- indexer + top-k

@pytest.mark.parametrize("chunk", [1, 7, 64, 256, 2048])
def test_index_topk_tiny_int_bit_exact_every_chunk(chunk):
    """Integer inputs: all arithmetic exact, so pool indices are bit-exact,
    and the result is the same for every query chunk."""
    wl = synth.WORKLOADS["tiny_int_s2048"]
    q_idx, k_idx, w = synth.indexer_inputs(wl)
    ref, _ = oracle.index_topk(q_idx, k_idx, w, wl.topk)
    got = dsa.dsa_index_topk(*_indexer_to_gpu(q_idx, k_idx, w), chunk=chunk, topk=wl.topk)
    dsa.dsa_sync_status()
    assert np.array_equal(got.cpu().numpy(), ref)


def test_index_topk_query_range_shards_concatenate():
    """Query-range shards computed separately equal the unsharded call (the
    query-sharded indexer: each shard scores only its own queries)."""
    wl = synth.WORKLOADS["tiny_int_s2048"]
    q, k, w = _indexer_to_gpu(*synth.indexer_inputs(wl))
    full = dsa.dsa_index_topk(q, k, w, chunk=256, topk=wl.topk)
    parts = [dsa.dsa_index_topk(q, k, w, chunk=100, topk=wl.topk, q_begin=a, q_end=b)
             for a, b in ((0, 333), (333, 1024), (1024, 1999), (1999, 2048))]
    dsa.dsa_sync_status()
    assert torch.equal(torch.cat(parts), full)


@pytest.mark.parametrize("S,Hi,topk,chunk", [(1, 1, 1, 1), (2, 3, 1, 5), (3, 1, 4, 2), (4, 2, 1, 4), (5, 1, 1, 3),
                                             (9, 4, 1, 4), (37, 5, 3, 10), (255, 1, 2, 300), (257, 8, 16, 64),
                                             (1023, 2, 64, 129), (1030, 8, 255, 500), (3001, 16, 100, 1000),
                                             (3001, 4, 600, 256), (9001, 2, 2048, 700)])
def test_index_topk_edge_shapes_int(S, Hi, topk, chunk):
    """Ragged S (not a multiple of 4, smaller than a tile), topk larger than
    the available pools, chunk not dividing S, a single head."""
    q_idx = synth.int_bf16(S, 1, (S, Hi, 64), -3, 3)
    k_idx = synth.int_bf16(S, 2, (S, 64), -3, 3)
    w = synth.int_f32(S, 3, (S, Hi), -1, 3)
    ref, _ = oracle.index_topk(q_idx, k_idx, w, topk)
    got = dsa.dsa_index_topk(*_indexer_to_gpu(q_idx, k_idx, w), chunk=chunk, topk=topk)
    dsa.dsa_sync_status()
    assert np.array_equal(got.cpu().numpy(), ref)


def test_index_topk_result_does_not_depend_on_workspace_size():
    """The workspace's slot count only changes how many chunks are in flight:
    the two-slot minimum and the recommended size give the same pool indices
    bit for bit, on float inputs too (S = 20480 also takes the sampled
    thresholds: rows past 4096 pools)."""
    wl = synth.Workload("t", 20480, seed=21)
    q, k, w = _indexer_to_gpu(*synth.indexer_inputs(wl))
    S = wl.S
    full = dsa.dsa_index_topk(q, k, w, chunk=wl.chunk, topk=wl.topk)
    minimum = dsa.index_topk_workspace_size(S, wl.Hi, 64, wl.chunk, wl.topk, slots=2)
    assert minimum < dsa.index_topk_workspace_size(S, wl.Hi, 64, wl.chunk, wl.topk)
    ws = torch.empty(minimum, dtype=torch.uint8, device=DEV)
    small = dsa.dsa_index_topk(q, k, w, chunk=wl.chunk, topk=wl.topk, workspace=ws)
    dsa.dsa_sync_status()
    assert torch.equal(small, full)


@pytest.mark.parametrize("nbuf", [2, 3, 5, 8])
@pytest.mark.parametrize("chunk", [1, 37, 128])
def test_index_topk_every_buffer_ring_size_bit_exact(nbuf, chunk):
    """The fused kernel's item dependencies for every slot-ring size the
    workspace can give (2 to 8 chunk slots; thresholds handed out
    L = min(3, (nbuf-1)/2) steps after their samples and rows L steps after
    their tiles, so L = 0, 1, 2 and 3 here): integer inputs give the oracle's
    pool indices bit for bit."""
    wl = synth.WORKLOADS["tiny_int_s2048"]
    q_idx, k_idx, w = synth.indexer_inputs(wl)
    S = wl.S
    nbytes = dsa.index_topk_workspace_size(S, wl.Hi, 64, chunk, wl.topk, slots=nbuf)
    ws = torch.empty(nbytes, dtype=torch.uint8, device=DEV)
    got = dsa.dsa_index_topk(*_indexer_to_gpu(q_idx, k_idx, w), chunk=chunk, topk=wl.topk, workspace=ws)
    dsa.dsa_sync_status()
    ref, _ = oracle.index_topk(q_idx, k_idx, w, wl.topk)
    assert np.array_equal(got.cpu().numpy(), ref)


def _int_indexer(S, Hi, seed, w_lo=0, w_hi=3):
    return (synth.int_bf16(seed, 1, (S, Hi, 64), -3, 3), synth.int_bf16(seed, 2, (S, 64), -3, 3),
            synth.int_f32(seed, 3, (S, Hi), w_lo, w_hi))


@pytest.mark.parametrize("S,Hi,topk,chunk,slots", [(24577, 8, 64, 256, None), (24577, 8, 512, 256, None),
                                                    (24577, 8, 100, 300, 2), (24577, 8, 512, 1000, 3),
                                                    (40001, 2, 1024, 256, None), (40001, 2, 600, 384, 2)])
def test_index_topk_sampled_thresholds_bit_exact(S, Hi, topk, chunk, slots):
    """Rows past `cap` pools (4096, or 8192 for topk 1024) take their
    candidates from a threshold on every sigma-th pool's score.  Integer inputs
    make every score exact and tie often, so the composite (score, -index)
    threshold and the tie cut at the k-th score are both exercised, for one
    warp per row (topk <= 512) and one 128-thread group per row (topk > 512);
    pool indices equal the oracle's bit for bit, whatever the slot count."""
    q_idx, k_idx, w = _int_indexer(S, Hi, 31 + topk)
    ref, _ = oracle.index_topk(q_idx, k_idx, w, topk)
    ws = None
    if slots is not None:
        ws = torch.empty(dsa.index_topk_workspace_size(S, Hi, 64, chunk, topk, slots=slots), dtype=torch.uint8,
                         device=DEV)
    got = dsa.dsa_index_topk(*_indexer_to_gpu(q_idx, k_idx, w), chunk=chunk, topk=topk, workspace=ws)
    dsa.dsa_sync_status()
    assert np.array_equal(got.cpu().numpy(), ref)


@pytest.mark.parametrize("mode", ["hot_samples", "cold_samples"])
def test_index_topk_fallback_rows_bit_exact(mode):
    """Keys built so that the sampled threshold cannot certify rows: with
    every 64th pool far above the rest ("hot_samples"), the threshold lands
    among those pools and fewer than topk pools reach it; with every 4th pool
    far below the rest ("cold_samples"), nearly every pool reaches it and the
    candidate list overflows.  Those rows go to the fallback kernel, which
    recomputes their scores in full: pool indices still equal the oracle's bit
    for bit, and the call reports the rows it sent there.  (Hot pools all
    tie, so the top-k keeps the lowest-indexed of them.)"""
    S, Hi, topk = 24577, 4, 64
    q_idx = synth.int_bf16(41, 1, (S, Hi, 64), 0, 2)      # non-negative queries and keys: nearly
    k_idx = synth.int_bf16(41, 2, (S, 64), 0, 2)          # every score is positive
    pools = np.arange(S) // 4
    big = np.uint16(0x4100)    # bf16 8.0
    small = np.uint16(0xC100)  # bf16 -8.0
    if mode == "hot_samples":
        k_idx[(pools % 64 == 0)] = big
    else:
        k_idx[(pools % 4 == 0)] = small
    w = np.ones((S, Hi), np.float32)
    ref, _ = oracle.index_topk(q_idx, k_idx, w, topk)
    ws = torch.empty(dsa.index_topk_workspace_size(S, Hi, 64, 256, topk), dtype=torch.uint8, device=DEV)
    got = dsa.dsa_index_topk(*_indexer_to_gpu(q_idx, k_idx, w), chunk=256, topk=topk, workspace=ws)
    dsa.dsa_sync_status()
    assert np.array_equal(got.cpu().numpy(), ref)
    assert dsa.index_topk_stats(ws)["fallback_rows"] > 0


def test_index_topk_all_ties_take_lowest_pools():
    """All scores equal (zero queries): every row keeps pools 0..topk-1."""
    S, Hi, topk = 1500, 4, 17
    q_idx = np.zeros((S, Hi, 64), np.uint16)
    k_idx = synth.int_bf16(5, 2, (S, 64), -3, 3)
    w = np.ones((S, Hi), np.float32)
    got = dsa.dsa_index_topk(*_indexer_to_gpu(q_idx, k_idx, w), chunk=256, topk=topk).cpu().numpy()
    ref, _ = oracle.index_topk(q_idx, k_idx, w, topk)
    assert np.array_equal(got, ref)
    assert np.array_equal(got[-1], np.arange(topk))


def test_index_topk_s16k_float_selection_within_tolerance():
    """bf16 N(0,1) inputs at S=16384, 32 heads, top 512, chunk 256: every GPU
    row is a valid selection and every selected pool scores within 1e-3 of
    the oracle's k-th score."""
    wl = synth.WORKLOADS["s16k"]
    q_idx, k_idx, w = synth.indexer_inputs(wl)
    got = dsa.dsa_index_topk(*_indexer_to_gpu(q_idx, k_idx, w), chunk=wl.chunk, topk=wl.topk).cpu().numpy()
    rows = np.unique(np.concatenate([np.arange(0, 4100, 7), np.arange(wl.S - 64, wl.S),
                                     np.random.RandomState(0).randint(2052, wl.S, 400)]))
    check_selection_valid(got[rows], rows, wl.topk)
    scores = oracle.index_scores(q_idx, k_idx, w, rows=rows)
    ref, kth = oracle.index_topk(q_idx, k_idx, w, wl.topk, rows=rows)
    check_selection_scores(got[rows], rows, scores, kth, wl.topk)
    agree = np.mean([len(np.intersect1d(a[a >= 0], b[b >= 0])) / (b >= 0).sum()
                     for a, b in zip(got[rows], ref) if (b >= 0).any()])
    assert agree > 0.99, agree


# --------------------------------------------------------------------------- query-range sharding

@pytest.mark.parametrize("world", [2, 3])
def test_zigzag_sharded_layer_equals_unsharded(world):
    """Every rank's zig-zag ranges through dsa_index_topk and the range forms
    of the attention calls (local q/o/dO/dq rows, whole-sequence k/v): pool_idx,
    o, lse and dq equal the unsharded calls bit for bit, and the ranges' dk/dv
    contributions add up to the unsharded gradient."""
    wl = synth.WORKLOADS["tiny_int_s2048"]
    q_idx, k_idx, w = synth.indexer_inputs(wl)
    qi, ki, wi = _indexer_to_gpu(q_idx, k_idx, w)
    qt, kt, vt, dOt = _attn_to_gpu(*synth.attention_inputs(wl), synth.grad_output(wl))
    S, scale = wl.S, 0.02
    full_sel = dsa.dsa_index_topk(qi, ki, wi, chunk=256, topk=wl.topk)
    o_full, lse_full = dsa.dsa_sparse_attn_fwd(qt, kt, vt, full_sel, scale=scale)
    dq_full, dk_full, dv_full = dsa.dsa_sparse_attn_bwd(dOt, qt, kt, vt, o_full, lse_full, full_sel, scale=scale)
    sel = torch.full_like(full_sel, -7)
    o, lse, dq = torch.zeros_like(o_full), torch.zeros_like(lse_full), torch.zeros_like(dq_full)
    dk_sum = torch.zeros(dk_full.shape, dtype=torch.float32, device=DEV)
    dv_sum, dk_abs, dv_abs = torch.zeros_like(dk_sum), torch.zeros_like(dk_sum), torch.zeros_like(dk_sum)
    for rank in range(world):
        for b, e in dsa.zigzag_ranges(S, world, rank):
            if b == e:
                continue
            s_ = dsa.dsa_index_topk(qi, ki, wi, chunk=100, topk=wl.topk, q_begin=b, q_end=e)
            ql, dl = qt[b:e].contiguous(), dOt[b:e].contiguous()
            o_, l_ = dsa.dsa_sparse_attn_fwd(ql, kt, vt, s_, scale=scale, q_begin=b)
            dq_, dk_, dv_ = dsa.dsa_sparse_attn_bwd(dl, ql, kt, vt, o_, l_, s_, scale=scale, q_begin=b)
            sel[b:e], o[b:e], lse[b:e], dq[b:e] = s_, o_, l_, dq_
            dk_sum += dk_.float()
            dv_sum += dv_.float()
            dk_abs += dk_.float().abs()
            dv_abs += dv_.float().abs()
    dsa.dsa_sync_status()
    assert torch.equal(sel, full_sel)
    assert torch.equal(o, o_full) and torch.equal(lse, lse_full) and torch.equal(dq, dq_full)
    # each contribution is rounded to bf16 (half an ulp: 2^-9 relative) before the sum
    for got, ref, mag in ((dk_sum, dk_full.float(), dk_abs), (dv_sum, dv_full.float(), dv_abs)):
        assert ((got - ref).abs() <= 2 ** -8 * (mag + ref.abs()) + 1e-6).all()
    ref_sel, _ = oracle.index_topk(q_idx, k_idx, w, wl.topk)
    assert np.array_equal(sel.cpu().numpy(), ref_sel)


# --------------------------------------------------------------------------- packed variable-length batches

def test_varlen_packed_batch_equals_each_sequence_alone():
    """Five sequences packed end to end (lengths 1, 6, 1030, 3, 2051): every
    sequence's pool_idx (counted from its own first token) equals the oracle's
    for that sequence alone, bit for bit, and its forward and backward match
    the oracle run on that sequence alone."""
    lens = [1, 6, 1030, 3, 2051]
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, Hi, topk, scale = int(cu[-1]), 8, 64, 0.05
    q_idx = synth.int_bf16(T, 1, (T, Hi, 64), -3, 3)
    k_idx = synth.int_bf16(T, 2, (T, 64), -3, 3)
    w = synth.int_f32(T, 3, (T, Hi), -1, 3)
    wl = synth.Workload("t", T, topk=topk, seed=17)
    q, k, v = synth.attention_inputs(wl)
    dO = synth.grad_output(wl)
    qi, ki, wi = _indexer_to_gpu(q_idx, k_idx, w)
    qt, kt, vt, dOt = _attn_to_gpu(q, k, v, dO)
    sel = dsa.dsa_index_topk_varlen(qi, ki, wi, cu, chunk=300, topk=topk)
    o, lse = dsa.dsa_sparse_attn_fwd_varlen(qt, kt, vt, sel, cu, scale=scale)
    dq, dk, dv = dsa.dsa_sparse_attn_bwd_varlen(dOt, qt, kt, vt, o, lse, sel, cu, scale=scale)
    dsa.dsa_sync_status()
    sel, go, gl = sel.cpu().numpy(), torch_bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)
    gdq, gdk, gdv = torch_bf16_to_f64(dq), torch_bf16_to_f64(dk), torch_bf16_to_f64(dv)
    for a, b in zip(cu[:-1], cu[1:]):
        ref_sel, _ = oracle.index_topk(q_idx[a:b], k_idx[a:b], w[a:b], topk)
        assert np.array_equal(sel[a:b], ref_sel)
        seq = (q[a:b], k[a:b], v[a:b])
        ro, rl = oracle.attn_fwd(*seq, ref_sel, scale=scale)
        assert_close(go[a:b], ro, "o")
        assert_close(gl[a:b], rl, "lse", bf16_out=False)
        assert_close(gdq[a:b], oracle.attn_bwd_dq(dO[a:b], *seq, ref_sel, scale=scale), "dq")
        rdk, rdv = oracle.attn_bwd_dkdv(dO[a:b], *seq, ref_sel, scale=scale)
        assert_close(gdk[a:b], rdk, "dk")
        assert_close(gdv[a:b], rdv, "dv")


def test_varlen_many_sequences_across_launch_batches():
    """300 packed sequences (more than one 256-sequence launch table; most
    short enough that every row keeps all its pools, some indexed): every
    sequence matches the oracle run on it alone -- pool_idx bit for bit,
    forward and backward within tolerance -- and the record shows the short
    sequences filled without the persistent indexer."""
    rng = np.random.default_rng(5)
    lens = np.concatenate([rng.integers(1, 65, 280), rng.integers(265, 700, 20)])
    rng.shuffle(lens)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, Hi, topk, scale = int(cu[-1]), 8, 64, 0.05
    q_idx = synth.int_bf16(T, 11, (T, Hi, 64), -3, 3)
    k_idx = synth.int_bf16(T, 12, (T, 64), -3, 3)
    w = synth.int_f32(T, 13, (T, Hi), 0, 3)
    wl = synth.Workload("t", T, topk=topk, seed=19)
    q, k, v = synth.attention_inputs(wl)
    dO = synth.grad_output(wl)
    qi, ki, wi = _indexer_to_gpu(q_idx, k_idx, w)
    qt, kt, vt, dOt = _attn_to_gpu(q, k, v, dO)
    sel = dsa.dsa_index_topk_varlen(qi, ki, wi, cu, chunk=256, topk=topk)
    cfg = dsa.last_kernel_config()
    assert cfg["params"]["short_sequences"] == int((lens <= 4 * topk + 4).sum()) == 280
    assert dict(cfg["kernels"])["short_rows"] == 2 and cfg["params"]["indexed_sequences"] == 20
    o, lse = dsa.dsa_sparse_attn_fwd_varlen(qt, kt, vt, sel, cu, scale=scale)
    assert dsa.last_kernel_config()["kernels"] == [["attn_fwd", 2]]
    dq, dk, dv = dsa.dsa_sparse_attn_bwd_varlen(dOt, qt, kt, vt, o, lse, sel, cu, scale=scale)
    assert [n for n, _ in dsa.last_kernel_config()["kernels"]] == ["attn_bwd_pre", "attn_bwd", "attn_bwd_cast"]
    dsa.dsa_sync_status()
    sel, go, gl = sel.cpu().numpy(), torch_bf16_to_f64(o), lse.cpu().numpy().astype(np.float64)
    gdq, gdk, gdv = torch_bf16_to_f64(dq), torch_bf16_to_f64(dk), torch_bf16_to_f64(dv)
    for a, b in zip(cu[:-1], cu[1:]):
        ref_sel, _ = oracle.index_topk(q_idx[a:b], k_idx[a:b], w[a:b], topk)
        assert np.array_equal(sel[a:b], ref_sel), (a, b)
        seq = (q[a:b], k[a:b], v[a:b])
        ro, rl = oracle.attn_fwd(*seq, ref_sel, scale=scale)
        assert_close(go[a:b], ro, "o")
        assert_close(gl[a:b], rl, "lse", bf16_out=False)
        assert_close(gdq[a:b], oracle.attn_bwd_dq(dO[a:b], *seq, ref_sel, scale=scale), "dq")
        rdk, rdv = oracle.attn_bwd_dkdv(dO[a:b], *seq, ref_sel, scale=scale)
        assert_close(gdk[a:b], rdk, "dk")
        assert_close(gdv[a:b], rdv, "dv")


def test_varlen_indexer_same_result_for_any_workspace():
    """Long sequences with few indexer tiles run several at once when the
    workspace holds a slice for each (helper streams, a share of the SMs
    each), else one after another on the caller's stream: the pool indices
    are bit-identical either way, and the oracle's for each sequence alone."""
    rng = np.random.default_rng(9)
    lens = rng.integers(300, 2500, 9)  # topk 64: every sequence runs the indexer, each under 304 tiles
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int64)
    T, Hi, topk = int(cu[-1]), 8, 64
    q_idx = synth.int_bf16(T, 21, (T, Hi, 64), -3, 3)
    k_idx = synth.int_bf16(T, 22, (T, 64), -3, 3)
    w = synth.int_f32(T, 23, (T, Hi), 0, 3)
    qi, ki, wi = _indexer_to_gpu(q_idx, k_idx, w)
    one = dsa.index_topk_workspace_size(int(lens.max()), Hi, 64, 256, topk)
    cu_c = (ctypes.c_int64 * len(cu))(*cu.tolist())
    assert dsa.load().dsa_index_topk_varlen_workspace(cu_c, len(lens), Hi, 64, 256, topk) == 4 * one
    ref = None
    for slices in (1, 2, 3, 4):
        ws = torch.empty(one * slices, dtype=torch.uint8, device=DEV)
        sel = dsa.dsa_index_topk_varlen(qi, ki, wi, cu, chunk=256, topk=topk, workspace=ws)
        params = dsa.last_kernel_config()["params"]
        assert params["helper_streams"] == (slices if slices >= 2 else 0), params
        assert params["indexed_at_once"] == (len(lens) if slices >= 2 else 0), params
        dsa.dsa_sync_status()
        if ref is None:
            ref = sel.clone()
        else:
            assert torch.equal(sel, ref), slices
    got = ref.cpu().numpy()
    for a, b in zip(cu[:-1], cu[1:]):
        ref_sel, _ = oracle.index_topk(q_idx[a:b], k_idx[a:b], w[a:b], topk)
        assert np.array_equal(got[a:b], ref_sel), (a, b)


# --------------------------------------------------------------------------- attention forward

def _fwd_check(q, k, v, sel, rows=None, scale=0.0, fwd=None):
    qt, kt, vt = _attn_to_gpu(q, k, v)
    o, lse = (fwd or dsa.dsa_sparse_attn_fwd)(qt, kt, vt, torch.from_numpy(sel).to(DEV), scale=scale)
    dsa.dsa_sync_status()
    ro, rl = oracle.attn_fwd(q, k, v, sel, scale=scale, rows=rows)
    go = torch_bf16_to_f64(o)
    gl = lse.cpu().numpy().astype(np.float64)
    if rows is not None:
        go, gl = go[rows], gl[rows]
    assert_close(go, ro, "o")
    assert_close(gl, rl, "lse", bf16_out=False)


def test_attn_fwd_tiny_int_with_oracle_selection():
    wl = synth.WORKLOADS["tiny_int_s2048"]
    sel, _ = oracle.index_topk(*synth.indexer_inputs(wl), wl.topk)
    _fwd_check(*synth.attention_inputs(wl), sel)


@pytest.mark.parametrize("S,topk", [(1, 1), (2, 4), (5, 1), (7, 3), (64, 16), (301, 8), (4096, 512), (4099, 100)])
def test_attn_fwd_normal_edge_shapes(S, topk):
    wl = synth.Workload("t", S, topk=topk, seed=S)
    q, k, v = synth.attention_inputs(wl)
    sel = synth.stand_in_selection(wl)
    _fwd_check(q, k, v, sel, scale=0.0 if S % 2 else 0.07)


# The tcgen05 forward: one persistent CTA per SM walks many queries (S > 152
# exercises the query-parity buffers and the producers' row prefetch), and
# topk = 2048 takes its single row-buffer path.
def test_attn_fwd_tc_tiny_int_with_oracle_selection():
    wl = synth.WORKLOADS["tiny_int_s2048"]
    sel, _ = oracle.index_topk(*synth.indexer_inputs(wl), wl.topk)
    _fwd_check(*synth.attention_inputs(wl), sel, fwd=dsa.dsa_sparse_attn_fwd_tc)


@pytest.mark.parametrize("S,topk", [(1, 1), (2, 4), (5, 1), (7, 3), (64, 16), (301, 8), (4096, 512), (4099, 100)])
def test_attn_fwd_tc_normal_edge_shapes(S, topk):
    wl = synth.Workload("t", S, topk=topk, seed=S)
    q, k, v = synth.attention_inputs(wl)
    sel = synth.stand_in_selection(wl)
    _fwd_check(q, k, v, sel, scale=0.0 if S % 2 else 0.07, fwd=dsa.dsa_sparse_attn_fwd_tc)


def test_attn_fwd_tc_topk_2048_sampled_rows():
    wl = synth.Workload("t", 8300, topk=2048, seed=83)
    q, k, v = synth.attention_inputs(wl)
    sel = synth.stand_in_selection(wl)
    rows = np.unique(np.concatenate([np.arange(0, 40), np.random.RandomState(5).randint(0, wl.S, 160),
                                     np.arange(wl.S - 8, wl.S)]))
    _fwd_check(q, k, v, sel, rows=rows, fwd=dsa.dsa_sparse_attn_fwd_tc)


def test_attn_fwd_tc_matches_default_forward():
    """Both forwards on one input: the same softmax, so o agrees to bf16
    rounding and lse to fp32 rounding."""
    wl = synth.Workload("t", 20000, topk=512, seed=11)
    q, k, v = _attn_to_gpu(*synth.attention_inputs(wl))
    sel = torch.from_numpy(synth.stand_in_selection(wl)).to(DEV)
    o1, l1 = dsa.dsa_sparse_attn_fwd(q, k, v, sel)
    o2, l2 = dsa.dsa_sparse_attn_fwd_tc(q, k, v, sel)
    dsa.dsa_sync_status()
    assert (o1.float() - o2.float()).abs().max().item() <= 1.6e-2
    assert (l1 - l2).abs().max().item() <= 1e-4


# --------------------------------------------------------------------------- attention backward

def _bwd_check(q, k, v, dO, sel, q_rows=None, key_rows=None, scale=0.0, deterministic=False):
    qt, kt, vt, dOt = _attn_to_gpu(q, k, v, dO)
    st = torch.from_numpy(sel).to(DEV)
    o, lse = dsa.dsa_sparse_attn_fwd(qt, kt, vt, st, scale=scale)
    bwd = dsa.dsa_sparse_attn_bwd_deterministic if deterministic else dsa.dsa_sparse_attn_bwd
    dq, dk, dv = bwd(dOt, qt, kt, vt, o, lse, st, scale=scale)
    dsa.dsa_sync_status()
    rdq = oracle.attn_bwd_dq(dO, q, k, v, sel, scale=scale, rows=q_rows)
    rdk, rdv = oracle.attn_bwd_dkdv(dO, q, k, v, sel, scale=scale, key_rows=key_rows)
    gdq, gdk, gdv = torch_bf16_to_f64(dq), torch_bf16_to_f64(dk), torch_bf16_to_f64(dv)
    if q_rows is not None:
        gdq = gdq[q_rows]
    if key_rows is not None:
        gdk, gdv = gdk[key_rows], gdv[key_rows]
    assert_close(gdq, rdq, "dq")
    assert_close(gdk, rdk, "dk")
    assert_close(gdv, rdv, "dv")


def test_attn_bwd_tiny_int():
    wl = synth.WORKLOADS["tiny_int_s2048"]
    sel, _ = oracle.index_topk(*synth.indexer_inputs(wl), wl.topk)
    q, k, v = synth.attention_inputs(wl)
    # integer values in [-2, 2] give large logits; a small scale keeps the softmax soft
    _bwd_check(q, k, v, synth.grad_output(wl), sel, scale=0.02)


@pytest.mark.parametrize("S,topk", [(1, 1), (6, 2), (67, 4), (4096, 256), (2051, 512)])
def test_attn_bwd_normal_edge_shapes(S, topk):
    wl = synth.Workload("t", S, topk=topk, seed=100 + S)
    q, k, v = synth.attention_inputs(wl)
    _bwd_check(q, k, v, synth.grad_output(wl), synth.stand_in_selection(wl))


def test_attn_bwd_repeatable_within_rounding():
    """dK/dV use atomic reductions: two runs agree to fp32 rounding."""
    wl = synth.Workload("t", 4096, topk=256, seed=7, values="zipf")
    q, k, v = synth.attention_inputs(wl)
    qt, kt, vt, dOt = _attn_to_gpu(q, k, v, synth.grad_output(wl))
    st = torch.from_numpy(synth.stand_in_selection(wl)).to(DEV)
    o, lse = dsa.dsa_sparse_attn_fwd(qt, kt, vt, st)
    a = dsa.dsa_sparse_attn_bwd(dOt, qt, kt, vt, o, lse, st)
    b = dsa.dsa_sparse_attn_bwd(dOt, qt, kt, vt, o, lse, st)
    assert torch.equal(a[0], b[0])
    for x, y in zip(a[1:], b[1:]):
        # element by element: the fp32 sums differ only in rounding order, so
        # after the bf16 rounding two runs differ by at most one bf16 step of
        # the element itself (a lost or doubled contribution would not)
        xf, yf = x.float(), y.float()
        bound = 2 ** -7 * torch.maximum(xf.abs(), yf.abs()) + 1e-6 * xf.abs().max()
        assert bool(((xf - yf).abs() <= bound).all())


def test_attention_late_large_scores_move_the_softmax_reference():
    """Keys of the upper half of the sequence scaled by 8 (exact in bf16): a
    query's later key blocks (pools ascend) score far above its earlier ones,
    more than 2^8 in probability, so the forwards move their lagging softmax
    reference and rescale the accumulators mid-row.  Both forwards still
    match the oracle.  (The backward is left out: with one key holding ~99 %
    of a row's softmax, Delta = dO . o cancels against dO . v, and the bf16
    rounding of the forward's o, which the backward takes as its input, moves
    dq by as much as dq itself, exactly as the fp64 computation from the
    rounded o shows; the backward's own arithmetic is not involved.)"""
    wl = synth.Workload("t", 2048, topk=128, seed=21)
    q, k, v = synth.attention_inputs(wl)
    f = (k.astype(np.uint32) << 16).view(np.float32).copy()
    f[wl.S // 2:] *= 8.0
    k = (f.view(np.uint32) >> 16).astype(np.uint16)
    sel = synth.stand_in_selection(wl)
    _fwd_check(q, k, v, sel)
    _fwd_check(q, k, v, sel, fwd=dsa.dsa_sparse_attn_fwd_tc)


def test_debug_build_checks_pass_and_results_match():
    """The DSA_DEBUG build (range checks on gathered rows and shared-memory
    offsets that record DSA_ERR_INTERNAL) finds nothing on valid inputs, and
    its results are the default build's: bit for bit, except dK/dV, whose
    atomic sums agree to rounding."""
    from long_context_sparse_index_gb300 import _binding
    from long_context_sparse_index_gb300 import build as libbuild
    dbg = _binding.load_library(libbuild.build(debug=True))
    wl = synth.WORKLOADS["tiny_int_s2048"]
    q_idx, k_idx, w = _indexer_to_gpu(*synth.indexer_inputs(wl))
    q, k, v, dO = _attn_to_gpu(*synth.attention_inputs(wl), synth.grad_output(wl))
    S, topk, chunk = wl.S, wl.topk, wl.chunk
    Hi, Di = q_idx.shape[1], q_idx.shape[2]
    stream = torch.cuda.current_stream().cuda_stream

    def ok(rc):
        assert rc == 0, dbg.dsa_last_error()

    ref_sel = dsa.dsa_index_topk(q_idx, k_idx, w, chunk=chunk, topk=topk)
    ref_o, ref_lse = dsa.dsa_sparse_attn_fwd(q, k, v, ref_sel)
    ref_otc, ref_lsetc = dsa.dsa_sparse_attn_fwd_tc(q, k, v, ref_sel)
    ref_g = dsa.dsa_sparse_attn_bwd(dO, q, k, v, ref_o, ref_lse, ref_sel)
    dsa.dsa_sync_status()

    sel = torch.empty_like(ref_sel)
    ws = torch.empty(dbg.dsa_index_topk_workspace(S, Hi, Di, chunk, topk), dtype=torch.uint8, device=DEV)
    ok(dbg.dsa_index_topk(q_idx.data_ptr(), k_idx.data_ptr(), w.data_ptr(), S, Hi, Di, chunk, topk, 0, S,
                          sel.data_ptr(), ws.data_ptr(), ws.numel(), stream))
    o, lse = torch.empty_like(ref_o), torch.empty_like(ref_lse)
    otc, lsetc = torch.empty_like(ref_o), torch.empty_like(ref_lse)
    Hq, D = q.shape[1], q.shape[2]
    for fn, oo, ll in ((dbg.dsa_sparse_attn_fwd, o, lse), (dbg.dsa_sparse_attn_fwd_tc, otc, lsetc)):
        ok(fn(q.data_ptr(), k.data_ptr(), v.data_ptr(), sel.data_ptr(), S, Hq, D, topk, 0.0, oo.data_ptr(),
              ll.data_ptr(), stream))
    g = [torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)]
    wsb = torch.empty(dbg.dsa_sparse_attn_bwd_workspace(S, Hq, D), dtype=torch.uint8, device=DEV)
    ok(dbg.dsa_sparse_attn_bwd(dO.data_ptr(), q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(), lse.data_ptr(),
                               sel.data_ptr(), S, Hq, D, topk, 0.0, g[0].data_ptr(), g[1].data_ptr(), g[2].data_ptr(),
                               wsb.data_ptr(), wsb.numel(), stream))
    assert dbg.dsa_sync_status(None) == 0, dbg.dsa_last_error()
    assert torch.equal(sel, ref_sel)
    assert torch.equal(o, ref_o) and torch.equal(lse, ref_lse)
    assert torch.equal(otc, ref_otc) and torch.equal(lsetc, ref_lsetc)
    assert torch.equal(g[0], ref_g[0])
    for x, y in zip(g[1:], ref_g[1:]):
        xf, yf = x.float(), y.float()
        bound = 2 ** -7 * torch.maximum(xf.abs(), yf.abs()) + 1e-6 * xf.abs().max()
        assert bool(((xf - yf).abs() <= bound).all())


# --------------------------------------------------------------------------- deterministic backward

def test_attn_bwd_deterministic_tiny_int():
    wl = synth.WORKLOADS["tiny_int_s2048"]
    sel, _ = oracle.index_topk(*synth.indexer_inputs(wl), wl.topk)
    q, k, v = synth.attention_inputs(wl)
    _bwd_check(q, k, v, synth.grad_output(wl), sel, scale=0.02, deterministic=True)


# S < 4 (no selectable pool), a ragged last pool, pool lists longer than one
# 1024-query segment (S=4096, 2051 at top 256/512), and a topk that is not a
# power of two
@pytest.mark.parametrize("S,topk", [(1, 1), (3, 2), (6, 2), (67, 4), (4096, 256), (2051, 512), (5003, 37)])
def test_attn_bwd_deterministic_normal_edge_shapes(S, topk):
    wl = synth.Workload("t", S, topk=topk, seed=200 + S)
    q, k, v = synth.attention_inputs(wl)
    _bwd_check(q, k, v, synth.grad_output(wl), synth.stand_in_selection(wl), deterministic=True)


def test_attn_bwd_deterministic_bit_reproducible_and_near_default():
    """Zipf-popular pools (the longest per-pool query lists): two runs give the
    same bits for dq, dk and dv, and they agree with the atomic default within
    the parity tolerance."""
    wl = synth.Workload("t", 8192, topk=256, seed=11, values="zipf")
    q, k, v = synth.attention_inputs(wl)
    qt, kt, vt, dOt = _attn_to_gpu(q, k, v, synth.grad_output(wl))
    st = torch.from_numpy(synth.stand_in_selection(wl)).to(DEV)
    o, lse = dsa.dsa_sparse_attn_fwd(qt, kt, vt, st)
    a = dsa.dsa_sparse_attn_bwd_deterministic(dOt, qt, kt, vt, o, lse, st)
    torch.cuda.synchronize()
    torch.cuda.empty_cache()
    b = dsa.dsa_sparse_attn_bwd_deterministic(dOt, qt, kt, vt, o, lse, st)
    ref = dsa.dsa_sparse_attn_bwd(dOt, qt, kt, vt, o, lse, st)
    dsa.dsa_sync_status()
    for x, y, r, name in zip(a, b, ref, ("dq", "dk", "dv")):
        assert torch.equal(x, y), name
        assert_close(torch_bf16_to_f64(x), torch_bf16_to_f64(r), name)


def test_attn_bwd_deterministic_rejects_small_workspace():
    wl = synth.Workload("t", 256, topk=8, seed=4)
    q, k, v = _attn_to_gpu(*synth.attention_inputs(wl))
    st = torch.from_numpy(synth.stand_in_selection(wl)).to(DEV)
    o, lse = dsa.dsa_sparse_attn_fwd(q, k, v, st)
    need = dsa.sparse_attn_bwd_deterministic_workspace_size(256, 16, 128, 8)
    ws = torch.empty(need - 256, dtype=torch.uint8, device=DEV)
    with pytest.raises(dsa.DsaError) as ei:
        dsa.dsa_sparse_attn_bwd_deterministic(q, q, k, v, o, lse, st, workspace=ws)
    assert ei.value.status == dsa.DSA_ERR_WORKSPACE


# --------------------------------------------------------------------------- device status / bounded waits

def test_bounded_wait_timeout_reports_status():
    """With fault injection the indexer's producer issues no copies, so every
    bounded wait runs out; the kernels return, the host reads DSA_ERR_TIMEOUT,
    and the context stays usable."""
    wl = synth.WORKLOADS["tiny_int_s2048"]
    q, k, w = _indexer_to_gpu(*synth.indexer_inputs(wl))
    dsa.dsa_clear_status()
    os.environ["DSA_FAULT_INJECT"] = "timeout"
    try:
        dsa.dsa_index_topk(q, k, w, chunk=2048, topk=wl.topk)
        with pytest.raises(dsa.DsaError) as ei:
            dsa.dsa_sync_status()
        assert ei.value.status == dsa.DSA_ERR_TIMEOUT
    finally:
        del os.environ["DSA_FAULT_INJECT"]
    dsa.dsa_clear_status()
    got = dsa.dsa_index_topk(q, k, w, chunk=2048, topk=wl.topk)
    dsa.dsa_sync_status()
    ref, _ = oracle.index_topk(*synth.indexer_inputs(wl), wl.topk)
    assert np.array_equal(got.cpu().numpy(), ref)


def test_malformed_selection_is_reported_not_read():
    """An ineligible pool index is never dereferenced and is reported as DSA_ERR_INTERNAL."""
    S, topk = 256, 8
    wl = synth.Workload("t", S, topk=topk, seed=3)
    q, k, v = _attn_to_gpu(*synth.attention_inputs(wl))
    sel = synth.stand_in_selection(wl)
    sel[200, 0] = 10 ** 6
    dsa.dsa_clear_status()
    dsa.dsa_sparse_attn_fwd(q, k, v, torch.from_numpy(sel).to(DEV))
    with pytest.raises(dsa.DsaError) as ei:
        dsa.dsa_sync_status()
    assert ei.value.status == dsa.DSA_ERR_INTERNAL
    dsa.dsa_clear_status()
    # the deterministic backward leaves the entry out of its lists and reports it too
    good = torch.from_numpy(synth.stand_in_selection(wl)).to(DEV)
    o, lse = dsa.dsa_sparse_attn_fwd(q, k, v, good)
    dsa.dsa_sync_status()
    dsa.dsa_sparse_attn_bwd_deterministic(q, q, k, v, o, lse, torch.from_numpy(sel).to(DEV))
    with pytest.raises(dsa.DsaError) as ei:
        dsa.dsa_sync_status()
    assert ei.value.status == dsa.DSA_ERR_INTERNAL
    dsa.dsa_clear_status()
    # the tcgen05 forward reports it the same way, and only that row changes
    o_tc, _ = dsa.dsa_sparse_attn_fwd_tc(q, k, v, torch.from_numpy(sel).to(DEV))
    with pytest.raises(dsa.DsaError) as ei:
        dsa.dsa_sync_status()
    assert ei.value.status == dsa.DSA_ERR_INTERNAL
    dsa.dsa_clear_status()
    keep = torch.arange(S, device=DEV) != 200
    assert (o_tc[keep].float() - o[keep].float()).abs().max().item() <= 1.6e-2


def test_binding_refuses_bad_outputs_and_shapes():
    """Caller-supplied outputs and workspaces must be contiguous CUDA tensors
    of the right dtype and shape, and the inputs' extents must agree: a host
    pointer or a short buffer never reaches a kernel."""
    wl = synth.Workload("t", 64, topk=8, seed=5)
    q, k, v = _attn_to_gpu(*synth.attention_inputs(wl))
    st = torch.from_numpy(synth.stand_in_selection(wl)).to(DEV)
    with pytest.raises(ValueError):
        dsa.dsa_sparse_attn_fwd(q, k, v, st, o=torch.empty(q.shape, dtype=torch.bfloat16))  # host tensor
    with pytest.raises(ValueError):
        dsa.dsa_sparse_attn_fwd(q, k, v, st, lse=torch.empty((63, 16), dtype=torch.float32, device=DEV))
    with pytest.raises(ValueError):
        dsa.dsa_sparse_attn_fwd(q, k, v, st[:32])
    o, lse = dsa.dsa_sparse_attn_fwd(q, k, v, st)
    with pytest.raises(ValueError):
        dsa.dsa_sparse_attn_bwd(q, q, k, v, o, lse[:32], st)
    with pytest.raises(ValueError):
        dsa.dsa_sparse_attn_bwd(q, q, k, v, o, lse, st, workspace=torch.empty(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError):
        dsa.dsa_sparse_attn_bwd_deterministic(q, q, k, v, o, lse, st, dk=torch.empty((64, 64), dtype=torch.bfloat16,
                                                                                       device=DEV))
    dsa.dsa_sync_status()


def test_last_kernel_config_names_the_kernels_that_ran():
    """Each call's record names the kernels it launched, in order, and its plan."""
    wl = synth.WORKLOADS["tiny_int_s2048"]
    q, k, w = _indexer_to_gpu(*synth.indexer_inputs(wl))
    sel = dsa.dsa_index_topk(q, k, w, chunk=wl.chunk, topk=wl.topk)
    cfg = dsa.last_kernel_config()
    assert cfg["entry"] == "dsa_index_topk"
    assert [name for name, _ in cfg["kernels"]] == ["pool_keys", "index_topk", "index_fallback"]
    assert cfg["params"]["topk"] == wl.topk and cfg["params"]["chunk"] == wl.chunk
    assert 1 <= cfg["params"]["chunk_slots"] <= 8
    wa = synth.Workload("t", 4096, topk=256, seed=7)
    qa, ka, va = synth.attention_inputs(wa)
    qt, kt, vt, dOt = _attn_to_gpu(qa, ka, va, synth.grad_output(wa))
    st = torch.from_numpy(synth.stand_in_selection(wa)).to(DEV)
    o, lse = dsa.dsa_sparse_attn_fwd(qt, kt, vt, st)
    cfg = dsa.last_kernel_config()
    # the binding calls the range form, which the record names
    assert cfg["entry"] in ("dsa_sparse_attn_fwd", "dsa_sparse_attn_fwd_range") and cfg["kernels"] == [["attn_fwd", 1]]
    dsa.dsa_sparse_attn_bwd(dOt, qt, kt, vt, o, lse, st)
    cfg = dsa.last_kernel_config()
    assert cfg["variant"].startswith("atomic")
    assert [name for name, _ in cfg["kernels"]] == ["attn_bwd_pre", "attn_bwd", "attn_bwd_cast"]
    dsa.dsa_sparse_attn_bwd_deterministic(dOt, qt, kt, vt, o, lse, st)
    cfg = dsa.last_kernel_config()
    assert cfg["variant"].startswith("deterministic")
    assert dict(cfg["kernels"])["det_span"] == cfg["params"]["spans"]
    torch.cuda.synchronize()
    assert sel.shape == (wl.S, wl.topk)
