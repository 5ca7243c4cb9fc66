"""Query-range sharding of the layer (context parallelism), host side, on the CPU.

A rank that holds only some of the sequence's queries runs the layer on its
own query ranges, with global positions ([CP-lesson §改进二]: the sequence is
split across GPUs by query rows; every rank still sees all keys).  Under
zig-zag sharding the sequence is cut into 2N segments and rank r takes
segments r and 2N-1-r, which equalises the causal work.  These tests pin the
ranges libdsa hands out (dsa_zigzag_ranges) to the pages' worked example and
closed form, and run the sharded path with two gloo ranks: each rank computes
its ranges with the oracle and the int32 pool indices are all-gathered, as the
pages' query-sharded indexer does.  GPU runs of the same ranges are in
test_gpu_parity.py.
"""
import os
import socket

import numpy as np
import pytest

import oracle
import synth

torch = pytest.importorskip("torch")


@pytest.fixture(scope="module")
def dsa():
    from long_context_sparse_index_gb300 import build as b
    b.build()
    import long_context_sparse_index_gb300 as d
    return d


def _causal_pairs(b, e):
    """(i, j) pairs with j <= i for queries i in [b, e): sum of (i + 1)."""
    return sum(i + 1 for i in range(b, e))


def _rank_pairs(dsa, S, world, count=_causal_pairs):
    return [sum(count(b, e) for b, e in dsa.zigzag_ranges(S, world, r)) for r in range(world)]


def test_zigzag_worked_example(dsa):
    """[CP-lesson §改进二]: 16 tokens on 4 GPUs: a contiguous split gives the
    GPUs 10 : 26 : 42 : 58 causal pairs, zig-zag gives each of them 34; with
    32 tokens on 8 GPUs zig-zag is again exactly equal."""
    S, N = 16, 4
    contiguous = [_causal_pairs(r * S // N, (r + 1) * S // N) for r in range(N)]
    assert contiguous == [10, 26, 42, 58]
    assert _rank_pairs(dsa, S, N) == [34, 34, 34, 34]
    per = _rank_pairs(dsa, 32, 8)
    assert len(set(per)) == 1 and sum(per) == 32 * 33 // 2


@pytest.mark.parametrize("N", [1, 2, 3, 4, 8])
@pytest.mark.parametrize("a", [1, 2, 5, 9])
def test_zigzag_closed_form(dsa, N, a):
    """Segment k (length a) holds k*a^2 + a(a+1)/2 causal pairs, so ranks r
    and 2N-1-r pair up to (2N-1)*a^2 + a(a+1) whatever r is."""
    for k in range(2 * N):
        assert _causal_pairs(k * a, (k + 1) * a) == k * a * a + a * (a + 1) // 2
    S = 2 * N * a
    assert _rank_pairs(dsa, S, N) == [(2 * N - 1) * a * a + a * (a + 1)] * N


@pytest.mark.parametrize("S", [1, 2, 7, 16, 1000, 2051, 131072])
@pytest.mark.parametrize("N", [1, 2, 3, 5, 8])
def test_zigzag_ranges_partition_the_sequence(dsa, S, N):
    covered = np.zeros(S, np.int32)
    for r in range(N):
        for b, e in dsa.zigzag_ranges(S, N, r):
            assert 0 <= b <= e <= S
            covered[b:e] += 1
    assert (covered == 1).all()


def test_zigzag_balances_the_indexer_work(dsa):
    """The indexer's work for query i is floor(i/4) pools: zig-zag keeps the
    ranks within 0.1% of each other at S = 131072 on 8 ranks, where a
    contiguous split's slowest rank does 1.87x the mean."""
    S, N = 131072, 8
    i = np.arange(S, dtype=np.int64)
    pools = i // 4
    per = [sum(int(pools[b:e].sum()) for b, e in dsa.zigzag_ranges(S, N, r)) for r in range(N)]
    assert max(per) / min(per) < 1.001
    contiguous = [int(pools[r * S // N:(r + 1) * S // N].sum()) for r in range(N)]
    assert max(contiguous) / np.mean(contiguous) > 1.8


def test_zigzag_rejects_bad_arguments(dsa):
    for S, N, r in ((0, 2, 0), (16, 0, 0), (16, 2, 2), (16, 2, -1)):
        with pytest.raises(dsa.DsaError) as ei:
            dsa.zigzag_ranges(S, N, r)
        assert ei.value.status == dsa.DSA_ERR_INVALID_ARG


# --------------------------------------------------------------------------- two gloo ranks

def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _init(rank, world, port):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)


def _sharded_layer_worker(rank, world, port):
    """One rank: its zig-zag ranges of the tiny integer workload through the
    oracle (indexer + top-k, then the forward), then an all-gather of every
    rank's rows; rank 0 checks the assembled result against the unsharded
    oracle."""
    import long_context_sparse_index_gb300 as d
    _init(rank, world, port)
    try:
        wl = synth.WORKLOADS["tiny_int_s2048"]
        q_idx, k_idx, w = synth.indexer_inputs(wl)
        q, k, v = synth.attention_inputs(wl)
        S = wl.S
        rows = np.concatenate([np.arange(b, e) for b, e in d.zigzag_ranges(S, world, rank)]).astype(np.int64)
        sel_mine, _ = oracle.index_topk(q_idx, k_idx, w, wl.topk, rows=rows)
        full_sel = np.full((S, wl.topk), -1, np.int32)
        full_sel[rows] = sel_mine
        _, lse_mine = oracle.attn_fwd(q, k, v, full_sel, scale=0.02, rows=rows)
        # all-gather: rows, pool indices and lse of every rank (equal shard sizes: 2 | S)
        g_rows = [torch.empty(rows.size, dtype=torch.int64) for _ in range(world)]
        g_sel = [torch.empty(sel_mine.shape, dtype=torch.int32) for _ in range(world)]
        g_lse = [torch.empty(lse_mine.shape, dtype=torch.float64) for _ in range(world)]
        torch.distributed.all_gather(g_rows, torch.from_numpy(rows))
        torch.distributed.all_gather(g_sel, torch.from_numpy(np.ascontiguousarray(sel_mine)))
        torch.distributed.all_gather(g_lse, torch.from_numpy(lse_mine))
        if rank == 0:
            sel = np.full((S, wl.topk), -7, np.int32)
            lse = np.full((S, wl.Hq), np.nan)
            for r_, s_, l_ in zip(g_rows, g_sel, g_lse):
                sel[r_.numpy()] = s_.numpy()
                lse[r_.numpy()] = l_.numpy()
            ref_sel, _ = oracle.index_topk(q_idx, k_idx, w, wl.topk)
            assert np.array_equal(sel, ref_sel)
            _, ref_lse = oracle.attn_fwd(q, k, v, ref_sel, scale=0.02)
            assert np.array_equal(lse, ref_lse)
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_zigzag_sharded_indexer_and_forward(dsa):
    torch.multiprocessing.spawn(_sharded_layer_worker, args=(2, _free_port()), nprocs=2, join=True)


def _sharded_backward_worker(rank, world, port):
    """One rank: the backward of its zig-zag ranges through the oracle (its dq
    rows and its contribution to every key's dK/dV), then the two exchanges a
    context-parallel backward needs: an all-reduce that sums the ranks' dK/dV
    contributions and an all-gather of the dq rows; every rank checks the sums
    against the unsharded oracle backward."""
    import long_context_sparse_index_gb300 as d
    _init(rank, world, port)
    try:
        wl = synth.WORKLOADS["tiny_int_s2048"]
        sel, _ = oracle.index_topk(*synth.indexer_inputs(wl), wl.topk)
        q, k, v = synth.attention_inputs(wl)
        dO = synth.grad_output(wl)
        S = wl.S
        rows = np.concatenate([np.arange(b, e) for b, e in d.zigzag_ranges(S, world, rank)]).astype(np.int64)
        dq_mine, dk_mine, dv_mine = oracle.attn_bwd_rows(dO, q, k, v, sel, scale=0.02, rows=rows)
        dk_t, dv_t = torch.from_numpy(dk_mine.copy()), torch.from_numpy(dv_mine.copy())
        torch.distributed.all_reduce(dk_t)
        torch.distributed.all_reduce(dv_t)
        g_rows = [torch.empty(rows.size, dtype=torch.int64) for _ in range(world)]
        g_dq = [torch.empty(dq_mine.shape, dtype=torch.float64) for _ in range(world)]
        torch.distributed.all_gather(g_rows, torch.from_numpy(rows))
        torch.distributed.all_gather(g_dq, torch.from_numpy(dq_mine))
        ref_dq, ref_dk, ref_dv = oracle.attn_bwd_rows(dO, q, k, v, sel, scale=0.02)
        dq = np.full_like(ref_dq, np.nan)
        for r_, g_ in zip(g_rows, g_dq):
            dq[r_.numpy()] = g_.numpy()
        assert np.array_equal(dq, ref_dq)
        # integer inputs: every contribution is a dyadic rational far from fp64
        # rounding, so the two-term sum is the unsharded sum up to rounding order
        scale = np.abs(ref_dk).max() + np.abs(ref_dv).max()
        assert np.abs(dk_t.numpy() - ref_dk).max() <= 1e-12 * scale
        assert np.abs(dv_t.numpy() - ref_dv).max() <= 1e-12 * scale
        # each rank's contribution alone is not the whole gradient
        assert np.abs(dk_mine - ref_dk).max() > 1e-3
        torch.distributed.barrier()
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_zigzag_sharded_backward_sums_dkdv(dsa):
    torch.multiprocessing.spawn(_sharded_backward_worker, args=(2, _free_port()), nprocs=2, join=True)


def _max_worker(rank, world, port):
    import bench
    _init(rank, world, port)
    try:
        got = bench.max_over_ranks(1.5 + rank, torch.device("cpu"))
        assert got == 1.5 + world - 1
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_benchmark_takes_the_slowest_rank():
    """bench.py times N ranks as the slowest rank's time (max over ranks)."""
    torch.multiprocessing.spawn(_max_worker, args=(2, _free_port()), nprocs=2, join=True)


@pytest.mark.parametrize("n", [1, 2, 8, 64])
def test_benchmark_varlen_mix_partitions_the_tokens(n):
    """bench.py --varlen N packs the workload's S tokens as N sequences of a
    seeded length mix: positive multiples of 256 that sum to S, the same mix
    on every run."""
    import bench
    S = 131072
    lens = bench.varlen_lengths(S, n)
    assert len(lens) == n and int(lens.sum()) == S
    assert (lens > 0).all() and (lens % 256 == 0).all()
    assert (bench.varlen_lengths(S, n) == lens).all()


@pytest.mark.parametrize("S,topk", [(1, 1), (7, 2), (1030, 64), (4099, 512)])
def test_benchmark_work_counts_match_brute_force(S, topk):
    """The roofline's units: query i scores floor(i/4) pools and attends to
    4 * min(topk, floor(i/4)) selected keys plus its own i mod 4 + 1."""
    import bench
    import synth
    wl = synth.Workload("t", S, topk=topk, seed=1)
    pairs, keys = bench.workload_counts(wl)
    assert pairs == sum(i // 4 for i in range(S))
    assert keys == sum(4 * min(topk, i // 4) + (i - 4 * (i // 4)) + 1 for i in range(S))
    w = bench.algorithmic_work(wl)
    assert w["index_topk"]["flops"] == 2 * wl.Hi * wl.Di * pairs
