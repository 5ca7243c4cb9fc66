"""Pins of the CPU oracle to things other than itself (CPU only).

Each test checks an oracle function against a hand-worked fixture, an exact
identity evaluated another way, a brute-force enumeration, or a textbook
library routine (torch's scaled_dot_product_attention and autograd in fp64),
so that a dropped term, a wrong sign or index, or a transposed operand in the
oracle fails at least one of them.
"""
import itertools
import json
import os

import numpy as np
import pytest
import torch

import oracle
import synth

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def bf16_bits(x):
    """float array -> bf16 bit patterns (the values used here are exact in bf16)."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    back = t.to(torch.float32).numpy()
    assert np.array_equal(back, np.asarray(x, dtype=np.float32)), "fixture value not exact in bf16"
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_round_bits(x):
    """float array -> nearest bf16 bit patterns."""
    t = torch.tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- pooling

def test_pool_keys_golden_summation_order():
    g = load("pool_sum_order.json")
    khat = oracle.pool_keys(bf16_bits(g["k_idx"]))
    assert khat.shape == (1, g["Di"])
    assert np.array_equal(khat, np.array(g["khat"], np.float32))


def test_pool_keys_integer_identity():
    # on integer keys the fp32 mean is exact: 4*Khat equals the integer sum
    k = synth.int_bf16(11, 2, (4 * 37 + 3, 64), -3, 3)
    khat = oracle.pool_keys(k)
    ki = synth.bf16_to_f32(k).astype(np.int64)
    sums = ki[: 4 * 37].reshape(37, 4, 64).sum(axis=1)
    assert khat.shape == (37, 64)
    assert np.array_equal((4 * khat).astype(np.int64), sums)
    assert np.array_equal(4 * khat, sums.astype(np.float32))


# --------------------------------------------------------------------------- indexer scores

def _indexer_fixture():
    g = load("indexer_tiny.json")
    S, Hi, Di = g["S"], g["Hi"], g["Di"]
    q = np.zeros((S, Hi, Di), np.float32)
    w = np.zeros((S, Hi), np.float32)
    for i, v in g["q_idx_nonzero"].items():
        q[int(i)] = v
    for i, v in g["w_nonzero"].items():
        w[int(i)] = v
    return g, bf16_bits(q), bf16_bits(g["k_idx"]), w


def test_index_scores_golden():
    g, q, k, w = _indexer_fixture()
    sc = oracle.index_scores(q, k, w, rows=np.arange(g["S"]))
    for i, exp in g["expected_scores"].items():
        i = int(i)
        assert np.array_equal(sc[i, : i // 4], np.array(exp)), (i, sc[i, : i // 4], exp)
        assert np.all(np.isnan(sc[i, i // 4:]))


def test_index_topk_golden_ties_and_padding():
    g, q, k, w = _indexer_fixture()
    idx, kth = oracle.index_topk(q, k, w, g["topk"])
    for i, exp in g["expected_top1"].items():
        assert idx[int(i), 0] == exp, (i, idx[int(i)], exp)
    assert kth[8] == 6.0 and kth[11] == -2.0 and np.isneginf(kth[0])


@pytest.mark.parametrize("S,Hi", [(64, 3), (203, 8)])
def test_index_scores_unpooled_identity(S, Hi):
    """q.Khat_p = (1/4) sum_t q.k_{4p+t}: computed from the raw keys with an
    integer matmul (library routine), exact on integer inputs."""
    rng_seed = S + Hi
    q = synth.int_bf16(rng_seed, 1, (S, Hi, 64), -3, 3)
    k = synth.int_bf16(rng_seed, 2, (S, 64), -3, 3)
    w = synth.int_f32(rng_seed, 3, (S, Hi), -2, 3)
    sc = oracle.index_scores(q, k, w)
    qi = synth.bf16_to_f32(q).astype(np.int64)
    ki = synth.bf16_to_f32(k).astype(np.int64)
    wi = w.astype(np.int64)
    for i in range(S):
        n = i // 4
        if n == 0:
            continue
        dots4 = qi[i] @ ki[: 4 * n].T                   # [Hi, 4n] token dots, 4x the pooled dot
        pooled4 = dots4.reshape(Hi, n, 4).sum(axis=2)    # 4 * (q . Khat_p)
        exp4 = (wi[i][:, None] * np.maximum(pooled4, 0)).sum(axis=0)
        assert np.array_equal(sc[i, :n] * 4, exp4.astype(np.float64)), i


def test_index_scores_single_head_is_matmul():
    """Hi = 1, w = 1, q and keys positive: every ReLU passes, score = q . Khat."""
    S = 96
    q = bf16_round_bits(np.abs(synth.bf16_to_f32(synth.normal_bf16(5, 1, (S, 1, 64)))) + 0.25)
    k = bf16_round_bits(np.abs(synth.bf16_to_f32(synth.normal_bf16(5, 2, (S, 64)))) + 0.25)
    w = np.ones((S, 1), np.float32)
    sc = oracle.index_scores(q, k, w)
    khat = torch.tensor(synth.bf16_to_f32(k).reshape(S // 4, 4, 64)).double().mean(dim=1)
    full = torch.tensor(synth.bf16_to_f32(q)[:, 0, :]).double() @ khat.T
    for i in range(S):
        n = i // 4
        np.testing.assert_allclose(sc[i, :n], full[i, :n].numpy(), rtol=1e-6, atol=0)


def test_index_scores_causality_and_pool_index():
    """Row i depends only on keys of pools p < floor(i/4); changing token 4p+t
    changes exactly score(i, p)."""
    S, Hi = 48, 4
    # q_idx positive so that a large positive key makes every head's dot positive
    q = bf16_round_bits(np.abs(synth.bf16_to_f32(synth.normal_bf16(9, 1, (S, Hi, 64)))))
    k = synth.normal_bf16(9, 2, (S, 64))
    w = synth.uniform_f32(9, 3, (S, Hi)) + 0.1
    base = oracle.index_scores(q, k, w)
    for tok in (0, 5, 22, 31, 44):
        k2 = k.copy()
        k2[tok] = bf16_bits(np.full(64, 64.0))
        sc = oracle.index_scores(q, k2, w)
        p = tok // 4
        for i in range(S):
            n = i // 4
            changed = np.flatnonzero(sc[i, :n] != base[i, :n])
            assert set(changed.tolist()) <= {p}, (tok, i, changed)
            if p < n:
                assert p in changed.tolist(), (tok, i)


# --------------------------------------------------------------------------- top-k

def test_topk_brute_force_subsets():
    """The kept set is the unique subset T with every member ahead of every
    non-member in (score desc, index asc) order; found by enumeration."""
    rs = np.random.RandomState(0)
    for trial in range(300):
        n = rs.randint(1, 9)
        k = rs.randint(1, 10)
        scores = rs.randint(-2, 3, size=n).astype(np.float64) * 0.5   # many ties
        got, kth = oracle.topk(scores, k)
        m = min(n, k)
        best = None
        for T in itertools.combinations(range(n), m):
            rest = [b for b in range(n) if b not in T]
            if all(scores[a] > scores[b] or (scores[a] == scores[b] and a < b) for a in T for b in rest):
                assert best is None
                best = T
        assert best is not None
        assert list(got[:m]) == list(best) and all(got[m:] == -1), (scores, k, got, best)
        assert kth == min(scores[list(best)])


def test_topk_matches_lexsort():
    rs = np.random.RandomState(1)
    for n, k in [(1000, 64), (5000, 512), (300, 512)]:
        scores = np.round(rs.randn(n) * 4) / 4
        got, _ = oracle.topk(scores, k)
        order = np.lexsort((np.arange(n), -scores.astype(np.float32)))
        m = min(n, k)
        assert np.array_equal(got[:m], np.sort(order[:m])) and np.all(got[m:] == -1)


# --------------------------------------------------------------------------- attention forward

def _torch_dense_masked(q, k, v, mask, scale):
    """Textbook attention through torch SDPA (fp64, CPU): q [S,Hq,D], k,v [S,D], mask [S,S] bool (True = attend)."""
    S, Hq, D = q.shape
    qt = q.permute(1, 0, 2).unsqueeze(0)                    # [1,Hq,S,D]
    kt = k.unsqueeze(0).unsqueeze(0).expand(1, Hq, S, D)
    vt = v.unsqueeze(0).unsqueeze(0).expand(1, Hq, S, D)
    o = torch.nn.functional.scaled_dot_product_attention(qt, kt, vt, attn_mask=mask, scale=scale)
    return o[0].permute(1, 0, 2)


def _mask_from_selection(pool_idx, S):
    m = torch.zeros(S, S, dtype=torch.bool)
    for i in range(S):
        for p in pool_idx[i]:
            if p >= 0:
                m[i, 4 * p: 4 * p + 4] = True
        m[i, 4 * (i // 4): i + 1] = True
    return m


def _attn_inputs(S, Hq, D, seed):
    q = synth.normal_bf16(seed, 4, (S, Hq, D))
    k = synth.normal_bf16(seed, 5, (S, D))
    v = synth.normal_bf16(seed, 6, (S, D))
    dO = synth.normal_bf16(seed, 7, (S, Hq, D))
    return q, k, v, dO


def _t(bits):
    return torch.tensor(synth.bf16_to_f32(bits)).double()


def test_attn_golden_closed_form():
    g = load("attn_tiny.json")
    q, k, v, dO = (bf16_bits(g[x]) for x in ("q", "k", "v", "dO"))
    sel = np.array(g["pool_idx"], np.int32)
    o, lse = oracle.attn_fwd(q, k, v, sel, scale=g["scale"])
    np.testing.assert_allclose(o, g["o"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(lse, g["lse"], rtol=0, atol=1e-14)
    dq = oracle.attn_bwd_dq(dO, q, k, v, sel, scale=g["scale"])
    dk, dv = oracle.attn_bwd_dkdv(dO, q, k, v, sel, scale=g["scale"])
    np.testing.assert_allclose(dq, g["dq"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dk, g["dk"], rtol=0, atol=1e-14)
    np.testing.assert_allclose(dv, g["dv"], rtol=0, atol=1e-14)


@pytest.mark.parametrize("S,topk", [(37, 16), (64, 16)])
def test_attn_all_pools_selected_is_dense_causal(S, topk):
    """With every eligible pool selected the layer is dense causal attention
    (textbook routine: torch SDPA with is_causal, fp64)."""
    Hq, D = 4, 32
    q, k, v, _ = _attn_inputs(S, Hq, D, 21)
    sel = synth.pool_selection(0, 8, S, topk)              # k >= floor(i/4): all pools
    assert np.all((sel >= 0).sum(axis=1) == np.minimum(np.arange(S) // 4, topk))
    o, lse = oracle.attn_fwd(q, k, v, sel)
    qt, kt, vt = _t(q), _t(k), _t(v)
    scale = 1 / np.sqrt(D)
    ref = torch.nn.functional.scaled_dot_product_attention(
        qt.permute(1, 0, 2)[None], kt[None, None].expand(1, Hq, S, D), vt[None, None].expand(1, Hq, S, D),
        is_causal=True, scale=scale)[0].permute(1, 0, 2)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)
    logits = torch.einsum("ihd,jd->ihj", qt, kt) * scale
    causal = torch.ones(S, S, dtype=torch.bool).tril()
    ref_lse = torch.logsumexp(logits.masked_fill(~causal[:, None, :], float("-inf")), dim=-1)
    np.testing.assert_allclose(lse, ref_lse.numpy(), rtol=1e-12, atol=1e-12)


def test_attn_sparse_selection_is_masked_dense():
    """An arbitrary selection equals dense attention under the selection mask."""
    S, Hq, D, topk = 160, 3, 16, 5
    q, k, v, _ = _attn_inputs(S, Hq, D, 22)
    sel = synth.pool_selection(3, 8, S, topk, hot=np.array([2, 7]))
    o, _ = oracle.attn_fwd(q, k, v, sel, scale=0.3)
    ref = _torch_dense_masked(_t(q), _t(k), _t(v), _mask_from_selection(sel, S), 0.3)
    np.testing.assert_allclose(o, ref.numpy(), rtol=1e-12, atol=1e-12)


def test_attn_online_softmax_equals_one_shot():
    """Blockwise online softmax over random key splits reproduces the one-shot
    result (context-parallel lesson, §改进二 and evidence row ②)."""
    S, Hq, D, topk = 200, 2, 8, 12
    q, k, v, _ = _attn_inputs(S, Hq, D, 23)
    sel = synth.pool_selection(4, 8, S, topk)
    o, lse = oracle.attn_fwd(q, k, v, sel)
    qt, kt, vt = _t(q).numpy(), _t(k).numpy(), _t(v).numpy()
    rs = np.random.RandomState(3)
    for i in (5, 77, 199):
        keys = [4 * p + t for p in sel[i] if p >= 0 for t in range(4)] + list(range(4 * (i // 4), i + 1))
        keys = rs.permutation(keys)
        cuts = np.sort(rs.choice(np.arange(1, len(keys)), size=min(3, len(keys) - 1), replace=False))
        for h in range(Hq):
            m, l, acc = -np.inf, 0.0, np.zeros(D)
            for blk in np.split(keys, cuts):
                s = (kt[blk] @ qt[i, h]) / np.sqrt(D)
                m_new = max(m, s.max())
                l = l * np.exp(m - m_new) + np.exp(s - m_new).sum()
                acc = acc * np.exp(m - m_new) + np.exp(s - m_new) @ vt[blk]
                m = m_new
            np.testing.assert_allclose(acc / l, o[i, h], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(m + np.log(l), lse[i, h], rtol=1e-13, atol=1e-13)


def test_attn_rejects_malformed_selection():
    S = 40
    q, k, v, _ = _attn_inputs(S, 2, 8, 24)
    sel = synth.pool_selection(5, 8, S, 4)
    bad = sel.copy()
    bad[30, 0] = 7            # pool 7 is not eligible for query 30 (floor(30/4) = 7)
    with pytest.raises(oracle.OracleError):
        oracle.attn_fwd(q, k, v, bad)
    bad = sel.copy()
    bad[39, :2] = bad[39, 1::-1]   # not ascending
    with pytest.raises(oracle.OracleError):
        oracle.attn_fwd(q, k, v, bad)


# --------------------------------------------------------------------------- attention backward

@pytest.mark.parametrize("dense", [True, False])
def test_attn_backward_matches_autograd(dense):
    """Gradients equal torch autograd through the textbook attention (fp64)."""
    S, Hq, D = 72, 3, 16
    topk = 32 if dense else 3
    q, k, v, dO = _attn_inputs(S, Hq, D, 25 + dense)
    sel = synth.pool_selection(6, 8, S, topk, hot=None if dense else np.array([1, 4]))
    scale = 0.21
    qt, kt, vt = (_t(x).requires_grad_(True) for x in (q, k, v))
    o = _torch_dense_masked(qt, kt, vt, _mask_from_selection(sel, S), scale)
    (o * _t(dO)).sum().backward()
    dq = oracle.attn_bwd_dq(dO, q, k, v, sel, scale=scale)
    dk, dv = oracle.attn_bwd_dkdv(dO, q, k, v, sel, scale=scale)
    np.testing.assert_allclose(dq, qt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dk, kt.grad.numpy(), rtol=1e-10, atol=1e-11)
    np.testing.assert_allclose(dv, vt.grad.numpy(), rtol=1e-10, atol=1e-11)


def test_attn_backward_key_subset_equals_full():
    S, Hq, D, topk = 90, 2, 8, 4
    q, k, v, dO = _attn_inputs(S, Hq, D, 27)
    sel = synth.pool_selection(7, 8, S, topk, hot=np.array([3]))
    dk, dv = oracle.attn_bwd_dkdv(dO, q, k, v, sel)
    keys = np.array([89, 12, 0, 13, 50])
    dk2, dv2 = oracle.attn_bwd_dkdv(dO, q, k, v, sel, key_rows=keys)
    np.testing.assert_allclose(dk2, dk[keys], rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dv2, dv[keys], rtol=1e-13, atol=1e-15)


def test_attn_backward_finite_differences():
    """Central differences of L = sum(dO * o) with respect to single entries."""
    S, Hq, D, topk = 24, 2, 8, 2
    q, k, v, dO = _attn_inputs(S, Hq, D, 28)
    sel = synth.pool_selection(8, 8, S, topk)
    dq = oracle.attn_bwd_dq(dO, q, k, v, sel)
    dk, dv = oracle.attn_bwd_dkdv(dO, q, k, v, sel)
    dOf = synth.bf16_to_f32(dO).astype(np.float64)

    # perturbations must stay exact bf16 values: move one entry by +-2^-4
    def loss(qb, kb, vb):
        o, _ = oracle.attn_fwd(qb, kb, vb, sel)
        return float((o * dOf).sum())

    def shifted(bits, idx, delta):
        f = synth.bf16_to_f32(bits).copy()
        f[idx] += delta
        return bf16_bits(f)

    h = 2.0 ** -4
    rs = np.random.RandomState(4)
    for _ in range(6):
        i, hh, d = rs.randint(S), rs.randint(Hq), rs.randint(D)
        base = synth.bf16_to_f32(q)[i, hh, d]
        if not (abs(base) < 1.9 and base * 16 == np.round(base * 16)):
            # choose a value on the 2^-4 grid so that base +- h is exact in bf16
            qf = synth.bf16_to_f32(q).copy()
            qf[i, hh, d] = 0.5
            q = bf16_bits(qf)
            dq = oracle.attn_bwd_dq(dO, q, k, v, sel)
            dk, dv = oracle.attn_bwd_dkdv(dO, q, k, v, sel)
        fd = (loss(shifted(q, (i, hh, d), h), k, v) - loss(shifted(q, (i, hh, d), -h), k, v)) / (2 * h)
        assert abs(fd - dq[i, hh, d]) < 2e-3 * max(1.0, abs(fd)), (fd, dq[i, hh, d])
        j, d2 = rs.randint(S), rs.randint(D)
        for arr, g, name in ((k, dk, "k"), (v, dv, "v")):
            af = synth.bf16_to_f32(arr).copy()
            af[j, d2] = 0.25
            a0 = bf16_bits(af)
            kk, vv = (a0, v) if name == "k" else (k, a0)
            gk, gv = oracle.attn_bwd_dkdv(dO, q, kk, vv, sel)
            gg = gk if name == "k" else gv
            lp = loss(q, shifted(kk, (j, d2), h) if name == "k" else kk, shifted(vv, (j, d2), h) if name == "v" else vv)
            lm = loss(q, shifted(kk, (j, d2), -h) if name == "k" else kk, shifted(vv, (j, d2), -h) if name == "v" else vv)
            fd = (lp - lm) / (2 * h)
            assert abs(fd - gg[j, d2]) < 2e-3 * max(1.0, abs(fd)), (name, fd, gg[j, d2])


def test_attn_backward_rows_whole_equals_per_key():
    """The row-set backward over every row equals the per-key form (pinned to autograd above)."""
    S, Hq, D, topk = 80, 2, 8, 3
    q, k, v, dO = _attn_inputs(S, Hq, D, 29)
    sel = synth.pool_selection(9, 8, S, topk, hot=np.array([2]))
    dq, dk, dv = oracle.attn_bwd_rows(dO, q, k, v, sel)
    dq2 = oracle.attn_bwd_dq(dO, q, k, v, sel)
    dk2, dv2 = oracle.attn_bwd_dkdv(dO, q, k, v, sel)
    np.testing.assert_allclose(dq, dq2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(dk, dk2, rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(dv, dv2, rtol=1e-12, atol=1e-14)
