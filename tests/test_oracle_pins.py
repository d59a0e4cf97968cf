"""Pins of the CPU oracle to facts fixed outside the oracle itself.

Each test checks the oracle against a closed form, a hand-derived worked
example (``tests/golden/``), brute force on a tiny input, a library special
case (textbook softmax attention, torch CPU SDPA / autograd) or finite
differences.  Page tags: [P4] is the mindverse page "Optimierung der Effizienz
von Video-Diffusionsmodellen durch SpargeAttention2".
"""

import itertools
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle as O
from conftest import GOLDEN


def _load(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


# --------------------------------------------------------------------------- pooling
def test_pool_ramp_closed_form():
    """[P4 "Maskierungsstrategien"]: block pooling; ramp fixture, partial block."""
    g = _load("pool_ramp.json")
    n, d, b = g["N"], g["d"], g["block"]
    x = np.repeat(np.arange(n, dtype=np.float64)[:, None], d, axis=1)[None, None]
    out = O.pool_blocks(x, b)
    assert out.shape == (1, 1, len(g["means"]), d)
    np.testing.assert_array_equal(out[0, 0, :, 0], np.array(g["means"]))
    np.testing.assert_array_equal(out[0, 0, :, 0], out[0, 0, :, d - 1])


def test_pool_affine_ramp_any_block():
    """Mean of a + c*t over tokens lo..hi-1 is a + c*(lo+hi-1)/2 (closed form)."""
    rng = np.random.default_rng(1)
    for n, b in [(1, 64), (63, 64), (64, 64), (65, 64), (1000, 128), (1031, 7)]:
        a = rng.normal(size=5)
        c = rng.normal(size=5)
        t = np.arange(n, dtype=np.float64)[:, None]
        x = (a[None] + c[None] * t)[None, None]
        out = O.pool_blocks(x, b)[0, 0]
        for i in range(O.num_blocks(n, b)):
            lo, hi = i * b, min(n, (i + 1) * b)
            np.testing.assert_allclose(out[i], a + c * (lo + hi - 1) / 2.0, rtol=1e-12, atol=1e-12)


# --------------------------------------------------------------------------- pooled map
def test_pooled_map_hand_2x2():
    g = _load("pooled_map_2x2.json")
    lg = O.pooled_logits(np.array(g["qbar"], float), np.array(g["kbar"], float), g["scale"])
    np.testing.assert_allclose(lg, np.array(g["logits"]), atol=0, rtol=0)
    pr = O.row_softmax(lg)
    np.testing.assert_allclose(pr, np.array(g["prob"]), rtol=0, atol=1e-15)


def test_pooled_map_rows_are_distributions_and_uniform_on_equal_keys():
    rng = np.random.default_rng(2)
    q = rng.normal(size=(1, 2, 300, 16))
    k = rng.normal(size=(1, 2, 300, 16))
    _, _, lg, pr = O.pooled_map(q, k, 32, 16)
    assert pr.shape == (1, 2, 10, 19)
    np.testing.assert_allclose(pr.sum(-1), 1.0, atol=1e-12)
    assert (pr > 0).all()
    # identical pooled keys -> uniform row
    k2 = np.broadcast_to(rng.normal(size=(1, 1, 1, 16)), (1, 2, 300, 16)).copy()
    _, _, _, pr2 = O.pooled_map(q, k2, 32, 16)
    np.testing.assert_allclose(pr2, 1.0 / 19, atol=1e-15)
    # default scale is 1/sqrt(d)
    qb, kb = O.pool_blocks(q, 32), O.pool_blocks(k, 16)
    np.testing.assert_allclose(lg[0, 1, 3, 5], qb[0, 1, 3] @ kb[0, 1, 5] / 4.0, rtol=1e-13)


# --------------------------------------------------------------------------- selection
def test_topk_count_table():
    g = _load("topk_counts.json")
    for c in g["cases"]:
        assert O.topk_count(c["k_frac"], c["mk"]) == c["K"], c


@pytest.mark.parametrize("case", _load("select_worked_examples.json")["cases"], ids=lambda c: c["name"])
def test_selection_worked_examples(case):
    prob = np.array(case["prob"], dtype=np.float32)
    k, p = case["k_frac"], case["p"]
    assert O.topk_count(k, prob.size) == case["topk_count"]
    assert O.topp_count(prob, p) == case["topp_count"]
    assert O.topk_set(prob, k) == set(case["topk_set"])
    assert O.topp_set(prob, p) == set(case["topp_set"])
    row = O.hybrid_row(prob, k, p)
    assert set(np.nonzero(row)[0].tolist()) == set(case["hybrid_set"])


def _fixed_point(prob):
    return [int(math.floor(float(x) * 2.0 ** 40)) for x in np.asarray(prob, np.float32)]


def test_topp_brute_force_minimum_cardinality():
    """Over all subsets of small rows: m_p is the minimum size of any subset
    whose fixed-point mass reaches p, and the chosen prefix attains it."""
    rng = np.random.default_rng(3)
    for trial in range(60):
        mk = int(rng.integers(1, 11))
        raw = rng.gamma(shape=rng.choice([0.2, 1.0, 5.0]), size=mk)
        if trial % 5 == 0:
            raw = np.round(raw * 3) + 1  # many exact ties
        prob = (raw / raw.sum()).astype(np.float32)
        p = float(np.float32(rng.choice([0.1, 0.5, 0.9, 0.97, rng.uniform()])))
        u = _fixed_point(prob)
        total = sum(u)
        thresh = p * float(total)
        best = None
        for r in range(0, mk + 1):
            for sub in itertools.combinations(range(mk), r):
                if float(sum(u[j] for j in sub)) >= thresh:
                    best = r
                    break
            if best is not None:
                break
        m = O.topp_count(prob, p)
        assert m == best, (prob, p, m, best)
        chosen = O.selection_order(prob)[:m]
        assert float(sum(u[j] for j in chosen)) >= thresh


def test_topp_fixed_point_agrees_with_real_valued_away_from_boundary():
    rng = np.random.default_rng(4)
    for _ in range(200):
        mk = int(rng.integers(2, 600))
        lg = rng.normal(scale=rng.choice([0.1, 1.0, 4.0]), size=mk)
        prob = O.row_softmax(lg).astype(np.float32)
        p = float(np.float32(rng.uniform(0.05, 0.99)))
        m_fp = O.topp_count(prob, p)
        m_re = O.topp_count_real(prob, p)
        if m_fp != m_re:
            cs = np.cumsum(np.sort(prob.astype(np.float64))[::-1]) / prob.astype(np.float64).sum()
            assert np.min(np.abs(cs - p)) < mk * 2.0 ** -38
    # the textbook case: probabilities from a closed form
    prob = np.full(10, 0.1, dtype=np.float32)
    assert O.topp_count(prob, 0.35) == 4


def test_hybrid_invariants():
    rng = np.random.default_rng(5)
    for _ in range(150):
        mk = int(rng.integers(1, 80))
        prob = O.row_softmax(rng.normal(scale=rng.choice([0.05, 1, 5]), size=mk)).astype(np.float32)
        ks = sorted(float(np.float32(x)) for x in rng.uniform(0.001, 1.0, size=2))
        ps = sorted(float(np.float32(x)) for x in rng.uniform(0.0, 1.0, size=2))
        rows = {}
        for k in ks:
            for p in ps:
                row = O.hybrid_row(prob, k, p)
                kept = set(np.nonzero(row)[0].tolist())
                assert kept >= O.topk_set(prob, k)
                assert kept >= O.topp_set(prob, p)
                assert len(kept) >= 1
                c = max(O.topk_count(k, mk), O.topp_count(prob, p))
                assert kept == set(O.selection_order(prob)[:c].tolist())
                rows[(k, p)] = kept
        # monotone in k and in p
        assert rows[(ks[0], ps[0])] <= rows[(ks[1], ps[0])]
        assert rows[(ks[0], ps[0])] <= rows[(ks[0], ps[1])]


def test_mask_encodings():
    mask = np.zeros((1, 1, 3, 40), dtype=bool)
    mask[0, 0, 0, [0, 5, 31, 32, 39]] = True
    mask[0, 0, 2, [1]] = True
    bm = O.pack_bitmask(mask)
    assert bm.shape == (1, 1, 3, 2) and bm.dtype == np.uint32
    assert bm[0, 0, 0, 0] == (1 << 0) | (1 << 5) | (1 << 31)
    assert bm[0, 0, 0, 1] == (1 << 0) | (1 << 7)
    assert bm[0, 0, 1].tolist() == [0, 0]
    assert bm[0, 0, 2].tolist() == [2, 0]
    idx, cnt = O.mask_to_csr(mask)
    assert cnt[0, 0].tolist() == [5, 0, 1]
    assert idx[0, 0, 0, :5].tolist() == [0, 5, 31, 32, 39]
    cidx, ccnt = O.mask_to_csc(mask)
    assert ccnt[0, 0, 0] == 1 and cidx[0, 0, 0, 0] == 0
    assert ccnt[0, 0, 1] == 1 and cidx[0, 0, 1, 0] == 2
    assert ccnt[0, 0].sum() == mask.sum()


# --------------------------------------------------------------------------- attention
def _rand_qkv(rng, b, h, n, d, scale=1.0):
    return [rng.normal(scale=scale, size=(b, h, n, d)) for _ in range(4)]


def _textbook_attention(q, k, v, s):
    sc = s * (q @ np.swapaxes(k, -1, -2))
    sc = sc - sc.max(-1, keepdims=True)
    w = np.exp(sc)
    w = w / w.sum(-1, keepdims=True)
    return w @ v


def test_all_kept_equals_dense_attention_and_sdpa():
    """k = 100% or p >= 1 keeps every block: equals softmax(QK^T s) V."""
    rng = np.random.default_rng(6)
    q, k, v, _ = _rand_qkv(rng, 1, 2, 150, 16)
    mq, mk = O.num_blocks(150, 32), O.num_blocks(150, 16)
    for kf, p in [(1.0, 0.5), (0.05, 1.0)]:
        mask, _ = O.hybrid_mask(q, k, 32, 16, kf, p)
        assert mask.all() and mask.shape == (1, 2, mq, mk)
        out, lse = O.sparse_attention_dense(q, k, v, mask, 32, 16)
        np.testing.assert_allclose(out, _textbook_attention(q, k, v, 0.25), rtol=1e-10, atol=1e-12)
        ref = torch.nn.functional.scaled_dot_product_attention(
            torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v))
        np.testing.assert_allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12)
        lse_ref = np.log(np.exp(0.25 * q @ np.swapaxes(k, -1, -2)).sum(-1))
        np.testing.assert_allclose(lse, lse_ref, rtol=1e-12)


def test_block_mask_equals_sdpa_with_additive_mask():
    rng = np.random.default_rng(7)
    n, bq, bk = 133, 32, 16
    q, k, v, _ = _rand_qkv(rng, 2, 2, n, 8)
    mask = rng.random((2, 2, O.num_blocks(n, bq), O.num_blocks(n, bk))) < 0.3
    mask[..., 0] |= ~mask.any(-1)  # every row keeps a block
    out, _ = O.sparse_attention_dense(q, k, v, mask, bq, bk)
    allowed = O.expand_block_mask(mask, n, bq, bk)
    bias = torch.from_numpy(np.where(allowed, 0.0, -np.inf))
    ref = torch.nn.functional.scaled_dot_product_attention(
        torch.from_numpy(q), torch.from_numpy(k), torch.from_numpy(v), attn_mask=bias)
    np.testing.assert_allclose(out, ref.numpy(), rtol=1e-10, atol=1e-12)


def test_block_gather_equals_dense_and_rows():
    rng = np.random.default_rng(8)
    n, bq, bk = 301, 64, 32
    q, k, v, do = _rand_qkv(rng, 1, 3, n, 16)
    mask = rng.random((1, 3, O.num_blocks(n, bq), O.num_blocks(n, bk))) < 0.4
    mask[0, 1, 2, :] = False  # an empty row: O = 0, LSE = -inf
    o1, l1 = O.sparse_attention_dense(q, k, v, mask, bq, bk)
    o2, l2 = O.sparse_attention_blocks(q, k, v, mask, bq, bk)
    np.testing.assert_allclose(o1, o2, rtol=1e-11, atol=1e-12)
    np.testing.assert_array_equal(np.isinf(l1), np.isinf(l2))
    fin = np.isfinite(l1)
    np.testing.assert_allclose(l1[fin], l2[fin], rtol=1e-12)
    assert np.all(o1[0, 1, 128:192] == 0) and np.all(np.isneginf(l1[0, 1, 128:192]))
    rows = [0, 5, 127, 128, 300]
    o3, l3 = O.sparse_attention_rows(q, k, v, mask, bq, bk, 0, 2, rows)
    np.testing.assert_allclose(o3, o1[0, 2, rows], rtol=1e-11, atol=1e-12)
    g1 = O.sparse_attention_dense_bwd(q, k, v, do, mask, bq, bk)
    g2 = O.sparse_attention_blocks_bwd(q, k, v, do, mask, bq, bk)
    for a, b in zip(g1, g2):
        np.testing.assert_allclose(a, b, rtol=1e-10, atol=1e-12)


def test_single_token_block_returns_its_value():
    """A row whose only kept block holds one token attends to that token only."""
    rng = np.random.default_rng(9)
    n, bq, bk = 65, 32, 64
    q, k, v, _ = _rand_qkv(rng, 1, 1, n, 8)
    mask = np.zeros((1, 1, 3, 2), dtype=bool)
    mask[..., 1] = True  # kv-block 1 = token 64 only
    out, lse = O.sparse_attention_dense(q, k, v, mask, bq, bk)
    np.testing.assert_allclose(out[0, 0], np.broadcast_to(v[0, 0, 64], (n, 8)), rtol=1e-14)
    np.testing.assert_allclose(lse[0, 0], q[0, 0] @ k[0, 0, 64] / math.sqrt(8), rtol=1e-13)


# --------------------------------------------------------------------------- gradients
def test_gradients_match_central_finite_differences():
    rng = np.random.default_rng(10)
    n, d, bq, bk = 200, 16, 32, 16
    q, k, v, do = _rand_qkv(rng, 1, 1, n, d)
    mask = rng.random((1, 1, O.num_blocks(n, bq), O.num_blocks(n, bk))) < 0.35
    mask[..., 0] |= ~mask.any(-1)
    dq, dk, dv = O.sparse_attention_dense_bwd(q, k, v, do, mask, bq, bk)

    def loss(qq, kk, vv):
        o, _ = O.sparse_attention_dense(qq, kk, vv, mask, bq, bk)
        return float((o * do).sum())

    eps = 1e-6
    for t in range(20):
        dirs = [rng.normal(size=q.shape) for _ in range(3)]
        which = t % 4
        if which < 3:  # one input at a time
            dirs = [x if i == which else np.zeros_like(x) for i, x in enumerate(dirs)]
        fd = (loss(q + eps * dirs[0], k + eps * dirs[1], v + eps * dirs[2])
              - loss(q - eps * dirs[0], k - eps * dirs[1], v - eps * dirs[2])) / (2 * eps)
        an = float((dq * dirs[0]).sum() + (dk * dirs[1]).sum() + (dv * dirs[2]).sum())
        assert abs(fd - an) <= 1e-6 * max(1.0, abs(an)), (t, fd, an)


def test_gradients_match_torch_autograd_with_additive_mask():
    rng = np.random.default_rng(11)
    n, d, bq, bk = 97, 8, 16, 16
    q, k, v, do = _rand_qkv(rng, 1, 2, n, d)
    mask = rng.random((1, 2, O.num_blocks(n, bq), O.num_blocks(n, bk))) < 0.5
    mask[..., 0] |= ~mask.any(-1)
    dq, dk, dv = O.sparse_attention_dense_bwd(q, k, v, do, mask, bq, bk)
    tq, tk, tv = (torch.tensor(x, requires_grad=True) for x in (q, k, v))
    bias = torch.from_numpy(np.where(O.expand_block_mask(mask, n, bq, bk), 0.0, -np.inf))
    o = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, attn_mask=bias)
    (o * torch.from_numpy(do)).sum().backward()
    for a, t in ((dq, tq), (dk, tk), (dv, tv)):
        np.testing.assert_allclose(a, t.grad.numpy(), rtol=1e-9, atol=1e-12)
