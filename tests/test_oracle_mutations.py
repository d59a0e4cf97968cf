"""Plant plausible mistakes in the oracle (on the CPU, by monkeypatching) and
check that the pins in ``test_oracle_pins.py`` catch each of them."""

import math

import numpy as np
import pytest

import oracle
import oracle.sparge_oracle as S
import test_oracle_pins as P


def _patch(monkeypatch, name, fn):
    """Replace an oracle function both in its module and in the package."""
    monkeypatch.setattr(S, name, fn)
    if hasattr(oracle, name):
        monkeypatch.setattr(oracle, name, fn)


def _fails(fn, *args):
    try:
        fn(*args)
    except AssertionError:
        return True
    return False


def _all_select_cases_pass():
    for case in P._load("select_worked_examples.json")["cases"]:
        P.test_selection_worked_examples(case)


def test_pins_catch_reversed_tie_break(monkeypatch):
    def bad_order(prob_row):
        prob_row = np.asarray(prob_row, dtype=np.float64)
        idx = np.arange(prob_row.shape[0])
        return np.lexsort((-idx, -prob_row))
    _patch(monkeypatch, "selection_order", bad_order)
    assert _fails(_all_select_cases_pass)


def test_pins_catch_strict_reach(monkeypatch):
    real = S.topp_count

    def strict(prob_row, p):
        m = real(prob_row, p)
        order = S.selection_order(np.asarray(prob_row, np.float32))
        u = np.floor(np.asarray(prob_row, np.float32).astype(np.float64) * 2.0 ** 40)
        t = float(np.float32(p)) * float(u.sum())
        if 0 < m < len(order) and float(u[order[:m]].sum()) == t:
            return m + 1  # ">" instead of ">="
        return m
    _patch(monkeypatch, "topp_count", strict)
    assert _fails(_all_select_cases_pass)


def test_pins_catch_intersection_instead_of_union(monkeypatch):
    def inter(prob_row, k_frac, p):
        prob_row = np.asarray(prob_row, dtype=np.float32)
        keep = np.zeros(prob_row.shape[0], dtype=bool)
        keep[sorted(S.topk_set(prob_row, k_frac) & S.topp_set(prob_row, p))] = True
        return keep
    _patch(monkeypatch, "hybrid_row", inter)
    assert _fails(_all_select_cases_pass)


def test_pins_catch_floor_instead_of_ceil_for_k(monkeypatch):
    def floor_k(k_frac, mk):
        k = float(np.float32(k_frac))
        return mk if k >= 1 else max(1, min(mk, math.floor(k * mk)))
    _patch(monkeypatch, "topk_count", floor_k)
    assert _fails(P.test_topk_count_table)


def test_pins_catch_pool_dividing_by_block_size(monkeypatch):
    def bad_pool(x, block):
        x = np.asarray(x, dtype=np.float64)
        n = x.shape[-2]
        m = S.num_blocks(n, block)
        out = np.empty(x.shape[:-2] + (m, x.shape[-1]))
        for i in range(m):
            out[..., i, :] = x[..., i * block:min(n, (i + 1) * block), :].sum(-2) / block
        return out
    _patch(monkeypatch, "pool_blocks", bad_pool)
    assert _fails(P.test_pool_ramp_closed_form)


def test_pins_catch_missing_score_scale(monkeypatch):
    _patch(monkeypatch, "_scale", lambda d, scale: 1.0)
    assert _fails(P.test_all_kept_equals_dense_attention_and_sdpa)


def test_pins_catch_dropped_delta_term_in_backward(monkeypatch):
    def no_delta(q, k, v, dout, block_mask, bq, bk, scale=None):
        # same closed form but with D = 0 (dropped term)
        q = np.asarray(q, float); k = np.asarray(k, float); v = np.asarray(v, float)
        dout = np.asarray(dout, float)
        n, d = q.shape[-2], q.shape[-1]
        s = S._scale(d, scale)
        allowed = S.expand_block_mask(block_mask, n, bq, bk)
        sc = np.where(allowed, s * np.einsum("...td,...ud->...tu", q, k), -np.inf)
        m = sc.max(-1, keepdims=True)
        e = np.where(allowed, np.exp(sc - m), 0.0)
        prob = e / e.sum(-1, keepdims=True)
        dv = np.einsum("...tu,...td->...ud", prob, dout)
        ds = prob * np.einsum("...td,...ud->...tu", dout, v)
        return (s * np.einsum("...tu,...ud->...td", ds, k),
                s * np.einsum("...tu,...td->...ud", ds, q), dv)
    _patch(monkeypatch, "sparse_attention_dense_bwd", no_delta)
    assert _fails(P.test_gradients_match_central_finite_differences)


def test_pins_catch_transposed_dk(monkeypatch):
    real = S.sparse_attention_dense_bwd

    def swapped(*a, **kw):
        dq, dk, dv = real(*a, **kw)
        return dq, dv, dk  # dK and dV swapped
    _patch(monkeypatch, "sparse_attention_dense_bwd", swapped)
    assert _fails(P.test_gradients_match_torch_autograd_with_additive_mask)
