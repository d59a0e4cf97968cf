"""GPU parity of the block-sparse attention forward with the CPU oracle.
Contract: O within 2e-2 max-abs and 1e-2 relative L2 (bf16 output); LSE
within 2e-3 (fp32).  The oracle runs in fp64 on the same bf16 inputs and the
same block mask."""

import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_attention_sparge_gb300 import binding as B
from block_sparse_attention_sparge_gb300 import synth
from helpers import (LSE_ATOL, O_MAX_ABS, O_REL_L2, check_fwd_heads, mask_to_csr_tensors,
                     rel_l2, to_np, unpack_bitmask)

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _rand(b, h, n, d, seed, scale=1.0, count=3):
    g = torch.Generator().manual_seed(seed)
    return [(scale * torch.randn((b, h, n, d), generator=g)).to(torch.bfloat16)
            for _ in range(count)]


def _compare(o_gpu, lse_gpu, o_ref, lse_ref):
    o = to_np(o_gpu)
    err = np.abs(o - o_ref).max()
    rl = rel_l2(o, o_ref)
    assert err <= O_MAX_ABS and rl <= O_REL_L2, (err, rl)
    lg = to_np(lse_gpu)
    fin = np.isfinite(lse_ref)
    np.testing.assert_array_equal(np.isneginf(lg), ~fin)
    np.testing.assert_allclose(lg[fin], lse_ref[fin], atol=LSE_ATOL, rtol=0)
    return err, rl


def _run_with_mask(q, k, v, mask, scale=0.0):
    ridx, rcnt = mask_to_csr_tensors(mask, DEV)
    o, lse = B.sparge_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), ridx, rcnt, scale,
                               check_status=True)
    torch.cuda.synchronize()
    return o, lse


def test_fwd_tiny_workload_end_to_end():
    """Tiny workload: GPU mask (k=10%, p=0.9) then GPU forward vs fp64 oracle."""
    q, k, v, _ = synth.make_inputs("tiny")
    res = B.sparge_mask(q.to(DEV), k.to(DEV), 0.10, 0.9)
    o, lse = B.sparge_attn_fwd(q.to(DEV), k.to(DEV), v.to(DEV), res["row_idx"], res["row_cnt"],
                               check_status=True)
    torch.cuda.synchronize()
    mask = unpack_bitmask(res["bitmask"], 16)
    o_ref, lse_ref = O.sparse_attention_dense(to_np(q), to_np(k), to_np(v), mask, 128, 64)
    _compare(o, lse, o_ref, lse_ref)


@pytest.mark.parametrize("shape,density,seed", [
    ((1, 2, 1024, 64), 0.3, 1),
    ((1, 3, 1000, 128), 0.4, 2),     # ragged q and kv tails
    ((2, 2, 777, 128), 0.25, 3),
    ((1, 1, 65, 64), 0.5, 4),        # kv-block of one token
    ((1, 1, 1, 128), 1.0, 5),        # one token
    ((1, 2, 200, 64), 0.6, 6),
    ((1, 1, 4096, 128), 0.05, 7),    # long lists across many stages
])
def test_fwd_random_masks(shape, density, seed):
    q, k, v = _rand(*shape, seed=seed)
    n = shape[2]
    mq, mk = O.num_blocks(n, 128), O.num_blocks(n, 64)
    rng = np.random.default_rng(seed)
    mask = rng.random((shape[0], shape[1], mq, mk)) < density
    mask[..., rng.integers(0, mk)] = True
    o, lse = _run_with_mask(q, k, v, mask)
    o_ref, lse_ref = O.sparse_attention_dense(to_np(q), to_np(k), to_np(v), mask, 128, 64)
    _compare(o, lse, o_ref, lse_ref)


def test_fwd_empty_rows_give_zero_and_neg_inf():
    q, k, v = _rand(1, 2, 700, 128, seed=11)
    mq, mk = O.num_blocks(700, 128), O.num_blocks(700, 64)
    mask = np.zeros((1, 2, mq, mk), dtype=bool)
    mask[0, 0, 1, [0, 3]] = True
    mask[0, 1, :, -1] = True
    o, lse = _run_with_mask(q, k, v, mask)
    o_ref, lse_ref = O.sparse_attention_dense(to_np(q), to_np(k), to_np(v), mask, 128, 64)
    _compare(o, lse, o_ref, lse_ref)
    assert torch.count_nonzero(o[0, 0, :128]) == 0


def test_fwd_all_kept_equals_dense_sdpa():
    q, k, v = _rand(1, 2, 1500, 128, seed=12)
    mq, mk = O.num_blocks(1500, 128), O.num_blocks(1500, 64)
    mask = np.ones((1, 2, mq, mk), dtype=bool)
    o, lse = _run_with_mask(q, k, v, mask)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double())
    err = (o.double().cpu() - ref).abs().max().item()
    assert err <= O_MAX_ABS


def test_fwd_large_logits_exercise_rescaling():
    """Scores spanning far more than the lazy-rescale threshold (2^8).  Q and K
    are scaled up; V stays N(0, 1) so the bf16 output keeps its resolution."""
    q, k = _rand(1, 2, 2048, 128, seed=13, scale=3.0, count=2)
    (v,) = _rand(1, 2, 2048, 128, seed=113, count=1)
    mq, mk = O.num_blocks(2048, 128), O.num_blocks(2048, 64)
    mask = np.random.default_rng(13).random((1, 2, mq, mk)) < 0.5
    mask[..., 0] = True
    o, lse = _run_with_mask(q, k, v, mask)
    o_ref, lse_ref = O.sparse_attention_dense(to_np(q), to_np(k), to_np(v), mask, 128, 64)
    _compare(o, lse, o_ref, lse_ref)


def test_fwd_custom_scale():
    q, k, v = _rand(1, 1, 512, 64, seed=14)
    mask = np.random.default_rng(14).random((1, 1, 4, 8)) < 0.5
    mask[..., 2] = True
    o, lse = _run_with_mask(q, k, v, mask, scale=0.3)
    o_ref, lse_ref = O.sparse_attention_dense(to_np(q), to_np(k), to_np(v), mask, 128, 64,
                                              scale=0.3)
    _compare(o, lse, o_ref, lse_ref)


def test_fwd_deterministic():
    q, k, v = _rand(1, 2, 3000, 128, seed=15)
    mq, mk = O.num_blocks(3000, 128), O.num_blocks(3000, 64)
    mask = np.random.default_rng(15).random((1, 2, mq, mk)) < 0.3
    mask[..., 0] = True
    a, la = _run_with_mask(q, k, v, mask)
    b, lb = _run_with_mask(q, k, v, mask)
    assert torch.equal(a, b) and torch.equal(la, lb)


@pytest.fixture(scope="module")
def wan480():
    return synth.make_inputs("wan480")


@pytest.mark.parametrize("k_frac,p", [(0.05, 0.0), (0.05, 0.9)])
def test_fwd_wan480_whole_heads(wan480, k_frac, p):
    """Full 480p shape in the benchmark's launch configuration; every row of
    heads 0 and 11 (O and LSE) against the fp32 block-gather oracle."""
    q, k, v, _ = wan480
    qd, kd, vd = q.to(DEV), k.to(DEV), v.to(DEV)
    res = B.sparge_mask(qd, kd, k_frac, p)
    o, lse = B.sparge_attn_fwd(qd, kd, vd, res["row_idx"], res["row_cnt"], check_status=True)
    torch.cuda.synchronize()
    mask = unpack_bitmask(res["bitmask"], 512)
    check_fwd_heads(q, k, v, mask, o, lse, (0, 11), tag=f"480p k={k_frac} p={p}")
