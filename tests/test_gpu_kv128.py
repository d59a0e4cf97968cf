"""The 128-key kv-block variant (block_kv = 128): the mask is chosen on blocks
of 128 queries by 128 keys, and the forward and backward compute the kept
128 x 128 tiles.  The pages fix no block size ("Block-dünnbesetzte
Aufmerksamkeit": the tile is the kept unit); the oracle takes the block size
as a parameter.  Same contract as the 128 x 64 tests: the mask bit-exact on
the GPU's P, pooled map within 1e-3, O within 2e-2 max-abs / 1e-2 rel-L2, LSE
within 2e-3, dQ, dK, dV within 5e-2 rel-L2."""

import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_attention_sparge_gb300 import binding as B
from block_sparse_attention_sparge_gb300 import synth
from helpers import (GRAD_REL_L2, LSE_ATOL, MAP_ATOL, O_MAX_ABS, O_REL_L2, check_bwd_heads,
                     check_fwd_heads, mask_to_csc_tensors, mask_to_csr_tensors, rel_l2, to_np,
                     unpack_bitmask)

pytestmark = pytest.mark.gpu
DEV = "cuda"
BK = 128


def _rand(b, h, n, d, seed, count=4):
    g = torch.Generator().manual_seed(seed)
    return [torch.randn((b, h, n, d), generator=g).to(torch.bfloat16) for _ in range(count)]


@pytest.mark.parametrize("shape,density,seed", [
    ((1, 2, 1024, 64), 0.3, 1),
    ((1, 3, 1000, 128), 0.4, 2),     # ragged q and kv tails
    ((2, 1, 777, 128), 0.35, 3),
    ((1, 1, 65, 128), 1.0, 4),       # one block, 65 tokens
    ((1, 1, 4096, 128), 0.1, 7),     # long lists
])
def test_kv128_fwd_bwd_random_masks(shape, density, seed):
    q, k, v, do = _rand(*shape, seed=seed)
    n = shape[2]
    mq, mk = O.num_blocks(n, 128), O.num_blocks(n, BK)
    rng = np.random.default_rng(seed)
    mask = rng.random((shape[0], shape[1], mq, mk)) < density
    mask[..., rng.integers(0, mk)] = True
    ridx, rcnt = mask_to_csr_tensors(mask, DEV)
    cidx, ccnt = mask_to_csc_tensors(mask, DEV)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    o, lse = B.sparge_attn_fwd(qd, kd, vd, ridx, rcnt, check_status=True, block_kv=BK)
    grads = B.sparge_attn_bwd(qd, kd, vd, o, lse, dod, ridx, rcnt, cidx, ccnt, check_status=True,
                              block_kv=BK)
    torch.cuda.synchronize()
    o_ref, lse_ref = O.sparse_attention_dense(to_np(q), to_np(k), to_np(v), mask, 128, BK)
    og = to_np(o)
    assert np.abs(og - o_ref).max() <= O_MAX_ABS and rel_l2(og, o_ref) <= O_REL_L2
    fin = np.isfinite(lse_ref)
    np.testing.assert_allclose(to_np(lse)[fin], lse_ref[fin], atol=LSE_ATOL, rtol=0)
    refs = O.sparse_attention_dense_bwd(to_np(q), to_np(k), to_np(v), to_np(do), mask, 128, BK)
    for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
        assert rel_l2(to_np(g), r) <= GRAD_REL_L2, (shape, name)


def test_kv128_mask_small():
    q, k, _, _ = _rand(1, 3, 3000, 128, seed=9)
    res = B.sparge_mask(q.to(DEV), k.to(DEV), 0.2, 0.7, want_prob=True, want_logit=True,
                        block_kv=BK)
    torch.cuda.synchronize()
    mk = O.num_blocks(3000, BK)
    _, _, lg, pr = O.pooled_map(to_np(q), to_np(k), 128, BK)
    np.testing.assert_allclose(to_np(res["logit"]), lg, atol=MAP_ATOL, rtol=0)
    np.testing.assert_allclose(to_np(res["prob"]), pr, atol=MAP_ATOL, rtol=0)
    ref = O.hybrid_mask_from_prob(res["prob"].cpu().numpy(), 0.2, 0.7)
    assert (unpack_bitmask(res["bitmask"], mk) == ref).all()
    np.testing.assert_array_equal(res["row_cnt"].cpu().numpy(), ref.sum(-1))
    np.testing.assert_array_equal(res["col_cnt"].cpu().numpy(), ref.sum(-2))


@pytest.mark.parametrize("k_frac,p", [(0.05, 0.0), (0.05, 0.9)])
def test_kv128_wan480(k_frac, p):
    """The 480p shape with 128 x 128 blocks (Mk = 256; k = 5 % keeps 13 blocks
    per row at p = 0), in the launch configuration of ``bench.py --block-kv
    128``: mask bit-exact on the GPU's P, every row of the forward of heads 0
    and 11, and their dQ, dK, dV."""
    q, k, v, do = synth.video_inputs(synth.WORKLOADS["wan480"], device=DEV)
    res = B.sparge_mask(q, k, k_frac, p, want_prob=True, block_kv=BK)
    o, lse = B.sparge_attn_fwd(q, k, v, res["row_idx"], res["row_cnt"], check_status=True,
                               block_kv=BK)
    grads = B.sparge_attn_bwd(q, k, v, o, lse, do, res["row_idx"], res["row_cnt"],
                              res["col_idx"], res["col_cnt"], check_status=True, block_kv=BK)
    torch.cuda.synchronize()
    mk = 256
    ref = O.hybrid_mask_from_prob(res["prob"].cpu().numpy(), k_frac, p)
    assert (unpack_bitmask(res["bitmask"], mk) == ref).all()
    if p == 0.0:
        assert (ref.sum(-1) == 13).all()
    check_fwd_heads(q, k, v, ref, o, lse, (0, 11), bk=BK, tag=f"kv128 k={k_frac} p={p}")
    if p == 0.0:
        check_bwd_heads(q, k, v, do, ref, grads, (0, 11), bk=BK, tag="kv128")
