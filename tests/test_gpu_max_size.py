"""The largest supported shape: N = 524288 tokens, i.e. 4096 q-blocks and 8192
64-key kv-blocks per head (the selection's radix path at its widest rows, the
longest row and column lists, the largest TMA coordinates).  One head at
d = 64, k = 0.2 % (17 kv-blocks per row), every step against the oracle: the
pooled map within 1e-3, the mask and its lists bit-exact on the GPU's P, and
the forward and backward of the whole head within the usual bounds."""

import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_attention_sparge_gb300 import binding as B
from helpers import check_bwd_heads, check_fwd_heads, csr_lists, to_np, unpack_bitmask

pytestmark = pytest.mark.gpu
DEV = "cuda"
MAP_ATOL = 1e-3


def test_max_n_one_head():
    n, d, k_frac, p = 524288, 64, 0.002, 0.0
    g = torch.Generator().manual_seed(47)
    q, k, v, do = [torch.randn((1, 1, n, d), generator=g).to(torch.bfloat16) for _ in range(4)]
    mq, mk = O.num_blocks(n, 128), O.num_blocks(n, 64)
    assert (mq, mk) == (4096, 8192)
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    res = B.sparge_mask(qd, kd, k_frac, p, want_prob=True)
    o, lse = B.sparge_attn_fwd(qd, kd, vd, res["row_idx"], res["row_cnt"], check_status=True)
    grads = B.sparge_attn_bwd(qd, kd, vd, o, lse, dod, res["row_idx"], res["row_cnt"],
                              res["col_idx"], res["col_cnt"], check_status=True)
    torch.cuda.synchronize()

    prob = res["prob"].cpu().numpy()
    _, _, _, pr = O.pooled_map(to_np(q), to_np(k), 128, 64)
    np.testing.assert_allclose(prob, pr, atol=MAP_ATOL, rtol=0)
    ref = O.hybrid_mask_from_prob(prob, k_frac, p)
    mask = unpack_bitmask(res["bitmask"], mk)
    assert np.array_equal(mask, ref)
    assert (ref.sum(-1) == 17).all()
    ridx, rcnt = O.mask_to_csr(ref)
    assert csr_lists(res["row_idx"], res["row_cnt"]) == csr_lists(torch.from_numpy(ridx),
                                                                  torch.from_numpy(rcnt))
    cidx, ccnt = O.mask_to_csc(ref)
    assert csr_lists(res["col_idx"], res["col_cnt"]) == csr_lists(torch.from_numpy(cidx),
                                                                  torch.from_numpy(ccnt))
    check_fwd_heads(q, k, v, mask, o, lse, (0,), tag="N = 524288")
    check_bwd_heads(q, k, v, do, mask, grads, (0,), tag="N = 524288")
