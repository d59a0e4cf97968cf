"""The d = 64 kernels at full size: the 480p token grid (N = 32760 =
21x30x52) with 24 heads of width 64, blocks 128x64 (Mq = 256, Mk = 512), in the
launch configuration the benchmark uses (``--workload wan480_d64``).  The mask
is bit-exact on the GPU's P for every row, forward rows are sampled on two
heads, and dQ, dK, dV of two heads are checked against the fp32 oracle."""

import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_attention_sparge_gb300 import binding as B
from block_sparse_attention_sparge_gb300 import synth
from helpers import (GRAD_REL_L2, LSE_ATOL, MAP_ATOL, O_MAX_ABS, O_REL_L2, rel_l2, to_np,
                     unpack_bitmask)

pytestmark = pytest.mark.gpu
DEV = "cuda"
MK = 512
HEADS = (0, 23)


@pytest.fixture(scope="module")
def wan480_d64():
    return synth.video_inputs(synth.WORKLOADS["wan480_d64"], device=DEV)


@pytest.mark.parametrize("k_frac,p", [(0.05, 0.0), (0.05, 0.9)])
def test_d64_full_size(wan480_d64, k_frac, p):
    q, k, v, do = wan480_d64
    res = B.sparge_mask(q, k, k_frac, p, want_prob=True)
    o, lse = B.sparge_attn_fwd(q, k, v, res["row_idx"], res["row_cnt"], check_status=True)
    dq, dk, dv = B.sparge_attn_bwd(q, k, v, o, lse, do, res["row_idx"], res["row_cnt"],
                                   res["col_idx"], res["col_cnt"], check_status=True)
    torch.cuda.synchronize()
    _, _, _, pr = O.pooled_map(to_np(q[:, :1]), to_np(k[:, :1]), 128, 64)
    np.testing.assert_allclose(to_np(res["prob"][:, :1]), pr, atol=MAP_ATOL, rtol=0)
    ref = O.hybrid_mask_from_prob(res["prob"].cpu().numpy(), k_frac, p)
    got = unpack_bitmask(res["bitmask"], MK)
    assert (got == ref).all()
    np.testing.assert_array_equal(res["row_cnt"].cpu().numpy(), ref.sum(-1))
    rows = np.r_[0:4, 16380:16384, 32700:32760:11, 32759]
    for h in HEADS:
        sl = slice(h, h + 1)
        o_ref, lse_ref = O.sparse_attention_rows(to_np(q[:, sl]), to_np(k[:, sl]), to_np(v[:, sl]),
                                                 ref[:, sl], 128, 64, 0, 0, rows)
        o_g = to_np(o[0, h, rows])
        err = np.abs(o_g - o_ref).max()
        assert err <= O_MAX_ABS and rel_l2(o_g, o_ref) <= O_REL_L2, (h, err)
        np.testing.assert_allclose(to_np(lse[0, h, rows]), lse_ref, atol=LSE_ATOL, rtol=0)
        refs = O.sparse_attention_blocks_bwd(
            to_np(q[:, sl], np.float32), to_np(k[:, sl], np.float32), to_np(v[:, sl], np.float32),
            to_np(do[:, sl], np.float32), ref[:, sl], 128, 64, dtype=np.float32)
        for name, g, r in zip(("dq", "dk", "dv"), (dq[:, sl], dk[:, sl], dv[:, sl]), refs):
            assert rel_l2(to_np(g), r) <= GRAD_REL_L2, (h, name)
