"""The d = 64 kernels at full size: the 480p token grid (N = 32760 =
21x30x52) with 24 heads of width 64, blocks 128x64 (Mq = 256, Mk = 512), in the
launch configuration the benchmark uses (``--workload wan480_d64``).  The mask
is bit-exact on the GPU's P for every row; every row of the forward (O and LSE)
of two heads and their dQ, dK, dV are checked against the fp32 oracle."""

import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_attention_sparge_gb300 import binding as B
from block_sparse_attention_sparge_gb300 import synth
from helpers import MAP_ATOL, check_bwd_heads, check_fwd_heads, to_np, unpack_bitmask

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
    check_fwd_heads(q, k, v, ref, o, lse, HEADS, tag=f"d64 k={k_frac} p={p}")
    check_bwd_heads(q, k, v, do, ref, (dq, dk, dv), HEADS, tag=f"d64 k={k_frac} p={p}")
