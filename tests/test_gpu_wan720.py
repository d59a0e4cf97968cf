"""Full Wan2.1-14B 720p shape (B=1, H=40, N=75600 = 21x45x80, d=128, blocks
128x64: Mq = 591, Mk = 1182) in the launch configuration the benchmark uses.
Pooled logits and probabilities of two heads within 1e-3 of the fp64 oracle;
the mask bit-exact on the GPU's P for every row of every head (bitmask, row
counts and ascending row lists); forward rows sampled on two heads, computed
one by one by the oracle."""

import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_attention_sparge_gb300 import binding as B
from block_sparse_attention_sparge_gb300 import synth
from helpers import LSE_ATOL, MAP_ATOL, O_MAX_ABS, O_REL_L2, rel_l2, to_np, unpack_bitmask

pytestmark = pytest.mark.gpu
DEV = "cuda"
MQ, MK = 591, 1182
HEADS = (0, 39)


@pytest.fixture(scope="module")
def wan720():
    q, k, v, do = synth.video_inputs(synth.WORKLOADS["wan720"], device=DEV)
    del do
    torch.cuda.empty_cache()
    return q, k, v


def _check_rows_exact(res, ref):
    """Row counts and ascending row lists equal the oracle's, vectorised."""
    cnt = res["row_cnt"].cpu().numpy().reshape(-1)
    np.testing.assert_array_equal(cnt, ref.reshape(-1, MK).sum(-1))
    got = res["row_idx"].cpu().numpy().reshape(-1, MK)
    exp = np.sort(np.where(ref.reshape(-1, MK), np.arange(MK), MK), axis=-1)
    valid = np.arange(MK)[None, :] < cnt[:, None]
    np.testing.assert_array_equal(np.where(valid, got, -1), np.where(valid, exp, -1))


@pytest.mark.parametrize("k_frac,p", [(0.05, 0.9), (0.05, 0.0)])
def test_wan720_mask_and_fwd(wan720, k_frac, p):
    q, k, v = wan720
    res = B.sparge_mask(q, k, k_frac, p, want_prob=True, want_logit=True)
    o, lse = B.sparge_attn_fwd(q, k, v, res["row_idx"], res["row_cnt"], check_status=True)
    torch.cuda.synchronize()
    for h in HEADS:
        _, _, lg, pr = O.pooled_map(to_np(q[:, h:h + 1]), to_np(k[:, h:h + 1]), 128, 64)
        np.testing.assert_allclose(to_np(res["logit"][:, h:h + 1]), lg, atol=MAP_ATOL, rtol=0)
        np.testing.assert_allclose(to_np(res["prob"][:, h:h + 1]), pr, atol=MAP_ATOL, rtol=0)
    ref = O.hybrid_mask_from_prob(res["prob"].cpu().numpy(), k_frac, p)
    got = unpack_bitmask(res["bitmask"], MK)
    bad = np.argwhere(got != ref)
    assert bad.size == 0, f"{len(bad)} mask bits differ, first at {bad[:3].tolist()}"
    np.testing.assert_array_equal(res["bitmask"].cpu().numpy().astype(np.uint32),
                                  O.pack_bitmask(ref))
    _check_rows_exact(res, ref)
    cnt = ref.sum(-1)
    if p == 0.0:
        assert (cnt == 60).all()  # K = ceil(0.05 * 1182) = 60: 94.92% sparsity
    print(f"720p k={k_frac} p={p}: sparsity {1 - cnt.mean() / MK:.4f}")
    rows = np.r_[0:4, 127:129, 37800:37804, 75520:75600:13, 75599]
    for h in HEADS:
        o_ref, lse_ref = O.sparse_attention_rows(to_np(q[:, h:h + 1]), to_np(k[:, h:h + 1]),
                                                 to_np(v[:, h:h + 1]), ref[:, h:h + 1], 128, 64,
                                                 0, 0, rows)
        o_g = to_np(o[0, h, rows])
        err = np.abs(o_g - o_ref).max()
        assert err <= O_MAX_ABS and rel_l2(o_g, o_ref) <= O_REL_L2, (h, err)
        np.testing.assert_allclose(to_np(lse[0, h, rows]), lse_ref, atol=LSE_ATOL, rtol=0)
