"""Bounded device waits: a barrier nothing arrives at must give up, report
SPARGE_ERR_TIMEOUT in the status word and leave the context usable."""

import pytest
import torch

from block_sparse_attention_sparge_gb300 import binding as B

pytestmark = pytest.mark.gpu


def test_wait_probe_times_out_and_reports():
    code = B.sparge_debug_wait_probe(timeout_ns=20_000_000)  # 20 ms
    assert code == B.SPARGE_ERR_TIMEOUT
    # the context still works afterwards
    x = torch.ones(1024, device="cuda")
    assert float(x.sum()) == 1024.0


def test_normal_launch_leaves_status_clear():
    g = torch.Generator().manual_seed(0)
    q, k, v = [torch.randn((1, 1, 300, 64), generator=g).to(torch.bfloat16).cuda() for _ in range(3)]
    res = B.sparge_mask(q, k, 0.5, 0.5)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    B.sparge_attn_fwd(q, k, v, res["row_idx"], res["row_cnt"], status=st)
    assert B._read_status(st) == B.SPARGE_OK
