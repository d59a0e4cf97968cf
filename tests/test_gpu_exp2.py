"""The FMA-pipe 2^x polynomial used for part of the attention exponentials,
checked against CUDA's exp2 (torch.exp2 on the device)."""

import pytest
import torch

from block_sparse_attention_sparge_gb300 import binding as B

pytestmark = pytest.mark.gpu


def test_exp2_poly_relative_error_bound():
    x = torch.linspace(-126.0, 8.0, 2_000_001, device="cuda")
    x = torch.cat([x, torch.tensor([0.0, -1.0, 1.0, -0.5, 7.999, -125.99], device="cuda")])
    y = B.sparge_debug_exp2_poly(x)
    ref = torch.exp2(x.double())
    rel = ((y.double() - ref) / ref).abs().max().item()
    assert rel < 1e-4, rel


def test_exp2_poly_flushes_below_min_normal():
    x = torch.tensor([-126.5, -140.0, -1e30, float("-inf")], device="cuda")
    y = B.sparge_debug_exp2_poly(x)
    assert torch.equal(y, torch.zeros_like(y))
