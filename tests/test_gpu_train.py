"""The trainable path: autograd through the library's sparse attention, and the
velocity-distillation step (a sparse student block fitted to a frozen dense
teacher block).  Gradients are compared with the fp64 oracle; the distillation
loop must reduce the loss."""

import numpy as np
import pytest
import torch

import oracle as O
from block_sparse_attention_sparge_gb300 import binding as B
from block_sparse_attention_sparge_gb300 import train
from helpers import GRAD_REL_L2, O_MAX_ABS, rel_l2, to_np, unpack_bitmask

pytestmark = pytest.mark.gpu
DEV = "cuda"


def test_autograd_gradients_match_oracle():
    g = torch.Generator().manual_seed(31)
    q, k, v, w = (torch.randn((1, 2, 1000, 64), generator=g).to(torch.bfloat16) for _ in range(4))
    qd, kd, vd = (t.to(DEV).requires_grad_(True) for t in (q, k, v))
    o = train.sparse_attention(qd, kd, vd, 0.3, 0.5)
    (o.float() * w.to(DEV).float()).sum().backward()
    torch.cuda.synchronize()
    m = B.sparge_mask(q.to(DEV), k.to(DEV), 0.3, 0.5)
    mask = unpack_bitmask(m["bitmask"], O.num_blocks(1000, 64))
    o_ref, _ = O.sparse_attention_dense(to_np(q), to_np(k), to_np(v), mask, 128, 64)
    assert np.abs(to_np(o) - o_ref).max() <= O_MAX_ABS
    refs = O.sparse_attention_dense_bwd(to_np(q), to_np(k), to_np(v), to_np(w), mask, 128, 64)
    for name, gr, rf in zip(("dq", "dk", "dv"), (qd.grad, kd.grad, vd.grad), refs):
        assert rel_l2(to_np(gr), rf) <= GRAD_REL_L2, name


def test_dense_setting_matches_sdpa():
    """k_frac = 1 keeps every block: the teacher's attention is dense attention."""
    g = torch.Generator().manual_seed(32)
    q, k, v = (torch.randn((1, 2, 777, 64), generator=g).to(torch.bfloat16) for _ in range(3))
    o = train.sparse_attention(q.to(DEV), k.to(DEV), v.to(DEV), 1.0, 0.0)
    ref = torch.nn.functional.scaled_dot_product_attention(q.double(), k.double(), v.double())
    assert (o.double().cpu() - ref).abs().max().item() <= O_MAX_ABS


def test_distillation_reduces_loss():
    """A student with perturbed projections and a 10 % Top-k / p = 0.5 mask
    is fitted to a frozen dense teacher on a fixed batch of tokens."""
    torch.manual_seed(0)
    C, H, d, N = 128, 2, 64, 2048
    teacher = train.AttentionBlock(C, H, d, k_frac=1.0, p=0.0,
                                   generator=torch.Generator().manual_seed(1))
    student = train.AttentionBlock(C, H, d, k_frac=0.10, p=0.5,
                                   generator=torch.Generator().manual_seed(1))
    with torch.no_grad():
        gp = torch.Generator().manual_seed(2)
        for ps in student.parameters():
            ps.add_(0.5 * ps.std() * torch.randn(ps.shape, generator=gp).to(DEV))
    for pt in teacher.parameters():
        pt.requires_grad_(False)
    x = torch.randn((1, N, C), generator=torch.Generator().manual_seed(3)).to(DEV)
    opt = torch.optim.Adam(student.parameters(), lr=3e-3)
    losses = [train.distillation_step(student, teacher, x, opt) for _ in range(60)]
    assert np.isfinite(losses).all()
    assert losses[-1] < 0.5 * losses[0], (losses[0], losses[-1])
