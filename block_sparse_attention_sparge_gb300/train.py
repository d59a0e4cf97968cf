"""Trainable block-sparse attention on the library's kernels, and one
velocity-distillation training step at the level of an attention block.

Method: the page "SpargeAttention2: Trainable Sparse Attention via Hybrid
Top-k+Top-p Masking and Distillation Fine-Tuning", section "Abstract" (the
sparse attention is trainable and fine-tuned with a distillation objective),
and the mindverse page "Optimierung der Effizienz von Video-Diffusionsmodellen
durch SpargeAttention2", sections "Velocity Distillation Loss" (a frozen model
with full attention is the teacher, the sparse model the student, and the
student is fitted to the teacher's outputs instead of to the data) and
"Effiziente Kernel-Implementierung und Modellanpassung" (every attention layer
is replaced by the sparse one, then fine-tuned with that loss).

No diffusion model, weights or data exist here, so this module holds the
mechanics only: ``SparseAttentionFunction`` is a torch.autograd.Function whose
forward and backward are ``sparge_attn_fwd`` / ``sparge_attn_bwd``; the mask is
built from Q and K by ``sparge_mask`` and held constant (the selection is
piecewise constant, so no gradient flows through it). ``AttentionBlock`` is a
multi-head attention block (Q/K/V and output projections) whose attention is
either that sparse function or the same kernels with every block kept (dense).
``distillation_step`` runs one optimiser step of a student block against a
frozen dense teacher on the same input, with the mean squared error of the two
outputs as the loss. Projections run in torch (cuBLAS); every attention step
runs in the library's kernels. There is no CPU path: the binding raises when
the library or a GPU is missing.
"""

from __future__ import annotations

import torch

from . import binding as B


class SparseAttentionFunction(torch.autograd.Function):
    """O = block-sparse attention(Q, K, V) under a fixed block mask.

    Inputs are bf16 [B, H, N, d] CUDA tensors; the mask is given as the CSR
    and CSC lists ``sparge_mask`` returns. Gradients flow to Q, K and V."""

    @staticmethod
    def forward(ctx, q, k, v, row_idx, row_cnt, col_idx, col_cnt, softmax_scale):
        q, k, v = (t.contiguous() for t in (q, k, v))
        o, lse = B.sparge_attn_fwd(q, k, v, row_idx, row_cnt, softmax_scale)
        ctx.save_for_backward(q, k, v, o, lse, row_idx, row_cnt, col_idx, col_cnt)
        ctx.softmax_scale = softmax_scale
        return o

    @staticmethod
    def backward(ctx, dout):
        q, k, v, o, lse, row_idx, row_cnt, col_idx, col_cnt = ctx.saved_tensors
        dout = dout.to(torch.bfloat16).contiguous()
        dq, dk, dv = B.sparge_attn_bwd(q, k, v, o, lse, dout, row_idx, row_cnt, col_idx,
                                       col_cnt, ctx.softmax_scale)
        return dq, dk, dv, None, None, None, None, None


def sparse_attention(q, k, v, k_frac: float, p: float, softmax_scale: float = 0.0):
    """Hybrid-masked attention with autograd: the mask (Top-k fraction
    ``k_frac``, Top-p ``p``) is computed from the current Q and K, then held
    constant for the forward and backward of this call. ``k_frac = 1`` keeps
    every block (dense attention)."""
    with torch.no_grad():
        m = B.sparge_mask(q.detach().contiguous(), k.detach().contiguous(), k_frac, p,
                          softmax_scale, want_csc=True)
    return SparseAttentionFunction.apply(q, k, v, m["row_idx"], m["row_cnt"], m["col_idx"],
                                         m["col_cnt"], softmax_scale)


class AttentionBlock(torch.nn.Module):
    """Multi-head attention block on tokens x [B, N, C]: Q, K, V projections
    to H heads of width d, attention, output projection back to C. Weights are
    fp32; the attention runs in bf16 through the library.

    ``k_frac`` and ``p`` select the hybrid mask; ``k_frac = 1`` gives dense
    attention (every block kept)."""

    def __init__(self, channels: int, heads: int, head_dim: int, k_frac: float = 1.0,
                 p: float = 0.0, generator: torch.Generator | None = None, device="cuda"):
        super().__init__()
        self.heads, self.head_dim = heads, head_dim
        self.k_frac, self.p = k_frac, p
        inner = heads * head_dim
        std = channels ** -0.5

        def weight(rows, cols):
            w = torch.randn((rows, cols), generator=generator) * std
            return torch.nn.Parameter(w.to(device))

        self.wq = weight(channels, inner)
        self.wk = weight(channels, inner)
        self.wv = weight(channels, inner)
        self.wo = torch.nn.Parameter((torch.randn((inner, channels), generator=generator)
                                      * inner ** -0.5).to(device))

    def _heads(self, t, b, n):
        return (t.reshape(b, n, self.heads, self.head_dim).permute(0, 2, 1, 3)
                .to(torch.bfloat16).contiguous())

    def forward(self, x):
        b, n, _ = x.shape
        q = self._heads(x @ self.wq, b, n)
        k = self._heads(x @ self.wk, b, n)
        v = self._heads(x @ self.wv, b, n)
        o = sparse_attention(q, k, v, self.k_frac, self.p)
        o = o.float().permute(0, 2, 1, 3).reshape(b, n, self.heads * self.head_dim)
        return o @ self.wo


def distillation_step(student: AttentionBlock, teacher: AttentionBlock, x: torch.Tensor,
                      optimizer: torch.optim.Optimizer) -> float:
    """One fine-tuning step of the sparse student against the frozen dense
    teacher: loss = mean((student(x) - teacher(x))^2); backward through the
    library's sparse attention backward; optimiser step. Returns the loss."""
    with torch.no_grad():
        target = teacher(x)
    optimizer.zero_grad(set_to_none=True)
    loss = torch.mean((student(x) - target) ** 2)
    loss.backward()
    optimizer.step()
    return float(loss.item())
