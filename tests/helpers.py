"""Small helpers shared by the GPU parity tests (no method arithmetic here)."""

import numpy as np
import torch

# Tolerances of the GPU <-> oracle contract.
POOL_ATOL = 1e-5          # fp32 means of bf16 values
MAP_ATOL = 1e-3           # pooled logits and probabilities (fp32)
O_MAX_ABS = 2e-2          # attention output, bf16
O_REL_L2 = 1e-2
LSE_ATOL = 2e-3           # fp32 log-sum-exp
GRAD_REL_L2 = 5e-2        # dQ, dK, dV (bf16)


def to_np(t: torch.Tensor, dtype=np.float64) -> np.ndarray:
    return t.detach().float().cpu().numpy().astype(dtype)


def unpack_bitmask(bm: torch.Tensor, mk: int) -> np.ndarray:
    """[..., words] int32 (uint32 bits) -> [..., mk] bool; block j = bit j%32 of word j//32."""
    w = bm.cpu().numpy().astype(np.uint32)
    bits = ((w[..., :, None] >> np.arange(32, dtype=np.uint32)) & 1).astype(bool)
    return bits.reshape(w.shape[:-1] + (w.shape[-1] * 32,))[..., :mk]


def csr_lists(idx: torch.Tensor, cnt: torch.Tensor):
    """Python lists of the valid CSR entries per row (flattened rows)."""
    i = idx.cpu().numpy().reshape(-1, idx.shape[-1])
    c = cnt.cpu().numpy().reshape(-1)
    return [i[r, : c[r]].tolist() for r in range(c.size)]


def mask_to_csr_tensors(mask: np.ndarray, device):
    """bool [B,H,Mq,Mk] -> (row_idx int32, row_cnt int32) on device, ascending lists."""
    b, h, mq, mk = mask.shape
    idx = np.zeros((b, h, mq, mk), dtype=np.int32)
    cnt = mask.sum(-1).astype(np.int32)
    flat = mask.reshape(-1, mk)
    fi = idx.reshape(-1, mk)
    for r in range(flat.shape[0]):
        nz = np.nonzero(flat[r])[0]
        fi[r, : nz.size] = nz
    return torch.from_numpy(idx).to(device), torch.from_numpy(cnt).to(device)


def mask_to_csc_tensors(mask: np.ndarray, device):
    return mask_to_csr_tensors(np.ascontiguousarray(np.swapaxes(mask, -1, -2)), device)


def rel_l2(a: np.ndarray, b: np.ndarray) -> float:
    return float(np.linalg.norm((a - b).ravel()) / max(np.linalg.norm(b.ravel()), 1e-30))


def check_fwd_heads(q, k, v, mask, o, lse, heads, bq=128, bk=64, tag=""):
    """Every row of the listed heads (b = 0) against the fp32 block-gather
    oracle, element by element: O within the max-abs and relative-L2 bounds,
    LSE within LSE_ATOL (both -inf exactly where a q-block keeps nothing)."""
    import oracle as O
    for h in heads:
        sl = slice(h, h + 1)
        o_ref, lse_ref = O.sparse_attention_blocks(
            to_np(q[:, sl], np.float32), to_np(k[:, sl], np.float32),
            to_np(v[:, sl], np.float32), mask[:, sl], bq, bk, dtype=np.float32)
        o_g = to_np(o[:, sl])
        err = float(np.abs(o_g - o_ref).max())
        rl = rel_l2(o_g, o_ref)
        assert err <= O_MAX_ABS and rl <= O_REL_L2, (tag, h, err, rl)
        lg = to_np(lse[:, sl])
        fin = np.isfinite(lse_ref)
        np.testing.assert_array_equal(np.isneginf(lg), ~fin)
        np.testing.assert_allclose(lg[fin], lse_ref[fin], atol=LSE_ATOL, rtol=0)


def check_bwd_heads(q, k, v, do, mask, grads, heads, bq=128, bk=64, tag=""):
    """dQ, dK, dV of the listed heads (b = 0) within GRAD_REL_L2 of the fp32
    block-gather oracle."""
    import oracle as O
    for h in heads:
        sl = slice(h, h + 1)
        refs = O.sparse_attention_blocks_bwd(
            to_np(q[:, sl], np.float32), to_np(k[:, sl], np.float32),
            to_np(v[:, sl], np.float32), to_np(do[:, sl], np.float32), mask[:, sl], bq, bk,
            dtype=np.float32)
        for name, g, r in zip(("dq", "dk", "dv"), grads, refs):
            gn = to_np(g[:, sl])
            assert np.isfinite(gn).all(), (tag, h, name)
            rl = rel_l2(gn, r)
            assert rl <= GRAD_REL_L2, (tag, h, name, rl)
