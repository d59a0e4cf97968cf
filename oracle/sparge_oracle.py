"""Plain, slow, obviously-correct CPU restatement of the SpargeAttention2 hot path.

TEST INFRASTRUCTURE ONLY (see ``oracle/__init__.py``): tests, the smoke check
and the benchmark's CPU-baseline leg call it; the CUDA path never does.

Citations use these page tags:

* [P2]  "SpargeAttention2: Trainable Sparse Attention via Hybrid Top-k+Top-p
  Masking and Distillation Fine-Tuning" (chatpaper.ai), section "Abstract".
* [P4]  "Optimierung der Effizienz von Video-Diffusionsmodellen durch
  SpargeAttention2" (mindverse); the section name follows the tag.

The pages give the method in prose only.  Where they are silent this module
takes the plainest reading and says so in the docstring ("Reading: ...").

Shapes: Q, K, V, dO are [B, H, N, d]; blocks are ``bq`` query tokens by ``bk``
key tokens; Mq = ceil(N / bq), Mk = ceil(N / bk).  A partial last block holds
the remaining valid tokens only.

Arithmetic is fp64 unless a caller passes ``dtype=np.float32`` to the
block-gather routines used for full-size shapes.
"""

from __future__ import annotations

import math

import numpy as np

__all__ = [
    "num_blocks",
    "pool_blocks",
    "pooled_logits",
    "row_softmax",
    "pooled_map",
    "topk_count",
    "selection_order",
    "topp_count",
    "topp_count_real",
    "topk_set",
    "topp_set",
    "hybrid_row",
    "hybrid_mask_from_prob",
    "hybrid_mask",
    "pack_bitmask",
    "mask_to_csr",
    "mask_to_csc",
    "expand_block_mask",
    "sparse_attention_dense",
    "sparse_attention_dense_bwd",
    "sparse_attention_blocks",
    "sparse_attention_blocks_bwd",
    "sparse_attention_rows",
]

FIXED_POINT_BITS = 40  # Top-p fixed-point scale 2**40 (see ``topp_count``)


def num_blocks(n: int, block: int) -> int:
    """Number of blocks of ``block`` tokens covering ``n`` tokens (last may be partial)."""
    return (n + block - 1) // block


# ---------------------------------------------------------------------------
# Step 1: block pooling.  [P4 "Maskierungsstrategien: Top-k und Top-p"]: the
# full attention map is too expensive, so a block-pooled map stands in for it.
# Reading: the pooling operator is the arithmetic mean of the block's valid
# tokens (the pages name no operator; the mean is the plainest pooling).
# ---------------------------------------------------------------------------
def pool_blocks(x: np.ndarray, block: int) -> np.ndarray:
    """Mean of each run of ``block`` consecutive tokens along axis -2.

    x: [..., N, d] -> [..., ceil(N/block), d].  The last block averages only
    the tokens it actually holds (N - (M-1)*block of them).
    """
    x = np.asarray(x, dtype=np.float64)
    n = x.shape[-2]
    m = num_blocks(n, block)
    out = np.empty(x.shape[:-2] + (m, x.shape[-1]), dtype=np.float64)
    for i in range(m):
        lo, hi = i * block, min(n, (i + 1) * block)
        out[..., i, :] = x[..., lo:hi, :].sum(axis=-2) / float(hi - lo)
    return out


# ---------------------------------------------------------------------------
# Step 2: pooled attention map.  [P4 "Maskierungsstrategien: Top-k und Top-p"]
# applies Top-p to "cumulative probabilities" of a row of the pooled map, so
# each row is a probability distribution.  Reading: the pooled map is a
# miniature attention map, scaled like the real one (s = 1/sqrt(d) unless the
# caller overrides it) and softmax-normalised per row.
# ---------------------------------------------------------------------------
def pooled_logits(qbar: np.ndarray, kbar: np.ndarray, scale: float) -> np.ndarray:
    """L[..., i, j] = scale * <qbar_i, kbar_j>."""
    qbar = np.asarray(qbar, dtype=np.float64)
    kbar = np.asarray(kbar, dtype=np.float64)
    return float(scale) * np.einsum("...id,...jd->...ij", qbar, kbar)


def row_softmax(logits: np.ndarray) -> np.ndarray:
    """Softmax over the last axis, with the row maximum subtracted first."""
    logits = np.asarray(logits, dtype=np.float64)
    z = logits - logits.max(axis=-1, keepdims=True)
    e = np.exp(z)
    return e / e.sum(axis=-1, keepdims=True)


def pooled_map(q, k, bq: int, bk: int, scale: float | None = None):
    """Pool Q and K, then return (qbar, kbar, logits, prob)."""
    d = q.shape[-1]
    s = (1.0 / math.sqrt(d)) if (scale is None or scale == 0) else float(scale)
    qbar = pool_blocks(q, bq)
    kbar = pool_blocks(k, bk)
    logits = pooled_logits(qbar, kbar, s)
    return qbar, kbar, logits, row_softmax(logits)


# ---------------------------------------------------------------------------
# Steps 3-6: per-row selection.
# ---------------------------------------------------------------------------
def topk_count(k_frac: float, mk: int) -> int:
    """Number of blocks Top-k keeps in a row of ``mk`` blocks.

    [P4 "Maskierungsstrategien: Top-k und Top-p"]: Top-k keeps the k% largest
    positions of each row.  Reading: the count is ceil(k * Mk), with a 1e-4
    guard so that an fp32 k slightly above a round fraction (0.1f) does not
    add a block, clamped to [1, Mk] so every softmax row stays non-empty.
    ``k_frac`` is taken as an fp32 value (the library's argument type)
    widened to fp64.
    """
    k = float(np.float32(k_frac))
    if k >= 1.0:
        return mk
    c = math.ceil(k * mk - 1e-4)
    return max(1, min(mk, c))


def selection_order(prob_row: np.ndarray) -> np.ndarray:
    """Block indices ordered by probability descending, ties by lower index first.

    Reading: the pages give no tie-break; lower block index first.
    """
    prob_row = np.asarray(prob_row, dtype=np.float64)
    idx = np.arange(prob_row.shape[0])
    return np.lexsort((idx, -prob_row))  # primary key last: -P ascending, then idx


def topp_count(prob_row: np.ndarray, p: float) -> int:
    """Length of the Top-p prefix of the selection order.

    [P4 "Maskierungsstrategien: Top-k und Top-p"]: Top-p keeps the smallest
    set of positions whose cumulative probability reaches p.  The smallest
    such set is a prefix of the descending order.

    Reading ("reach" and the arithmetic are unstated): "reach" is ">=", and
    the cumulative sum is exact integer arithmetic on fixed-point weights so
    that the result does not depend on summation order:
      u_j = floor(P_j * 2**40)          (exact: P is fp32, scaling is exact)
      U   = sum_j u_j                   (exact integer)
      T   = fl64(p * U)                 (one round-to-nearest fp64 multiply)
      m_p = smallest m >= 0 with fl64(u_(1) + ... + u_(m)) >= T
    p <= 0 gives m_p = 0 (Top-p off); p >= 1 gives m_p = Mk (keep every
    block, even those whose probability underflowed to zero).
    ``p`` is an fp32 value widened to fp64, like ``k_frac``.
    """
    prob_row = np.asarray(prob_row, dtype=np.float32)  # the selection sees fp32 P
    mk = prob_row.shape[0]
    pf = float(np.float32(p))
    if pf >= 1.0:
        return mk
    if pf <= 0.0:
        return 0
    order = selection_order(prob_row)
    u = np.floor(prob_row.astype(np.float64) * float(2**FIXED_POINT_BITS)).astype(np.uint64)
    total = int(sum(int(v) for v in u))
    thresh = pf * float(total)
    partial = np.cumsum(u[order], dtype=np.uint64)  # exact: sum < 2**53
    reached = partial.astype(np.float64) >= thresh
    # m counts blocks; the empty prefix (m = 0) reaches T only when T == 0.
    if thresh <= 0.0:
        return 0
    if not reached.any():  # cannot happen for p < 1 (T <= U); kept for safety
        return mk
    return int(np.argmax(reached)) + 1


def topp_count_real(prob_row: np.ndarray, p: float) -> int:
    """Real-valued fp64 Top-p prefix length (diagnostic; may differ from the
    fixed-point rule only when a partial sum lies within Mk * 2**-40 of p)."""
    prob_row = np.asarray(prob_row, dtype=np.float32).astype(np.float64)
    mk = prob_row.shape[0]
    pf = float(np.float32(p))
    if pf >= 1.0:
        return mk
    if pf <= 0.0:
        return 0
    order = selection_order(prob_row)
    cs = np.cumsum(prob_row[order] / prob_row.sum())
    hit = np.nonzero(cs >= pf)[0]
    return int(hit[0]) + 1 if hit.size else mk


def topk_set(prob_row: np.ndarray, k_frac: float) -> set:
    """Block indices Top-k keeps in one row."""
    order = selection_order(np.asarray(prob_row, dtype=np.float32))
    return set(int(j) for j in order[: topk_count(k_frac, len(order))])


def topp_set(prob_row: np.ndarray, p: float) -> set:
    """Block indices Top-p keeps in one row."""
    order = selection_order(np.asarray(prob_row, dtype=np.float32))
    return set(int(j) for j in order[: topp_count(prob_row, p)])


def hybrid_row(prob_row: np.ndarray, k_frac: float, p: float) -> np.ndarray:
    """Boolean keep-vector of one row under the hybrid rule.

    [P4 "Hybride Top-k+Top-p Maskierung"], [P2 "Abstract"]: the hybrid rule
    combines Top-k and Top-p so that each covers the other's failure (Top-p
    adds blocks on near-uniform rows, Top-k adds blocks on sink-dominated
    rows).  Reading: the combination is the set union; only a union lets
    either rule add blocks the other missed.
    """
    prob_row = np.asarray(prob_row, dtype=np.float32)
    keep_set = topk_set(prob_row, k_frac) | topp_set(prob_row, p)
    keep = np.zeros(prob_row.shape[0], dtype=bool)
    keep[sorted(keep_set)] = True
    return keep


def hybrid_mask_from_prob(prob: np.ndarray, k_frac: float, p: float) -> np.ndarray:
    """Hybrid block mask [..., Mq, Mk] (bool) from a pooled probability map."""
    prob = np.asarray(prob, dtype=np.float32)
    flat = prob.reshape(-1, prob.shape[-1])
    out = np.zeros(flat.shape, dtype=bool)
    for r in range(flat.shape[0]):
        out[r] = hybrid_row(flat[r], k_frac, p)
    return out.reshape(prob.shape)


def hybrid_mask(q, k, bq: int, bk: int, k_frac: float, p: float, scale=None):
    """End-to-end mask: pool, pooled softmax map (rounded to fp32), hybrid select.

    The probabilities are rounded to fp32 before selection, matching the
    library's fp32 pooled map, which is the object the selection is defined on.
    Returns (mask, prob_fp64).
    """
    _, _, _, prob = pooled_map(q, k, bq, bk, scale)
    return hybrid_mask_from_prob(prob.astype(np.float32), k_frac, p), prob


# ---------------------------------------------------------------------------
# Mask encodings (library output formats).
# ---------------------------------------------------------------------------
def pack_bitmask(mask: np.ndarray) -> np.ndarray:
    """Pack [..., Mq, Mk] bool into [..., Mq, ceil(Mk/32)] uint32; block j is
    bit (j % 32) of word j // 32."""
    mask = np.asarray(mask, dtype=bool)
    mk = mask.shape[-1]
    words = (mk + 31) // 32
    out = np.zeros(mask.shape[:-1] + (words,), dtype=np.uint64)
    for j in range(mk):
        out[..., j // 32] |= mask[..., j].astype(np.uint64) << np.uint64(j % 32)
    return out.astype(np.uint32)


def mask_to_csr(mask: np.ndarray):
    """Kept kv-block indices per q-block row, ascending: (idx [..., Mq, Mk] int32
    padded with -1, cnt [..., Mq] int32)."""
    mask = np.asarray(mask, dtype=bool)
    flat = mask.reshape(-1, mask.shape[-1])
    idx = np.full(flat.shape, -1, dtype=np.int32)
    cnt = np.zeros(flat.shape[0], dtype=np.int32)
    for r in range(flat.shape[0]):
        nz = np.nonzero(flat[r])[0]
        idx[r, : nz.size] = nz
        cnt[r] = nz.size
    return idx.reshape(mask.shape), cnt.reshape(mask.shape[:-1])


def mask_to_csc(mask: np.ndarray):
    """Kept q-block indices per kv-block column, ascending: (idx [..., Mk, Mq],
    cnt [..., Mk])."""
    mask = np.asarray(mask, dtype=bool)
    return mask_to_csr(np.swapaxes(mask, -1, -2))


# ---------------------------------------------------------------------------
# Step 7: block-sparse attention.  [P4 "Grundlagen ..."]: scores, row softmax,
# binary mask keeping only the selected weights.  [P4 "Block-duennbesetzte
# Aufmerksamkeit"]: the mask is constant over each tile.  [P4 "Effiziente
# Kernel-Implementierung ..."]: masked tiles are skipped entirely.
# Reading: a skipped tile contributes nothing and the softmax is normalised
# over the kept keys only (masked scores are -inf).  No causal mask
# (non-autoregressive diffusion, [P4 "Maskierungsstrategien ..."]).
# ---------------------------------------------------------------------------
def _scale(d: int, scale) -> float:
    return (1.0 / math.sqrt(d)) if (scale is None or scale == 0) else float(scale)


def expand_block_mask(block_mask: np.ndarray, n: int, bq: int, bk: int) -> np.ndarray:
    """[..., Mq, Mk] block mask -> [..., N, N] token mask."""
    block_mask = np.asarray(block_mask, dtype=bool)
    qi = np.arange(n) // bq
    kj = np.arange(n) // bk
    return block_mask[..., qi[:, None], kj[None, :]]


def sparse_attention_dense(q, k, v, block_mask, bq: int, bk: int, scale=None):
    """Dense formulation: O = softmax(Q K^T s + M) V with M = 0 / -inf from the
    expanded block mask.  Returns (O, LSE); LSE_t = log sum over allowed keys u
    of exp(s Q_t . K_u).  A row with no allowed key gets O = 0, LSE = -inf."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    n, d = q.shape[-2], q.shape[-1]
    s = _scale(d, scale)
    allowed = expand_block_mask(block_mask, n, bq, bk)
    scores = s * np.einsum("...td,...ud->...tu", q, k)
    scores = np.where(allowed, scores, -np.inf)
    m = scores.max(axis=-1, keepdims=True)
    empty = ~np.isfinite(m)
    m = np.where(empty, 0.0, m)
    e = np.where(allowed, np.exp(scores - m), 0.0)
    l = e.sum(axis=-1, keepdims=True)
    prob = np.where(empty, 0.0, e / np.where(empty, 1.0, l))
    out = np.einsum("...tu,...ud->...td", prob, v)
    with np.errstate(divide="ignore"):
        lse = np.where(empty, -np.inf, m + np.log(np.where(empty, 1.0, l)))[..., 0]
    return out, lse


def sparse_attention_dense_bwd(q, k, v, dout, block_mask, bq: int, bk: int, scale=None):
    """Exact gradients of ``sparse_attention_dense`` w.r.t. Q, K, V for the loss
    <O, dO>, the mask held constant.

    [P2 "Abstract"] and [P4 "Effiziente Kernel-Implementierung ..."]: the
    sparse attention is trainable and has a backward pass.  Reading: the mask
    is piecewise constant in Q and K, so no gradient flows through it.
    Closed form of the masked softmax gradient:
      P = softmax(s Q K^T + M), O = P V
      dV = P^T dO;  dP = dO V^T;  D_t = sum_d dO_td O_td
      dS = P * (dP - D);  dQ = s dS K;  dK = s dS^T Q
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    dout = np.asarray(dout, dtype=np.float64)
    n, d = q.shape[-2], q.shape[-1]
    s = _scale(d, scale)
    allowed = expand_block_mask(block_mask, n, bq, bk)
    scores = np.where(allowed, s * np.einsum("...td,...ud->...tu", q, k), -np.inf)
    m = scores.max(axis=-1, keepdims=True)
    m = np.where(np.isfinite(m), m, 0.0)
    e = np.where(allowed, np.exp(scores - m), 0.0)
    l = e.sum(axis=-1, keepdims=True)
    prob = e / np.where(l > 0, l, 1.0)
    out = np.einsum("...tu,...ud->...td", prob, v)
    dv = np.einsum("...tu,...td->...ud", prob, dout)
    dprob = np.einsum("...td,...ud->...tu", dout, v)
    drow = (dout * out).sum(axis=-1, keepdims=True)
    ds = prob * (dprob - drow)
    dq = s * np.einsum("...tu,...ud->...td", ds, k)
    dk = s * np.einsum("...tu,...td->...ud", ds, q)
    return dq, dk, dv


def _kept_tokens(cols: np.ndarray, n: int, bk: int) -> np.ndarray:
    if cols.size == 0:
        return np.zeros(0, dtype=np.int64)
    return np.concatenate([np.arange(j * bk, min(n, (j + 1) * bk)) for j in cols])


def sparse_attention_blocks(q, k, v, block_mask, bq: int, bk: int, scale=None,
                            dtype=np.float64, heads=None, qblocks=None):
    """Block-gather formulation of ``sparse_attention_dense`` (same definition):
    for each q-block gather the tokens of its kept kv-blocks and run a plain
    softmax attention over them.  Used for shapes too large for the dense
    N x N form.  ``heads`` optionally restricts to a list of (b, h) pairs and
    ``qblocks`` to a list of q-block indices; other rows are left as NaN.
    Returns (O, LSE) in ``dtype``."""
    q = np.asarray(q)
    n, d = q.shape[-2], q.shape[-1]
    b_, h_ = q.shape[0], q.shape[1]
    s = _scale(d, scale)
    mq = num_blocks(n, bq)
    out = np.full(q.shape, np.nan, dtype=dtype)
    lse = np.full(q.shape[:-1], np.nan, dtype=dtype)
    pairs = heads if heads is not None else [(b, h) for b in range(b_) for h in range(h_)]
    for (b, h) in pairs:
        qh = np.asarray(q[b, h], dtype=dtype)
        kh = np.asarray(k[b, h], dtype=dtype)
        vh = np.asarray(v[b, h], dtype=dtype)
        for i in (range(mq) if qblocks is None else qblocks):
            lo, hi = i * bq, min(n, (i + 1) * bq)
            toks = _kept_tokens(np.nonzero(block_mask[b, h, i])[0], n, bk)
            if toks.size == 0:
                out[b, h, lo:hi] = 0
                lse[b, h, lo:hi] = -np.inf
                continue
            sc = (qh[lo:hi] @ kh[toks].T) * dtype(s)
            m = sc.max(axis=-1, keepdims=True)
            e = np.exp(sc - m)
            l = e.sum(axis=-1, keepdims=True)
            out[b, h, lo:hi] = (e / l) @ vh[toks]
            lse[b, h, lo:hi] = (m + np.log(l))[:, 0]
    return out, lse


def sparse_attention_blocks_bwd(q, k, v, dout, block_mask, bq: int, bk: int, scale=None,
                                dtype=np.float64, heads=None, qblocks=None):
    """Block-gather form of ``sparse_attention_dense_bwd`` (same closed form),
    accumulating dK and dV over the q-blocks that keep each kv-block.
    Returns (dQ, dK, dV); heads not listed in ``heads`` are NaN.  With
    ``qblocks`` only those q-blocks contribute (a partial sum, used to time
    a bounded sample of the work)."""
    q = np.asarray(q)
    n, d = q.shape[-2], q.shape[-1]
    b_, h_ = q.shape[0], q.shape[1]
    s = dtype(_scale(d, scale))
    mq = num_blocks(n, bq)
    dq = np.full(q.shape, np.nan, dtype=dtype)
    dk = np.full(q.shape, np.nan, dtype=dtype)
    dv = np.full(q.shape, np.nan, dtype=dtype)
    pairs = heads if heads is not None else [(b, h) for b in range(b_) for h in range(h_)]
    for (b, h) in pairs:
        qh = np.asarray(q[b, h], dtype=dtype)
        kh = np.asarray(k[b, h], dtype=dtype)
        vh = np.asarray(v[b, h], dtype=dtype)
        doh = np.asarray(dout[b, h], dtype=dtype)
        dkh = np.zeros_like(kh)
        dvh = np.zeros_like(vh)
        dqh = np.zeros_like(qh)
        for i in (range(mq) if qblocks is None else qblocks):
            lo, hi = i * bq, min(n, (i + 1) * bq)
            toks = _kept_tokens(np.nonzero(block_mask[b, h, i])[0], n, bk)
            if toks.size == 0:
                continue
            sc = (qh[lo:hi] @ kh[toks].T) * s
            m = sc.max(axis=-1, keepdims=True)
            e = np.exp(sc - m)
            prob = e / e.sum(axis=-1, keepdims=True)
            o = prob @ vh[toks]
            dprob = doh[lo:hi] @ vh[toks].T
            drow = (doh[lo:hi] * o).sum(axis=-1, keepdims=True)
            ds = prob * (dprob - drow)
            dqh[lo:hi] = s * (ds @ kh[toks])
            dkh[toks] += s * (ds.T @ qh[lo:hi])
            dvh[toks] += prob.T @ doh[lo:hi]
        dq[b, h], dk[b, h], dv[b, h] = dqh, dkh, dvh
    return dq, dk, dv


def sparse_attention_rows(q, k, v, block_mask, bq: int, bk: int, b: int, h: int,
                          rows, scale=None, dtype=np.float64):
    """O and LSE of selected query tokens ``rows`` of head (b, h), computed one
    token at a time from the definition (for spot checks at full size)."""
    n, d = q.shape[-2], q.shape[-1]
    s = _scale(d, scale)
    rows = np.asarray(rows, dtype=np.int64)
    out = np.zeros((rows.size, d), dtype=dtype)
    lse = np.zeros(rows.size, dtype=dtype)
    kh = None
    for r, t in enumerate(rows):
        toks = _kept_tokens(np.nonzero(block_mask[b, h, t // bq])[0], n, bk)
        if toks.size == 0:
            lse[r] = -np.inf
            continue
        if kh is None:
            kh = np.asarray(k[b, h], dtype=dtype)
            vh = np.asarray(v[b, h], dtype=dtype)
        sc = (kh[toks] @ np.asarray(q[b, h, t], dtype=dtype)) * dtype(s)
        m = sc.max()
        e = np.exp(sc - m)
        out[r] = (e / e.sum()) @ vh[toks]
        lse[r] = m + np.log(e.sum())
    return out, lse
