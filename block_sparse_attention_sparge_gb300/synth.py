"""Seeded synthetic inputs shaped like the video-diffusion attention workloads.

This module holds no arithmetic of the method itself: it only draws Q, K, V
and dO tensors.  Tests and the benchmark feed the same tensors to both the
CUDA library and the CPU oracle.

Workloads (stand-ins for the Wan2.1 video models the method is evaluated on;
no dataset, prompt or weight is used):

* ``tiny``:   B=1, H=2, N=1024, d=64; Q, K, V, dO ~ N(0, 1) drawn in that
  order from one ``torch.Generator`` seeded 0.
* ``wan480``: B=1, H=12, N=32760 = 21 x 30 x 52 latent tokens (t, h, w
  flattened row-major), d=128.
* ``wan720``: B=1, H=40, N=75600 = 21 x 45 x 80, d=128.

The video-shaped Q and K are spatially smooth Gaussian fields: white noise on
the (t, h, w) grid convolved with a separable Gaussian (sigma = 1, 3, 3
tokens, truncated at 3 sigma, zero padding), then each (head, channel)
restandardised to mean 0 and std 1.  Q and K are independent fields, except
in ``wan480_local``, where a latent field shared by Q and K (weight ``rho``,
its own smoothing) is mixed into both and Q is scaled by ``q_gain``.  Four
sink tokens (0..3) get a strong common direction ``u`` (unit
vector, per head) in K, and every query gets a weak component along ``u``:
K_s += 3 sqrt(d) u for s < 4, Q_t += 0.25 sqrt(d) u for all t, a token-level
logit margin of 0.75 sqrt(d).  V and dO are white N(0, 1).
Seeds: Q 1, K 2, V 3, dO 4, sink directions 5, shared latent 7.

Independent smooth fields give near-uniform pooled rows (pooled logit std
about 0.2 at the 480p shape), so Top-p at p = 0.9 keeps most blocks there;
a Top-k-only mask (p = 0) gives the 95% sparsity point.  The shared latent
of ``wan480_local`` makes each pooled row peak around its own neighbourhood,
so there the hybrid rule itself reaches high sparsity.
"""

from __future__ import annotations

import math
from dataclasses import dataclass

import torch

__all__ = [
    "Workload",
    "WORKLOADS",
    "tiny_inputs",
    "video_inputs",
    "uniform_inputs",
    "skewed_inputs",
    "make_inputs",
]


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    grid: tuple  # (t, h, w) latent grid, or (N,) for unstructured inputs
    d: int
    block_q: int = 128
    block_kv: int = 64
    k_frac: float = 0.05
    p: float = 0.9
    rho: float = 0.0              # weight of the latent field shared by Q and K
    shared_sigma: tuple = (1.0, 3.0, 3.0)  # smoothing of that shared field
    q_gain: float = 1.0           # Q is scaled by this before the sinks are added

    @property
    def N(self) -> int:
        return int(math.prod(self.grid))


WORKLOADS = {
    "tiny": Workload("tiny", 1, 2, (1024,), 64, 128, 64, 0.10, 0.9),
    "wan480": Workload("wan480", 1, 12, (21, 30, 52), 128, 128, 64, 0.05, 0.9),
    "wan720": Workload("wan720", 1, 40, (21, 45, 80), 128, 128, 64, 0.05, 0.9),
    # The 480p token grid with head width 64 (24 heads: the same model width):
    # the d = 64 variant of the kernels at full size.
    "wan480_d64": Workload("wan480_d64", 1, 24, (21, 30, 52), 64, 128, 64, 0.05, 0.9),
    # The 480p shape with local attention: Q and K share a smoother latent
    # field (sigma 2, 8, 8 tokens; weight 0.9) and Q carries a gain of 2.5, so
    # each pooled row peaks around its own neighbourhood and the hybrid rule at
    # k = 5 %, p = 0.9 keeps few blocks, with uneven counts per row.
    "wan480_local": Workload("wan480_local", 1, 12, (21, 30, 52), 128, 128, 64, 0.05, 0.9,
                             rho=0.9, shared_sigma=(2.0, 8.0, 8.0), q_gain=2.5),
}

# Generator constants (fixed once; recorded in the design notes).
SIGMA = (1.0, 3.0, 3.0)
SINK_TOKENS = 4
SINK_K_GAIN = 3.0    # K_s += SINK_K_GAIN * sqrt(d) * u for s < SINK_TOKENS
SINK_Q_GAIN = 0.25   # Q_t += SINK_Q_GAIN * sqrt(d) * u for every t


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def _gauss_kernel(sigma: float, device) -> torch.Tensor:
    r = int(math.ceil(3.0 * sigma))
    x = torch.arange(-r, r + 1, dtype=torch.float32, device=device)
    w = torch.exp(-0.5 * (x / sigma) ** 2)
    return w / w.sum()


def _smooth_axis(x: torch.Tensor, axis: int, sigma: float) -> torch.Tensor:
    """Zero-padded 1-D Gaussian convolution of ``x`` along ``axis``."""
    w = _gauss_kernel(sigma, x.device)
    r = (w.numel() - 1) // 2
    xt = x.movedim(axis, -1)
    shp = xt.shape
    y = torch.nn.functional.conv1d(xt.reshape(-1, 1, shp[-1]), w.view(1, 1, -1), padding=r)
    return y.reshape(shp).movedim(-1, axis)


def _smooth_field(H: int, grid, d: int, seed: int, device, sigma=SIGMA) -> torch.Tensor:
    """[H, N, d] fp32 smooth field, each (head, channel) mean 0, std 1."""
    g = _gen(seed, device)
    x = torch.randn((H,) + tuple(grid) + (d,), generator=g, device=device, dtype=torch.float32)
    for ax, s in zip((1, 2, 3), sigma):
        x = _smooth_axis(x, ax, s)
    x = x.reshape(H, -1, d)
    x = x - x.mean(dim=1, keepdim=True)
    x = x / x.std(dim=1, keepdim=True)
    return x


def tiny_inputs(device="cpu", seed: int = 0, H: int = 2, N: int = 1024, d: int = 64, B: int = 1):
    """Q, K, V, dO ~ N(0, 1) bf16 [B, H, N, d], drawn in that order from one generator."""
    g = _gen(seed, device)
    out = [torch.randn((B, H, N, d), generator=g, device=device, dtype=torch.float32)
           .to(torch.bfloat16) for _ in range(4)]
    return tuple(out)


def video_inputs(wl: Workload, device="cpu", heads=None, rho=None):
    """Video-shaped Q, K, V, dO bf16 [B, H, N, d] (B = 1); see the module docstring.

    ``heads`` (optional) limits generation to the first ``heads`` heads: each
    head's tensors depend only on the head index, so a prefix of heads equals
    the same heads of the full tensor.
    """
    H = wl.H if heads is None else int(heads)
    d, N = wl.d, wl.N
    rho = wl.rho if rho is None else float(rho)
    q = _smooth_field(H, wl.grid, d, 1, device)
    k = _smooth_field(H, wl.grid, d, 2, device)
    if rho > 0.0:
        shared = _smooth_field(H, wl.grid, d, 7, device, sigma=wl.shared_sigma)
        a = math.sqrt(max(0.0, 1.0 - rho * rho))
        q = rho * shared + a * q
        k = rho * shared + a * k
    if wl.q_gain != 1.0:
        q = wl.q_gain * q
    gu = _gen(5, device)
    u = torch.randn((H, d), generator=gu, device=device, dtype=torch.float32)
    u = u / u.norm(dim=1, keepdim=True)
    sd = math.sqrt(d)
    q = q + SINK_Q_GAIN * sd * u[:, None, :]
    k[:, :SINK_TOKENS, :] += SINK_K_GAIN * sd * u[:, None, :]
    v = torch.randn((H, N, d), generator=_gen(3, device), device=device, dtype=torch.float32)
    do = torch.randn((H, N, d), generator=_gen(4, device), device=device, dtype=torch.float32)
    return tuple(t.reshape(1, H, N, d).to(torch.bfloat16).contiguous() for t in (q, k, v, do))


def uniform_inputs(wl: Workload, device="cpu", heads=None, std: float = 0.05):
    """Near-uniform pooled rows: Q, K ~ N(0, std^2) i.i.d.; V, dO ~ N(0, 1)."""
    H = wl.H if heads is None else int(heads)
    g = _gen(11, device)
    shp = (1, H, wl.N, wl.d)
    q = std * torch.randn(shp, generator=g, device=device)
    k = std * torch.randn(shp, generator=g, device=device)
    v = torch.randn(shp, generator=g, device=device)
    do = torch.randn(shp, generator=g, device=device)
    return tuple(t.to(torch.bfloat16).contiguous() for t in (q, k, v, do))


def skewed_inputs(wl: Workload, device="cpu", heads=None):
    """Sink-dominated pooled rows: the whole kv-block 0 carries a strong common
    direction (K += 2 sqrt(d) u there, Q += 0.5 sqrt(d) u everywhere)."""
    H = wl.H if heads is None else int(heads)
    g = _gen(21, device)
    shp = (1, H, wl.N, wl.d)
    q = torch.randn(shp, generator=g, device=device)
    k = torch.randn(shp, generator=g, device=device)
    v = torch.randn(shp, generator=g, device=device)
    do = torch.randn(shp, generator=g, device=device)
    u = torch.randn((H, wl.d), generator=g, device=device)
    u = u / u.norm(dim=1, keepdim=True)
    sd = math.sqrt(wl.d)
    q = q + 0.5 * sd * u[None, :, None, :]
    k[:, :, : wl.block_kv, :] += 2.0 * sd * u[None, :, None, :]
    return tuple(t.to(torch.bfloat16).contiguous() for t in (q, k, v, do))


def make_inputs(name: str, device="cpu", heads=None):
    """Inputs of a named workload (``tiny``, ``wan480``, ``wan720``)."""
    wl = WORKLOADS[name]
    if name == "tiny":
        return tiny_inputs(device=device, H=wl.H if heads is None else heads, N=wl.N, d=wl.d)
    return video_inputs(wl, device=device, heads=heads)
