"""GB300-native (sm_103a) SpargeAttention2 hot path.

Hybrid Top-k + Top-p block-mask construction from a mean-pooled attention map,
followed by block-sparse attention forward and backward that compute only the
kept tiles.  The work runs in the CUDA kernels of ``libsparge.so`` (C ABI in
``include/sparge.h``); ``binding`` marshals torch tensors to it.
"""

from .binding import (  # noqa: F401
    SpargeError,
    load_library,
    sparge_attn_bwd,
    sparge_attn_fwd,
    sparge_debug_wait_probe,
    sparge_mask,
    sparge_mask_from_prob,
    sparge_pool,
)

__all__ = [
    "SpargeError",
    "load_library",
    "sparge_pool",
    "sparge_mask",
    "sparge_mask_from_prob",
    "sparge_attn_fwd",
    "sparge_attn_bwd",
    "sparge_debug_wait_probe",
]
