"""sparge_mask_noalloc: the mask entry point for callers that cannot allocate
device memory (a runtime that owns all device memory through its own pool
allocator, or a latency-critical loop where an allocation may synchronise the
device).  It keeps its scratch in a fixed device array inside the library.

Called here through the C ABI (ctypes) and compared with sparge_mask, the
entry point that takes a caller workspace, on two calls in a row with
different inputs (the second call must not see the first call's scratch).
This file is collected last so a failure here stops a -x run only after every
other test has run.
"""

import ctypes

import numpy as np
import pytest
import torch

from block_sparse_attention_sparge_gb300 import binding as B
from helpers import MAP_ATOL, csr_lists

pytestmark = pytest.mark.gpu
DEV = "cuda"


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _noalloc_mask(q, k, k_frac, p):
    lib = B.load_library()
    Bn, H, N, d = q.shape
    mq, mk = -(-N // 128), -(-N // 64)
    out = B._mask_outputs(Bn, H, mq, mk, q.device, True)
    for t in (out["bitmask"], out["row_idx"], out["row_cnt"], out["col_idx"], out["col_cnt"]):
        t.fill_(-7)  # stale garbage the call must overwrite
    out["prob"] = torch.full((Bn, H, mq, mk), float("nan"), device=q.device)
    out["logit"] = torch.full((Bn, H, mq, mk), float("nan"), device=q.device)
    shp = B.Shape(Bn, H, N, d, 128, 64)
    rc = lib.sparge_mask_noalloc(ctypes.byref(shp), _ptr(q), _ptr(k), float(k_frac), float(p), 0.0,
                                 _ptr(out["bitmask"]), _ptr(out["row_idx"]), _ptr(out["row_cnt"]),
                                 _ptr(out["col_idx"]), _ptr(out["col_cnt"]), _ptr(out["prob"]),
                                 _ptr(out["logit"]), None,
                                 ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == B.SPARGE_OK, B.status_string(rc)
    return out


@pytest.mark.parametrize("shape,k_frac,p", [((1, 12, 32760, 128), 0.05, 0.9),
                                            ((2, 3, 5000, 64), 0.1, 0.5)])
def test_noalloc_mask_matches_workspace_mask_on_two_calls(shape, k_frac, p):
    for call, seed in enumerate((101, 202)):
        g = torch.Generator(device=DEV).manual_seed(seed + sum(shape))
        q = torch.randn(shape, generator=g, device=DEV).to(torch.bfloat16)
        k = torch.randn(shape, generator=g, device=DEV).to(torch.bfloat16)
        ref = B.sparge_mask(q, k, k_frac, p, want_prob=True, want_logit=True)
        got = _noalloc_mask(q, k, k_frac, p)
        torch.cuda.synchronize()
        assert torch.equal(got["bitmask"], ref["bitmask"]), call
        assert torch.equal(got["row_cnt"], ref["row_cnt"]), call
        assert torch.equal(got["col_cnt"], ref["col_cnt"]), call
        assert csr_lists(got["row_idx"], got["row_cnt"]) == csr_lists(ref["row_idx"], ref["row_cnt"])
        assert csr_lists(got["col_idx"], got["col_cnt"]) == csr_lists(ref["col_idx"], ref["col_cnt"])
        np.testing.assert_allclose(got["prob"].cpu().numpy(), ref["prob"].cpu().numpy(),
                                   atol=MAP_ATOL, rtol=0)
        np.testing.assert_allclose(got["logit"].cpu().numpy(), ref["logit"].cpu().numpy(),
                                   atol=MAP_ATOL, rtol=0)


def test_noalloc_rejects_shapes_beyond_its_scratch():
    lib = B.load_library()
    q = torch.zeros(16, dtype=torch.bfloat16, device=DEV)  # never read: rejected first
    shp = B.Shape(1, 40, 75600, 128, 128, 64)  # needs about 148 MB of scratch
    rc = lib.sparge_mask_noalloc(ctypes.byref(shp), _ptr(q), _ptr(q), 0.05, 0.9, 0.0, _ptr(q),
                                 _ptr(q), _ptr(q), None, None, None, None, None, None)
    assert rc == B.SPARGE_ERR_WORKSPACE
