"""Host-side checks of the C ABI that need no GPU: the library builds and
loads, exports every entry point ``include/sparge.h`` declares, and rejects
invalid arguments before any CUDA call.

Every call below that passes fake pointers is built to FAIL validation, so it
returns before anything reaches the device (safe on a GPU machine too).
"""

import ctypes
import os
import re

import pytest

from block_sparse_attention_sparge_gb300 import _build, binding as B

HEADER = os.path.join(os.path.dirname(os.path.dirname(os.path.abspath(__file__))), "include",
                      "sparge.h")


@pytest.fixture(scope="module")
def lib():
    return B.load_library(build_if_missing=True)


def _declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(sparge_\w+)\s*\(", text)))


def test_library_builds_in_tree_and_loads(lib):
    assert os.path.dirname(_build.LIB_PATH) == os.path.dirname(os.path.abspath(B.__file__))
    assert os.path.exists(_build.LIB_PATH)
    assert lib.sparge_version() >= 100


def test_exports_every_declared_symbol(lib):
    names = _declared_functions()
    assert len(names) >= 10
    for n in names:
        assert hasattr(lib, n), n
    assert set(names) == set(B._SIGNATURES), "binding and header disagree"


def test_status_strings(lib):
    for code in range(0, -7, -1):
        s = lib.sparge_status_string(code).decode()
        assert s.startswith("SPARGE_")
    assert lib.sparge_status_string(-99).decode() == "SPARGE_ERR_UNKNOWN"


def _shape(B_=1, H=2, N=1024, d=128, bq=128, bk=64):
    return B.Shape(B_, H, N, d, bq, bk)


def test_workspace_sizes(lib):
    n = ctypes.c_size_t(0)
    s = _shape(1, 12, 32760, 128)
    assert lib.sparge_mask_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == 0
    mq, mk = 256, 512
    # Q and K means as bf16 pairs (hi, lo) and the fp32 pooled logits, each of
    # the five regions 256-byte aligned.
    expect = 2 * 12 * mq * 128 * 2 + 2 * 12 * mk * 128 * 2 + 12 * mq * mk * 4
    assert expect <= n.value <= expect + 5 * 256
    assert lib.sparge_attn_bwd_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == 0
    # D per token, the q-block order, four counters, five arrays over the dK/dV
    # items (12 heads x 256 key tiles plus 128 parts of cut tiles: tile and
    # part word in launch order, tile, part word and work in tile order), 1024
    # completion counters and 128 fp32 partial slots of 128 keys x (dV | dK),
    # each of the ten regions 256-byte aligned.
    items = 12 * 256 + 128
    expect = (12 * 32760 * 4 + 5 * items * 4 + 12 * 256 * 4 + 4 * 4 + 1024 * 4
              + 128 * 128 * 2 * 128 * 4)
    assert expect <= n.value <= expect + 10 * 256


@pytest.mark.parametrize("shape,code", [
    ((1, 2, 1024, 96, 128, 64), B.SPARGE_ERR_UNSUPPORTED),
    ((1, 2, 1024, 128, 64, 64), B.SPARGE_ERR_UNSUPPORTED),
    ((1, 2, 1024, 128, 128, 256), B.SPARGE_ERR_UNSUPPORTED),
    ((1, 2, 1024, 128, 128, 32), B.SPARGE_ERR_UNSUPPORTED),
    ((1, 2, 600000, 128, 128, 64), B.SPARGE_ERR_UNSUPPORTED),
    ((0, 2, 1024, 128, 128, 64), B.SPARGE_ERR_INVALID_ARG),
    ((1, 2, 0, 128, 128, 64), B.SPARGE_ERR_INVALID_ARG),
    ((1, -1, 16, 64, 128, 64), B.SPARGE_ERR_INVALID_ARG),
])
def test_shape_validation(lib, shape, code):
    s = B.Shape(*shape)
    n = ctypes.c_size_t(0)
    assert lib.sparge_mask_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == code
    assert lib.sparge_attn_bwd_workspace_bytes(ctypes.byref(s), ctypes.byref(n)) == code
    assert lib.sparge_mask_workspace_bytes(None, ctypes.byref(n)) == B.SPARGE_ERR_INVALID_ARG


FAKE = ctypes.c_void_p(0x10000)        # 16-byte aligned, never dereferenced
ODD = ctypes.c_void_p(0x10008)         # 8-byte aligned only


def test_mask_argument_validation(lib):
    s = _shape()
    ok_ws = ctypes.c_size_t(1 << 30)
    call = lambda **kw: lib.sparge_mask(  # noqa: E731
        ctypes.byref(s), kw.get("q", FAKE), kw.get("k", FAKE), kw.get("kf", 0.1), kw.get("p", 0.9),
        kw.get("scale", 0.0), kw.get("bm", FAKE), kw.get("ri", FAKE), kw.get("rc", FAKE),
        kw.get("ci", None), kw.get("cc", None), None, None, kw.get("ws", FAKE),
        kw.get("wsb", ok_ws), None, None)
    assert call(q=None) == B.SPARGE_ERR_INVALID_ARG
    assert call(q=ODD) == B.SPARGE_ERR_MISALIGNED
    assert call(kf=0.0) == B.SPARGE_ERR_INVALID_ARG
    assert call(kf=1.5) == B.SPARGE_ERR_INVALID_ARG
    assert call(kf=float("nan")) == B.SPARGE_ERR_INVALID_ARG
    assert call(p=-0.1) == B.SPARGE_ERR_INVALID_ARG
    assert call(p=1.01) == B.SPARGE_ERR_INVALID_ARG
    assert call(scale=float("inf")) == B.SPARGE_ERR_INVALID_ARG
    assert call(bm=None) == B.SPARGE_ERR_INVALID_ARG
    assert call(ci=FAKE) == B.SPARGE_ERR_INVALID_ARG  # col_idx without col_cnt
    assert call(ws=None) == B.SPARGE_ERR_WORKSPACE
    assert call(wsb=ctypes.c_size_t(16)) == B.SPARGE_ERR_WORKSPACE


def test_fwd_bwd_argument_validation(lib):
    s = _shape()
    assert lib.sparge_attn_fwd(ctypes.byref(s), FAKE, FAKE, None, FAKE, FAKE, 0.0, FAKE, None,
                               None, None) == B.SPARGE_ERR_INVALID_ARG
    assert lib.sparge_attn_fwd(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, ODD, None,
                               None, None) == B.SPARGE_ERR_MISALIGNED
    assert lib.sparge_attn_fwd(ctypes.byref(s), FAKE, FAKE, FAKE, FAKE, FAKE, float("nan"), FAKE,
                               None, None, None) == B.SPARGE_ERR_INVALID_ARG
    bad = B.Shape(1, 2, 1024, 80, 128, 64)
    assert lib.sparge_attn_fwd(ctypes.byref(bad), FAKE, FAKE, FAKE, FAKE, FAKE, 0.0, FAKE, None,
                               None, None) == B.SPARGE_ERR_UNSUPPORTED
    args = [FAKE] * 6 + [FAKE] * 4
    assert lib.sparge_attn_bwd(ctypes.byref(s), *args, 0.0, FAKE, FAKE, FAKE, None,
                               ctypes.c_size_t(1 << 30), None, None) == B.SPARGE_ERR_WORKSPACE
    assert lib.sparge_attn_bwd(ctypes.byref(s), *args, 0.0, FAKE, FAKE, FAKE, FAKE,
                               ctypes.c_size_t(4), None, None) == B.SPARGE_ERR_WORKSPACE
    assert lib.sparge_attn_bwd(ctypes.byref(s), *args, 0.0, None, FAKE, FAKE, FAKE,
                               ctypes.c_size_t(1 << 30), None, None) == B.SPARGE_ERR_INVALID_ARG
    assert lib.sparge_read_status(None, None, None) == B.SPARGE_ERR_INVALID_ARG
    assert lib.sparge_status_copy_async(None, None, None) == B.SPARGE_ERR_INVALID_ARG
    assert lib.sparge_status_copy_async(FAKE, None, None) == B.SPARGE_ERR_INVALID_ARG
    assert lib.sparge_debug_wait_probe(None, 10, None) == B.SPARGE_ERR_INVALID_ARG


def test_noalloc_checks_arguments_before_any_cuda_call(lib):
    """The allocation-free mask entry point validates every argument before it
    touches CUDA (here, with no GPU, any CUDA call would fail differently)."""
    s = _shape()
    args = dict(q=FAKE, k=FAKE, kf=0.1, p=0.9, scale=0.0, bm=FAKE, ri=FAKE, rc=FAKE, ci=None,
                cc=None, pr=None, lg=None, st=None)

    def call(**kw):
        a = dict(args, **kw)
        return lib.sparge_mask_noalloc(ctypes.byref(s), a["q"], a["k"], a["kf"], a["p"],
                                       a["scale"], a["bm"], a["ri"], a["rc"], a["ci"], a["cc"],
                                       a["pr"], a["lg"], a["st"], None)
    assert call(q=None) == B.SPARGE_ERR_INVALID_ARG
    assert call(k=ODD) == B.SPARGE_ERR_MISALIGNED
    assert call(kf=0.0) == B.SPARGE_ERR_INVALID_ARG
    assert call(p=2.0) == B.SPARGE_ERR_INVALID_ARG
    assert call(bm=None) == B.SPARGE_ERR_INVALID_ARG
    assert call(ci=FAKE) == B.SPARGE_ERR_INVALID_ARG
    assert call(scale=float("nan")) == B.SPARGE_ERR_INVALID_ARG
    big = B.Shape(1, 40, 75600, 128, 128, 64)
    assert lib.sparge_mask_noalloc(ctypes.byref(big), FAKE, FAKE, 0.05, 0.9, 0.0, FAKE, FAKE, FAKE,
                                   None, None, None, None, None, None) == B.SPARGE_ERR_WORKSPACE


def test_binding_fails_loudly_without_cuda_tensors():
    import torch
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16)
    with pytest.raises(ValueError):
        B.sparge_mask(q, q, 0.1, 0.9)
    with pytest.raises(ValueError):
        B.sparge_attn_fwd(q, q, q, None, None)
