"""Thin ctypes binding over ``libsparge.so`` (argument marshalling only).

Every step of the hot path runs in the library's CUDA kernels; this module
only allocates outputs with torch, passes raw device pointers, sizes and the
current CUDA stream, and turns a negative status into ``SpargeError``.  There
is no CPU fallback: if the library is missing or no GPU is present, calls
raise.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import _build

__all__ = [
    "SpargeError",
    "Shape",
    "load_library",
    "library_path",
    "status_string",
    "sparge_pool",
    "sparge_mask",
    "sparge_mask_from_prob",
    "sparge_attn_fwd",
    "sparge_attn_bwd",
    "sparge_debug_wait_probe",
    "num_blocks",
    "SPARGE_OK",
    "SPARGE_ERR_INVALID_ARG",
    "SPARGE_ERR_UNSUPPORTED",
    "SPARGE_ERR_MISALIGNED",
    "SPARGE_ERR_WORKSPACE",
    "SPARGE_ERR_CUDA",
    "SPARGE_ERR_TIMEOUT",
]

SPARGE_OK = 0
SPARGE_ERR_INVALID_ARG = -1
SPARGE_ERR_UNSUPPORTED = -2
SPARGE_ERR_MISALIGNED = -3
SPARGE_ERR_WORKSPACE = -4
SPARGE_ERR_CUDA = -5
SPARGE_ERR_TIMEOUT = -6

BLOCK_Q = 128
BLOCK_KV = 64


class SpargeError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {status_string(code)} ({code})")


class Shape(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("H", ctypes.c_int32), ("N", ctypes.c_int32),
                ("d", ctypes.c_int32), ("block_q", ctypes.c_int32), ("block_kv", ctypes.c_int32)]


_P = ctypes.c_void_p
_SZ = ctypes.c_size_t
_F = ctypes.c_float
_I = ctypes.c_int
_SHP = ctypes.POINTER(Shape)

_SIGNATURES = {
    "sparge_version": ([], _I),
    "sparge_status_string": ([_I], ctypes.c_char_p),
    "sparge_pool": ([_SHP, _P, _P, _P, _P, _P], _I),
    "sparge_mask_workspace_bytes": ([_SHP, ctypes.POINTER(_SZ)], _I),
    "sparge_mask": ([_SHP, _P, _P, _F, _F, _F, _P, _P, _P, _P, _P, _P, _P, _P, _SZ, _P, _P], _I),
    "sparge_mask_from_prob": ([_SHP, _P, _F, _F, _P, _P, _P, _P, _P, _P], _I),
    "sparge_mask_noalloc": ([_SHP, _P, _P, _F, _F, _F, _P, _P, _P, _P, _P, _P, _P, _P, _P], _I),
    "sparge_attn_fwd": ([_SHP, _P, _P, _P, _P, _P, _F, _P, _P, _P, _P], _I),
    "sparge_attn_bwd_workspace_bytes": ([_SHP, ctypes.POINTER(_SZ)], _I),
    "sparge_attn_bwd": ([_SHP, _P, _P, _P, _P, _P, _P, _P, _P, _P, _P, _F, _P, _P, _P, _P, _SZ,
                         _P, _P], _I),
    "sparge_status_copy_async": ([_P, _P, _P], _I),
    "sparge_read_status": ([_P, _P, ctypes.POINTER(ctypes.c_int32)], _I),
    "sparge_debug_wait_probe": ([_P, ctypes.c_uint64, _P], _I),
}

_lib = None


def library_path() -> str:
    return _build.LIB_PATH


def load_library(build_if_missing: bool = True):
    """Loads libsparge.so (building it first if it is absent or stale and nvcc
    is available).  Raises if it cannot be loaded: there is no fallback."""
    global _lib
    if _lib is not None:
        return _lib
    path = library_path()
    if build_if_missing and (not os.path.exists(path) or _build.is_stale()):
        _build.build()
    if not os.path.exists(path):
        raise RuntimeError(f"libsparge.so not found at {path}; run __graft_entry__.build()")
    lib = ctypes.CDLL(path)
    for name, (args, res) in _SIGNATURES.items():
        fn = getattr(lib, name)
        fn.argtypes = args
        fn.restype = res
    _lib = lib
    return lib


def status_string(code: int) -> str:
    try:
        return load_library(build_if_missing=False).sparge_status_string(int(code)).decode()
    except Exception:  # pragma: no cover - only while the library is unavailable
        return f"status {code}"


def _check(code: int, where: str):
    if code != SPARGE_OK:
        raise SpargeError(code, where)


def num_blocks(n: int, b: int) -> int:
    return (n + b - 1) // b


def _shape(q: torch.Tensor, block_q=BLOCK_Q, block_kv=BLOCK_KV) -> Shape:
    if q.dim() != 4:
        raise ValueError("expected a [B, H, N, d] tensor")
    B, H, N, d = q.shape
    return Shape(B, H, N, d, block_q, block_kv)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(device) -> ctypes.c_void_p:
    return ctypes.c_void_p(torch.cuda.current_stream(device).cuda_stream)


def _need_cuda_bf16(*ts):
    for t in ts:
        if not (t.is_cuda and t.dtype == torch.bfloat16 and t.is_contiguous()):
            raise ValueError("expected contiguous bf16 CUDA tensors")


def _read_status(status: torch.Tensor) -> int:
    lib = load_library()
    host = ctypes.c_int32(0)
    _check(lib.sparge_read_status(_ptr(status), _stream(status.device), ctypes.byref(host)),
           "sparge_read_status")
    return host.value


def _finish(status: torch.Tensor, check_status: bool, where: str):
    if check_status:
        code = _read_status(status)
        if code != SPARGE_OK:
            raise SpargeError(code, where + " (device)")


def sparge_pool(q: torch.Tensor, k: torch.Tensor, block_q=BLOCK_Q, block_kv=BLOCK_KV):
    """Block means (fp32) of Q over q-blocks and of K over kv-blocks."""
    _need_cuda_bf16(q, k)
    lib = load_library()
    shp = _shape(q, block_q, block_kv)
    B, H, N, d = q.shape
    qbar = torch.empty((B, H, num_blocks(N, block_q), d), dtype=torch.float32, device=q.device)
    kbar = torch.empty((B, H, num_blocks(N, block_kv), d), dtype=torch.float32, device=q.device)
    _check(lib.sparge_pool(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(qbar), _ptr(kbar),
                           _stream(q.device)), "sparge_pool")
    return qbar, kbar


def _mask_outputs(B, H, mq, mk, device, want_csc):
    out = {
        "bitmask": torch.empty((B, H, mq, (mk + 31) // 32), dtype=torch.int32, device=device),
        "row_idx": torch.empty((B, H, mq, mk), dtype=torch.int32, device=device),
        "row_cnt": torch.empty((B, H, mq), dtype=torch.int32, device=device),
        "col_idx": None,
        "col_cnt": None,
    }
    if want_csc:
        out["col_idx"] = torch.empty((B, H, mk, mq), dtype=torch.int32, device=device)
        out["col_cnt"] = torch.empty((B, H, mk), dtype=torch.int32, device=device)
    return out


def sparge_mask(q, k, k_frac: float, p: float, softmax_scale: float = 0.0, want_csc=True,
                want_prob=False, want_logit=False, block_q=BLOCK_Q, block_kv=BLOCK_KV,
                workspace=None, out=None):
    """Hybrid Top-k + Top-p block mask.  Returns a dict with ``bitmask``
    (int32 view of the uint32 words), ``row_idx``, ``row_cnt`` and, when asked
    for, ``col_idx``, ``col_cnt``, ``prob``, ``logit``."""
    _need_cuda_bf16(q, k)
    lib = load_library()
    shp = _shape(q, block_q, block_kv)
    B, H, N, d = q.shape
    mq, mk = num_blocks(N, block_q), num_blocks(N, block_kv)
    res = out if out is not None else _mask_outputs(B, H, mq, mk, q.device, want_csc)
    res.setdefault("prob", None)
    res.setdefault("logit", None)
    if want_prob and res["prob"] is None:
        res["prob"] = torch.empty((B, H, mq, mk), dtype=torch.float32, device=q.device)
    if want_logit and res["logit"] is None:
        res["logit"] = torch.empty((B, H, mq, mk), dtype=torch.float32, device=q.device)
    if workspace is None:
        nbytes = ctypes.c_size_t(0)
        _check(lib.sparge_mask_workspace_bytes(ctypes.byref(shp), ctypes.byref(nbytes)),
               "sparge_mask_workspace_bytes")
        workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=q.device)
    _check(lib.sparge_mask(ctypes.byref(shp), _ptr(q), _ptr(k), float(k_frac), float(p),
                           float(softmax_scale), _ptr(res["bitmask"]), _ptr(res["row_idx"]),
                           _ptr(res["row_cnt"]), _ptr(res["col_idx"]), _ptr(res["col_cnt"]),
                           _ptr(res["prob"]), _ptr(res["logit"]), _ptr(workspace),
                           workspace.numel(), None, _stream(q.device)), "sparge_mask")
    return res


def sparge_mask_from_prob(prob: torch.Tensor, k_frac: float, p: float, N: int, d: int = 128,
                          want_csc=True, block_q=BLOCK_Q, block_kv=BLOCK_KV):
    """Hybrid selection on a given fp32 pooled probability map [B, H, Mq, Mk]."""
    if not (prob.is_cuda and prob.dtype == torch.float32 and prob.is_contiguous()):
        raise ValueError("prob must be a contiguous fp32 CUDA tensor")
    lib = load_library()
    B, H, mq, mk = prob.shape
    if mq != num_blocks(N, block_q) or mk != num_blocks(N, block_kv):
        raise ValueError("prob shape does not match N and the block sizes")
    shp = Shape(B, H, N, d, block_q, block_kv)
    res = _mask_outputs(B, H, mq, mk, prob.device, want_csc)
    _check(lib.sparge_mask_from_prob(ctypes.byref(shp), _ptr(prob), float(k_frac), float(p),
                                     _ptr(res["bitmask"]), _ptr(res["row_idx"]),
                                     _ptr(res["row_cnt"]), _ptr(res["col_idx"]),
                                     _ptr(res["col_cnt"]), _stream(prob.device)),
           "sparge_mask_from_prob")
    return res


def sparge_attn_fwd(q, k, v, row_idx, row_cnt, softmax_scale: float = 0.0, check_status=False,
                    out=None, lse=None, status=None, block_kv=BLOCK_KV):
    """Block-sparse attention forward; returns (O bf16, LSE fp32).  The lists
    index kv-blocks of ``block_kv`` tokens (64 or 128)."""
    _need_cuda_bf16(q, k, v)
    lib = load_library()
    shp = _shape(q, BLOCK_Q, block_kv)
    B, H, N, d = q.shape
    o = out if out is not None else torch.empty_like(q)
    lse = lse if lse is not None else torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=q.device)
    _check(lib.sparge_attn_fwd(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(row_idx),
                               _ptr(row_cnt), float(softmax_scale), _ptr(o), _ptr(lse), _ptr(st),
                               _stream(q.device)), "sparge_attn_fwd")
    _finish(st, check_status, "sparge_attn_fwd")
    return o, lse


def sparge_attn_bwd(q, k, v, o, lse, dout, row_idx, row_cnt, col_idx, col_cnt,
                    softmax_scale: float = 0.0, check_status=False, workspace=None, out=None,
                    status=None, block_kv=BLOCK_KV):
    """Gradients (dQ, dK, dV) of the block-sparse attention, mask held fixed."""
    _need_cuda_bf16(q, k, v, o, dout)
    lib = load_library()
    shp = _shape(q, BLOCK_Q, block_kv)
    if out is None:
        dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    else:
        dq, dk, dv = out
    if workspace is None:
        nbytes = ctypes.c_size_t(0)
        _check(lib.sparge_attn_bwd_workspace_bytes(ctypes.byref(shp), ctypes.byref(nbytes)),
               "sparge_attn_bwd_workspace_bytes")
        workspace = torch.empty(nbytes.value, dtype=torch.uint8, device=q.device)
    st = status if status is not None else torch.zeros(1, dtype=torch.int32, device=q.device)
    _check(lib.sparge_attn_bwd(ctypes.byref(shp), _ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(lse),
                               _ptr(dout), _ptr(row_idx), _ptr(row_cnt), _ptr(col_idx),
                               _ptr(col_cnt), float(softmax_scale), _ptr(dq), _ptr(dk), _ptr(dv),
                               _ptr(workspace), workspace.numel(), _ptr(st), _stream(q.device)),
           "sparge_attn_bwd")
    _finish(st, check_status, "sparge_attn_bwd")
    return dq, dk, dv


def sparge_debug_wait_probe(timeout_ns: int = 10_000_000, device="cuda") -> int:
    """Runs the bounded-wait probe kernel; returns the device status it wrote."""
    lib = load_library()
    st = torch.zeros(1, dtype=torch.int32, device=device)
    _check(lib.sparge_debug_wait_probe(_ptr(st), int(timeout_ns), _stream(st.device)),
           "sparge_debug_wait_probe")
    return _read_status(st)
