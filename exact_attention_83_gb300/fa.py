"""Thin Python binding over libfa's C ABI (include/fa.h).

Argument marshalling only: every step of the attention path runs in libfa's
CUDA kernels.  torch supplies device memory and the current stream.  If the
library has not been built, every call raises: there is no other code path.

API
  fwd(q, k, v, o, lse, causal, scale)               -> None   (fa_fwd)
  bwd_preprocess(o, do, delta)                       -> None   (fa_bwd_preprocess)
  bwd(q, k, v, do, lse, delta, dq, dk, dv, causal, scale) -> None (fa_bwd)
  attention_fwd(q, k, v, causal, scale)             -> (o, lse)   allocates outputs
  attention_bwd(q, k, v, o, lse, do, causal, scale) -> (dq, dk, dv)
  attention(q, k, v, causal, scale)                 -> o with autograd; double
                                                       backward raises
Tensors are CUDA [B, H, N, D] with unit last stride (any other strides), all of
one dtype (float32, float16, bfloat16); lse and delta are contiguous float32
[B, H, N].
"""

from __future__ import annotations

import ctypes
import math
import os
import threading

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libfa.so")

FA_F32, FA_F16, FA_BF16 = 0, 1, 2
_DTYPE_CODE = {torch.float32: FA_F32, torch.float16: FA_F16, torch.bfloat16: FA_BF16}
FA_PATH_AUTO, FA_PATH_FFMA = 0, 1

STATUS_NAMES = {
    0: "FA_OK", 1: "FA_ERR_NULL", 2: "FA_ERR_SHAPE", 3: "FA_ERR_HEADDIM",
    4: "FA_ERR_DTYPE", 5: "FA_ERR_STRIDE", 6: "FA_ERR_ALIGN", 7: "FA_ERR_LAUNCH",
    8: "FA_ERR_TIMEOUT", 9: "FA_ERR_ARCH", 10: "FA_ERR_SCALE", 11: "FA_ERR_ARG",
    12: "FA_ERR_SCRATCH",
}

EXPORTED = ("fa_fwd", "fa_bwd_preprocess", "fa_bwd", "fa_get_device_status",
            "fa_status_string", "fa_set_path", "fa_set_wait_timeout_ns",
            "fa_set_profile_events", "fa_version", "fa_bwd_noalloc",
            "fa_test_withhold_next_arrival")


class FAError(RuntimeError):
    def __init__(self, code: int, where: str):
        self.code = code
        super().__init__(f"{where}: {STATUS_NAMES.get(code, code)}")


_lock = threading.Lock()
_lib = None
_i64 = ctypes.c_int64
_vp = ctypes.c_void_p
_s4 = ctypes.POINTER(ctypes.c_int64)


def load_library(path: str = LIB_PATH):
    """Load libfa.so and declare its signatures.  Raises if it is missing."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(path):
            raise RuntimeError(f"libfa.so is not built ({path}); run __graft_entry__.build()")
        lib = ctypes.CDLL(path)
        lib.fa_fwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _i64, _i64, _i64, _i64,
                               _s4, _s4, _s4, _s4, ctypes.c_int, ctypes.c_float,
                               ctypes.c_int, _vp]
        lib.fa_fwd.restype = ctypes.c_int
        lib.fa_bwd_preprocess.argtypes = [_vp, _vp, _vp, _i64, _i64, _i64, _i64,
                                          _s4, _s4, ctypes.c_int, _vp]
        lib.fa_bwd_preprocess.restype = ctypes.c_int
        lib.fa_bwd.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                               _i64, _i64, _i64, _i64, _s4, _s4, _s4, _s4, _s4,
                               _s4, _s4, ctypes.c_int, ctypes.c_float, ctypes.c_int,
                               _vp]
        lib.fa_bwd.restype = ctypes.c_int
        lib.fa_bwd_noalloc.argtypes = [_vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp, _vp,
                                       _i64, _i64, _i64, _i64, _s4, _s4, _s4, _s4, _s4,
                                       _s4, _s4, _s4, ctypes.c_int, ctypes.c_float,
                                       ctypes.c_int, _vp]
        lib.fa_bwd_noalloc.restype = ctypes.c_int
        lib.fa_get_device_status.argtypes = [_vp]
        lib.fa_get_device_status.restype = ctypes.c_int
        lib.fa_status_string.argtypes = [ctypes.c_int]
        lib.fa_status_string.restype = ctypes.c_char_p
        lib.fa_set_path.argtypes = [ctypes.c_int]
        lib.fa_set_path.restype = ctypes.c_int
        lib.fa_set_wait_timeout_ns.argtypes = [ctypes.c_uint64]
        lib.fa_set_wait_timeout_ns.restype = None
        lib.fa_set_profile_events.argtypes = [ctypes.c_void_p]
        lib.fa_set_profile_events.restype = None
        lib.fa_version.restype = ctypes.c_int
        lib.fa_test_withhold_next_arrival.argtypes = []
        lib.fa_test_withhold_next_arrival.restype = None
        if os.environ.get("FA_WAIT_TIMEOUT_NS"):
            lib.fa_set_wait_timeout_ns(int(os.environ["FA_WAIT_TIMEOUT_NS"]))
        _lib = lib
        return lib


def _strides(t: torch.Tensor):
    return (ctypes.c_int64 * 4)(*t.stride())


def _stream(t: torch.Tensor):
    return ctypes.c_void_p(torch.cuda.current_stream(t.device).cuda_stream)


def _check(code: int, where: str):
    if code != 0:
        raise FAError(code, where)


def _dims(q: torch.Tensor):
    if q.dim() != 4:
        raise ValueError("expected [B, H, N, D] tensors")
    if q.dtype not in _DTYPE_CODE:
        raise TypeError(f"unsupported dtype {q.dtype}")
    if not q.is_cuda:
        raise ValueError("tensors must be on a CUDA device")
    return q.shape


def _same(ref: torch.Tensor, *ts):
    for t in ts:
        if t.shape != ref.shape or t.dtype != ref.dtype or t.device != ref.device:
            raise ValueError("q, k, v, o, do, dq, dk, dv must share shape, dtype and device")


def _scale(D: int, scale):
    return 1.0 / math.sqrt(D) if scale is None else float(scale)


def fwd(q, k, v, o, lse, causal: bool, scale=None):
    B, H, N, D = _dims(q)
    _same(q, k, v, o)
    lib = load_library()
    with torch.cuda.device(q.device):
        code = lib.fa_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                          lse.data_ptr(), B, H, N, D, _strides(q), _strides(k),
                          _strides(v), _strides(o), int(bool(causal)),
                          _scale(D, scale), _DTYPE_CODE[q.dtype], _stream(q))
    _check(code, "fa_fwd")


def bwd_preprocess(o, do, delta):
    B, H, N, D = _dims(o)
    _same(o, do)
    lib = load_library()
    with torch.cuda.device(o.device):
        code = lib.fa_bwd_preprocess(o.data_ptr(), do.data_ptr(), delta.data_ptr(),
                                     B, H, N, D, _strides(o), _strides(do),
                                     _DTYPE_CODE[o.dtype], _stream(o))
    _check(code, "fa_bwd_preprocess")


def bwd(q, k, v, do, lse, delta, dq, dk, dv, causal: bool, scale=None):
    B, H, N, D = _dims(q)
    _same(q, k, v, do, dq, dk, dv)
    lib = load_library()
    with torch.cuda.device(q.device):
        code = lib.fa_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), do.data_ptr(),
                          lse.data_ptr(), delta.data_ptr(), dq.data_ptr(),
                          dk.data_ptr(), dv.data_ptr(), B, H, N, D, _strides(q),
                          _strides(k), _strides(v), _strides(do), _strides(dq),
                          _strides(dk), _strides(dv), int(bool(causal)),
                          _scale(D, scale), _DTYPE_CODE[q.dtype], _stream(q))
    _check(code, "fa_bwd")


def bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, causal: bool, scale=None):
    """fa_bwd_noalloc: the backward for callers that cannot allocate device
    memory; Delta lives in a fixed buffer inside libfa (B*H*N must not exceed
    its FA_NOALLOC_MAX_ROWS rows).  Calls must not overlap on the GPU."""
    B, H, N, D = _dims(q)
    _same(q, k, v, o, do, dq, dk, dv)
    lib = load_library()
    with torch.cuda.device(q.device):
        code = lib.fa_bwd_noalloc(q.data_ptr(), k.data_ptr(), v.data_ptr(), o.data_ptr(),
                                  do.data_ptr(), lse.data_ptr(), dq.data_ptr(), dk.data_ptr(),
                                  dv.data_ptr(), B, H, N, D, _strides(q), _strides(k),
                                  _strides(v), _strides(o), _strides(do), _strides(dq),
                                  _strides(dk), _strides(dv), int(bool(causal)),
                                  _scale(D, scale), _DTYPE_CODE[q.dtype], _stream(q))
    _check(code, "fa_bwd_noalloc")


def device_status(device=None) -> int:
    """fa_get_device_status on the current stream of `device` (syncs it)."""
    dev = torch.device("cuda", torch.cuda.current_device()) if device is None else torch.device(device)
    lib = load_library()
    with torch.cuda.device(dev):
        return lib.fa_get_device_status(ctypes.c_void_p(torch.cuda.current_stream(dev).cuda_stream))


def set_path(path: int) -> None:
    _check(load_library().fa_set_path(int(path)), "fa_set_path")


def set_wait_timeout_ns(ns: int) -> None:
    load_library().fa_set_wait_timeout_ns(int(ns))


def set_profile_events(events) -> None:
    """events: three torch.cuda.Event(enable_timing=True) recorded by later
    fa_bwd calls before dK/dV, between dK/dV and dQ, and after dQ; None turns
    the hook off."""
    lib = load_library()
    if events is None:
        lib.fa_set_profile_events(None)
        return
    handles = (ctypes.c_void_p * 3)(*[ev.cuda_event for ev in events])
    lib.fa_set_profile_events(ctypes.cast(handles, ctypes.c_void_p))


def attention_fwd(q, k, v, causal: bool = False, scale=None):
    B, H, N, D = _dims(q)
    o = torch.empty((B, H, N, D), dtype=q.dtype, device=q.device)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    fwd(q, k, v, o, lse, causal, scale)
    return o, lse


def attention_bwd(q, k, v, o, lse, do, causal: bool = False, scale=None):
    B, H, N, D = _dims(q)
    delta = torch.empty((B, H, N), dtype=torch.float32, device=q.device)
    bwd_preprocess(o, do, delta)
    dq = torch.empty((B, H, N, D), dtype=q.dtype, device=q.device)
    dk = torch.empty_like(dq)
    dv = torch.empty_like(dq)
    bwd(q, k, v, do, lse, delta, dq, dk, dv, causal, scale)
    return dq, dk, dv


class _Attention(torch.autograd.Function):
    @staticmethod
    def forward(ctx, q, k, v, causal, scale):
        o, lse = attention_fwd(q, k, v, causal, scale)
        ctx.save_for_backward(q, k, v, o, lse)
        ctx.causal, ctx.scale = causal, scale
        return o

    @staticmethod
    @torch.autograd.function.once_differentiable
    def backward(ctx, do):
        q, k, v, o, lse = ctx.saved_tensors
        if do.stride(-1) != 1:
            do = do.contiguous()
        dq, dk, dv = attention_bwd(q, k, v, o, lse, do, ctx.causal, ctx.scale)
        return dq, dk, dv, None, None


def attention(q, k, v, causal: bool = False, scale=None):
    """Exact softmax attention with autograd.  Second-order gradients are
    refused (once_differentiable raises) rather than silently wrong."""
    return _Attention.apply(q, k, v, causal, scale)
