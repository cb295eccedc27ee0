"""fp64 CPU oracle for exact attention (forward and backward).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the library never does.  It computes the
plain definition of softmax attention and its gradient in double precision
(see ``oracle_attn.cpp`` for the formulas and their sources) and shares no code
with the CUDA path.

Every function takes numpy arrays in [B, H, N, D] (any dtype, any strides; they
are converted to contiguous float64 here, which is exact for fp16, bf16 and
fp32 values) and returns float64 arrays.

Parity is pinned for every function here; no function is unpinned.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle_attn.cpp")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lock = threading.Lock()
_lib = None

_dp = ctypes.POINTER(ctypes.c_double)
_i64 = ctypes.c_int64


def build(force: bool = False) -> str:
    """Compile oracle_attn.cpp into liboracle.so (plain g++, -O2, OpenMP)."""
    if (not force and os.path.exists(_LIB_PATH)
            and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC)):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp.%d" % os.getpid()
    cmd = ["g++", "-std=c++17", "-O2", "-fopenmp", "-fPIC", "-shared",
           _SRC, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_fwd.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                   ctypes.c_int, ctypes.c_double, _dp, _dp]
        lib.oracle_fwd_rows.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                        ctypes.c_int, ctypes.c_double, _i64,
                                        ctypes.POINTER(ctypes.c_int64), _dp, _dp]
        lib.oracle_fwd_bwd.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                       _i64, ctypes.c_int, ctypes.c_double,
                                       _dp, _dp, _dp, _dp, _dp, _dp]
        lib.oracle_dense.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                     ctypes.c_int, ctypes.c_double, _dp, _dp,
                                     _dp, _dp, _dp, _dp]
        lib.oracle_fwd_tiled.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                         ctypes.c_int, ctypes.c_double, _i64,
                                         _i64, _dp, _dp]
        lib.oracle_bwd_tiled.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64,
                                         _i64, _i64, _i64, ctypes.c_int,
                                         ctypes.c_double, _i64, _i64, _dp, _dp,
                                         _dp]
        lib.oracle_query_rows.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                          _i64, ctypes.c_int, ctypes.c_double,
                                          _i64, ctypes.POINTER(ctypes.c_int64),
                                          _dp, _dp, _dp, _dp, _dp, _dp]
        lib.oracle_key_rows.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64,
                                        _i64, ctypes.c_int, ctypes.c_double,
                                        _i64, ctypes.POINTER(ctypes.c_int64),
                                        _dp, _dp, _dp, _dp]
        lib.oracle_magnitudes.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                          ctypes.c_int, ctypes.c_double, _dp, _dp, _dp,
                                          _dp]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _f64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a CPU torch tensor: go through float64 exactly
        import torch
        x = x.detach().to("cpu", torch.float64).numpy()
    return np.ascontiguousarray(np.asarray(x, dtype=np.float64))


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _ptr_or_null(a):
    return None if a is None else _ptr(a)


def _shape(q: np.ndarray):
    if q.ndim != 4:
        raise ValueError("expected [B, H, N, D]")
    return q.shape


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def default_scale(D: int) -> float:
    return 1.0 / float(np.sqrt(D))


def fwd(q, k, v, causal: bool, scale: float | None = None):
    """O [B,H,N,D] and L [B,H,N] (natural-log log-sum-exp of the scaled scores)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, D = _shape(q)
    scale = default_scale(D) if scale is None else float(scale)
    o = np.empty((B, H, N, D)); L = np.empty((B, H, N))
    _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), B, H, N, D, int(bool(causal)),
                       scale, _ptr(o), _ptr(L))
    return o, L


def fwd_rows(q, k, v, causal: bool, rows, scale: float | None = None):
    """Forward for sampled rows.  rows: int array [n, 2] of (b*H + h, i)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, D = _shape(q)
    scale = default_scale(D) if scale is None else float(scale)
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    n = rows.shape[0]
    o = np.empty((n, D)); L = np.empty((n,))
    _load().oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), B, H, N, D,
                            int(bool(causal)), scale, n,
                            rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64)),
                            _ptr(o), _ptr(L))
    return o, L


def fwd_bwd(q, k, v, do, causal: bool, scale: float | None = None):
    """Returns dict with o, lse, delta, dq, dk, dv (all float64)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, D = _shape(q)
    scale = default_scale(D) if scale is None else float(scale)
    o = np.empty((B, H, N, D)); L = np.empty((B, H, N)); delta = np.empty((B, H, N))
    dq = np.empty_like(o); dk = np.empty_like(o); dv = np.empty_like(o)
    _load().oracle_fwd_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, H, N, D,
                           int(bool(causal)), scale, _ptr(o), _ptr(L),
                           _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv))
    return dict(o=o, lse=L, delta=delta, dq=dq, dk=dk, dv=dv)


def _rows(rows):
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    return rows, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def query_rows(q, k, v, do, causal: bool, rows, scale: float | None = None,
               magnitudes: bool = False):
    """Row-local outputs for sampled query rows (rows: [n, 2] of (b*H+h, i)).
    Returns dict o [n,D], lse [n], delta [n], dq [n,D]; with magnitudes=True
    also o_abs, dq_abs [n,D] (the sums of magnitudes()) for those rows."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, D = _shape(q)
    scale = default_scale(D) if scale is None else float(scale)
    rows, rp = _rows(rows)
    n = rows.shape[0]
    o = np.empty((n, D)); L = np.empty((n,)); delta = np.empty((n,)); dq = np.empty((n, D))
    oa = np.empty((n, D)) if magnitudes else None
    qa = np.empty((n, D)) if magnitudes else None
    _load().oracle_query_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, H, N, D,
                              int(bool(causal)), scale, n, rp, _ptr(o), _ptr(L),
                              _ptr(delta), _ptr(dq), _ptr_or_null(oa), _ptr_or_null(qa))
    out = dict(o=o, lse=L, delta=delta, dq=dq)
    if magnitudes:
        out.update(o_abs=oa, dq_abs=qa)
    return out


def key_rows(q, k, v, do, causal: bool, rows, scale: float | None = None,
             magnitudes: bool = False):
    """dK, dV for sampled key rows (rows: [n, 2] of (b*H+h, j)).
    Returns dict dk [n,D], dv [n,D]; with magnitudes=True also dk_abs, dv_abs."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, D = _shape(q)
    scale = default_scale(D) if scale is None else float(scale)
    rows, rp = _rows(rows)
    n = rows.shape[0]
    dk = np.empty((n, D)); dv = np.empty((n, D))
    ka = np.empty((n, D)) if magnitudes else None
    va = np.empty((n, D)) if magnitudes else None
    _load().oracle_key_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, H, N, D,
                            int(bool(causal)), scale, n, rp, _ptr(dk), _ptr(dv),
                            _ptr_or_null(ka), _ptr_or_null(va))
    out = dict(dk=dk, dv=dv)
    if magnitudes:
        out.update(dk_abs=ka, dv_abs=va)
    return out


def magnitudes(q, k, v, do, causal: bool, scale: float | None = None):
    """Componentwise magnitude sums for rounding-error bounds: dict o, dq, dk,
    dv of sum P|V|, scale sum |dS||K|, scale sum |dS||Q|, sum P|dO|."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, D = _shape(q)
    scale = default_scale(D) if scale is None else float(scale)
    o = np.empty((B, H, N, D)); dq = np.empty_like(o); dk = np.empty_like(o); dv = np.empty_like(o)
    _load().oracle_magnitudes(_ptr(q), _ptr(k), _ptr(v), _ptr(do), B, H, N, D,
                              int(bool(causal)), scale, _ptr(o), _ptr(dq), _ptr(dk), _ptr(dv))
    return dict(o=o, dq=dq, dk=dk, dv=dv)


def dense(q, k, v, do, causal: bool, scale: float | None = None,
          want_probs: bool = False):
    """Full N x N materialisation (small N only).  Same keys as fwd_bwd, plus
    'p' [B,H,N,N] when want_probs.  do may be None (forward only)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    B, H, N, D = _shape(q)
    if N > 4096:
        raise ValueError("dense oracle is for small N")
    scale = default_scale(D) if scale is None else float(scale)
    o = np.empty((B, H, N, D)); L = np.empty((B, H, N))
    dq = np.zeros_like(o); dk = np.zeros_like(o); dv = np.zeros_like(o)
    p = np.empty((B, H, N, N)) if want_probs else None
    gp = None
    if do is not None:
        do = _f64(do)
        gp = _ptr(do)
    _load().oracle_dense(_ptr(q), _ptr(k), _ptr(v), gp, B, H, N, D,
                         int(bool(causal)), scale, _ptr(o), _ptr(L), _ptr(dq),
                         _ptr(dk), _ptr(dv), _ptr(p) if p is not None else None)
    out = dict(o=o, lse=L)
    if do is not None:
        out.update(dq=dq, dk=dk, dv=dv)
    if p is not None:
        out["p"] = p
    return out


def tiled(q, k, v, do, causal: bool, bq: int, bk: int,
          scale: float | None = None):
    """fp64 restatement of the tiled FlashAttention-2 recurrences with query
    tiles of bq rows and key tiles of bk rows (tile-invariance pin only)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    B, H, N, D = _shape(q)
    scale = default_scale(D) if scale is None else float(scale)
    o = np.empty((B, H, N, D)); L = np.empty((B, H, N))
    lib = _load()
    lib.oracle_fwd_tiled(_ptr(q), _ptr(k), _ptr(v), B, H, N, D,
                         int(bool(causal)), scale, int(bq), int(bk), _ptr(o),
                         _ptr(L))
    dq = np.empty_like(o); dk = np.empty_like(o); dv = np.empty_like(o)
    lib.oracle_bwd_tiled(_ptr(q), _ptr(k), _ptr(v), _ptr(o), _ptr(L), _ptr(do),
                         B, H, N, D, int(bool(causal)), scale, int(bq), int(bk),
                         _ptr(dq), _ptr(dk), _ptr(dv))
    return dict(o=o, lse=L, dq=dq, dk=dk, dv=dv)
