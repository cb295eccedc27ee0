"""fp64 CPU oracle for exact attention (forward and backward).

TEST INFRASTRUCTURE ONLY: the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg use it; the library never does.  It computes the
plain definition of softmax attention and its gradient in double precision
(see ``oracle_attn.cpp`` for the formulas and their sources) and shares no code
with the CUDA path.

Every function takes numpy arrays (or CPU tensors) q, do [B, Hq, Nq, D] and
k, v [B, Hkv, Nk, D] (any dtype, any strides; they are converted to
contiguous float64 here, which is exact for fp16, bf16 and fp32 values) and
returns float64 arrays.  Optional: dropout=dropout_params(p, seed, offset).
varlen_fwd_bwd takes packed [total, H, D] sequences with their offsets.

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


class Dropout(ctypes.Structure):
    """oracle_dropout of oracle_attn.cpp."""
    _fields_ = [("on", ctypes.c_int), ("thr", ctypes.c_uint32), ("rscale", ctypes.c_double),
                ("key0", ctypes.c_uint32), ("key1", ctypes.c_uint32),
                ("offset", ctypes.c_uint32), ("bh0", ctypes.c_int64)]


def dropout_params(p: float = 0.0, seed: int = 0, offset: int = 0, bh0: int = 0):
    """The dropout description for probability p (taken as a float32 value, as
    the library takes it): keep iff the 16-bit Philox half is >=
    floor(p * 65536); kept weights scaled by 1 / (1 - p)."""
    p32 = float(np.float32(p))
    if not 0.0 <= p32 < 1.0:
        raise ValueError("dropout probability must be in [0, 1)")
    d = Dropout()
    if p32 > 0.0:
        d.on = 1
        d.thr = min(int(np.floor(p32 * 65536.0)), 65535)
        d.rscale = 1.0 / (1.0 - p32)
        d.key0 = int(seed) & 0xFFFFFFFF
        d.key1 = (int(seed) >> 32) & 0xFFFFFFFF
        d.offset = int(offset) & 0xFFFFFFFF
        d.bh0 = int(bh0)
    return d


_DIMS = [_i64] * 6          # B, Hq, Hkv, Nq, Nk, D
_COMMON = [ctypes.c_int, ctypes.c_double, ctypes.POINTER(Dropout)]   # causal, scale, dropout
_ROWS = [_i64, ctypes.POINTER(ctypes.c_int64)]


def _load():
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        build()
        lib = ctypes.CDLL(_LIB_PATH)
        lib.oracle_fwd.argtypes = [_dp] * 3 + _DIMS + _COMMON + [_dp, _dp]
        lib.oracle_fwd_rows.argtypes = [_dp] * 3 + _DIMS + _COMMON + _ROWS + [_dp, _dp]
        lib.oracle_fwd_bwd.argtypes = [_dp] * 4 + _DIMS + _COMMON + [_dp] * 6
        lib.oracle_query_rows.argtypes = [_dp] * 4 + _DIMS + _COMMON + _ROWS + [_dp] * 6
        lib.oracle_key_rows.argtypes = [_dp] * 4 + _DIMS + _COMMON + _ROWS + [_dp] * 4
        lib.oracle_magnitudes.argtypes = [_dp] * 4 + _DIMS + _COMMON + [_dp] * 4
        lib.oracle_philox4x32_10.argtypes = [ctypes.POINTER(ctypes.c_uint32)] * 3
        lib.oracle_dropout_z.argtypes = [ctypes.POINTER(Dropout), _i64, _i64, _i64, _i64, _dp]
        lib.oracle_dense.argtypes = [_dp, _dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                     ctypes.c_int, ctypes.c_double, _dp, _dp, _dp,
                                     _dp, _dp, _dp]
        lib.oracle_fwd_tiled.argtypes = [_dp, _dp, _dp, _i64, _i64, _i64, _i64,
                                         ctypes.c_int, ctypes.c_double, _i64, _i64,
                                         _dp, _dp]
        lib.oracle_bwd_tiled.argtypes = [_dp, _dp, _dp, _dp, _dp, _dp, _i64, _i64,
                                         _i64, _i64, ctypes.c_int, ctypes.c_double,
                                         _i64, _i64, _dp, _dp, _dp]
        lib.oracle_num_threads.restype = ctypes.c_int
        lib.oracle_set_num_threads.argtypes = [ctypes.c_int]
        _lib = lib
        return lib


def _f64(a) -> np.ndarray:
    if hasattr(a, "detach"):          # torch tensor
        a = a.detach().cpu().double().numpy()
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(_dp)


def _ptr_or_null(a):
    return None if a is None else _ptr(a)


def _shape(q: np.ndarray):
    if q.ndim != 4:
        raise ValueError("expected [B, H, N, D]")
    return q.shape


def _dims(q: np.ndarray, k: np.ndarray):
    """(B, Hq, Hkv, Nq, Nk, D) from q [B, Hq, Nq, D] and k [B, Hkv, Nk, D]."""
    B, Hq, Nq, D = _shape(q)
    Bk, Hkv, Nk, Dk = _shape(k)
    if Bk != B or Dk != D or Hkv < 1 or Hq % Hkv != 0:
        raise ValueError("k must be [B, Hkv, Nk, D] with Hq % Hkv == 0")
    return B, Hq, Hkv, Nq, Nk, D


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def default_scale(D: int) -> float:
    return 1.0 / float(np.sqrt(D))


def philox4x32_10(counter, key):
    """Philox4x32-10 of one counter (4 uint32) under one key (2 uint32)."""
    c = (ctypes.c_uint32 * 4)(*[int(x) & 0xFFFFFFFF for x in counter])
    kk = (ctypes.c_uint32 * 2)(*[int(x) & 0xFFFFFFFF for x in key])
    out = (ctypes.c_uint32 * 4)()
    _load().oracle_philox4x32_10(c, kk, out)
    return tuple(int(x) for x in out)


def dropout_z(dropout, bh: int, nq: int, nk: int, i0: int = 0) -> np.ndarray:
    """Z = keep / (1 - p) of the weights (i0 + r, j), r < nq, j < nk, of flat
    query head bh (positions within the sequence), [nq, nk] fp64: the factor
    the oracle's forward and backward apply."""
    z = np.empty((nq, nk), dtype=np.float64)
    _load().oracle_dropout_z(ctypes.byref(dropout), int(bh), int(i0), int(nq), int(nk), _ptr(z))
    return z


def _common(causal, scale, D, dropout):
    scale = default_scale(D) if scale is None else float(scale)
    dr = dropout if dropout is not None else Dropout()
    return int(bool(causal)), scale, ctypes.byref(dr)


def fwd(q, k, v, causal: bool, scale: float | None = None, dropout=None):
    """O [B,Hq,Nq,D] and L [B,Hq,Nq] (natural-log log-sum-exp of the scaled
    scores).  k, v: [B, Hkv, Nk, D].  dropout: dropout_params(...) or None."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    dims = _dims(q, k)
    B, Hq, Hkv, Nq, Nk, D = dims
    o = np.empty((B, Hq, Nq, D)); L = np.empty((B, Hq, Nq))
    _load().oracle_fwd(_ptr(q), _ptr(k), _ptr(v), *dims, *_common(causal, scale, D, dropout),
                       _ptr(o), _ptr(L))
    return o, L


def fwd_rows(q, k, v, causal: bool, rows, scale: float | None = None, dropout=None):
    """Forward for sampled rows.  rows: int array [n, 2] of (b*Hq + h, i)."""
    q, k, v = _f64(q), _f64(k), _f64(v)
    dims = _dims(q, k)
    D = dims[5]
    rows, rp = _rows(rows)
    n = rows.shape[0]
    o = np.empty((n, D)); L = np.empty((n,))
    _load().oracle_fwd_rows(_ptr(q), _ptr(k), _ptr(v), *dims,
                            *_common(causal, scale, D, dropout), n, rp, _ptr(o), _ptr(L))
    return o, L


def fwd_bwd(q, k, v, do, causal: bool, scale: float | None = None, dropout=None):
    """Returns dict with o, lse, delta, dq (query-shaped) and dk, dv
    (key-shaped), all float64."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dims = _dims(q, k)
    B, Hq, Hkv, Nq, Nk, D = dims
    o = np.empty((B, Hq, Nq, D)); L = np.empty((B, Hq, Nq)); delta = np.empty((B, Hq, Nq))
    dq = np.empty_like(o); dk = np.empty((B, Hkv, Nk, D)); dv = np.empty_like(dk)
    _load().oracle_fwd_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(do), *dims,
                           *_common(causal, scale, D, dropout), _ptr(o), _ptr(L),
                           _ptr(delta), _ptr(dq), _ptr(dk), _ptr(dv))
    return dict(o=o, lse=L, delta=delta, dq=dq, dk=dk, dv=dv)


def _rows(rows):
    rows = np.ascontiguousarray(np.asarray(rows, dtype=np.int64).reshape(-1, 2))
    return rows, rows.ctypes.data_as(ctypes.POINTER(ctypes.c_int64))


def query_rows(q, k, v, do, causal: bool, rows, scale: float | None = None,
               magnitudes: bool = False, dropout=None):
    """Row-local outputs for sampled query rows (rows: [n, 2] of (b*Hq+h, i)).
    Returns dict o [n,D], lse [n], delta [n], dq [n,D]; with magnitudes=True
    also o_abs, dq_abs [n,D] (the sums of magnitudes()) for those rows."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dims = _dims(q, k)
    D = dims[5]
    rows, rp = _rows(rows)
    n = rows.shape[0]
    o = np.empty((n, D)); L = np.empty((n,)); delta = np.empty((n,)); dq = np.empty((n, D))
    oa = np.empty((n, D)) if magnitudes else None
    qa = np.empty((n, D)) if magnitudes else None
    _load().oracle_query_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), *dims,
                              *_common(causal, scale, D, dropout), n, rp, _ptr(o), _ptr(L),
                              _ptr(delta), _ptr(dq), _ptr_or_null(oa), _ptr_or_null(qa))
    out = dict(o=o, lse=L, delta=delta, dq=dq)
    if magnitudes:
        out.update(o_abs=oa, dq_abs=qa)
    return out


def key_rows(q, k, v, do, causal: bool, rows, scale: float | None = None,
             magnitudes: bool = False, dropout=None):
    """dK, dV for sampled key rows (rows: [n, 2] of (b*Hkv+hk, j)).
    Returns dict dk [n,D], dv [n,D]; with magnitudes=True also dk_abs, dv_abs."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dims = _dims(q, k)
    D = dims[5]
    rows, rp = _rows(rows)
    n = rows.shape[0]
    dk = np.empty((n, D)); dv = np.empty((n, D))
    ka = np.empty((n, D)) if magnitudes else None
    va = np.empty((n, D)) if magnitudes else None
    _load().oracle_key_rows(_ptr(q), _ptr(k), _ptr(v), _ptr(do), *dims,
                            *_common(causal, scale, D, dropout), n, rp, _ptr(dk), _ptr(dv),
                            _ptr_or_null(ka), _ptr_or_null(va))
    out = dict(dk=dk, dv=dv)
    if magnitudes:
        out.update(dk_abs=ka, dv_abs=va)
    return out


def magnitudes(q, k, v, do, causal: bool, scale: float | None = None, dropout=None):
    """Componentwise magnitude sums for rounding-error bounds: dict o, dq (query-
    shaped), dk, dv (key-shaped) of sum ZP|V|, scale sum |dS||K|,
    scale sum |dS||Q|, sum ZP|dO|."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    dims = _dims(q, k)
    B, Hq, Hkv, Nq, Nk, D = dims
    o = np.empty((B, Hq, Nq, D)); dq = np.empty_like(o)
    dk = np.empty((B, Hkv, Nk, D)); dv = np.empty_like(dk)
    _load().oracle_magnitudes(_ptr(q), _ptr(k), _ptr(v), _ptr(do), *dims,
                              *_common(causal, scale, D, dropout), _ptr(o), _ptr(dq),
                              _ptr(dk), _ptr(dv))
    return dict(o=o, dq=dq, dk=dk, dv=dv)


def varlen_fwd_bwd(q, k, v, do, cu_q, cu_k, causal: bool, scale: float | None = None,
                   p: float = 0.0, seed: int = 0, offset: int = 0, magnitudes_too: bool = False):
    """Packed sequences: q, do [total_q, Hq, D]; k, v [total_k, Hkv, D]; cu_q,
    cu_k the B+1 offsets.  Each sequence is an independent attention problem
    (its own rows only, positions counted from its first row); sequence b's
    dropout mask numbers its heads b*Hq + h.  Returns o, dq [total_q, Hq, D],
    lse, delta [Hq, total_q], dk, dv [total_k, Hkv, D] (and the *_abs
    magnitude sums when magnitudes_too)."""
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(do)
    cu_q = [int(x) for x in np.asarray(cu_q)]
    cu_k = [int(x) for x in np.asarray(cu_k)]
    Tq, Hq, D = q.shape
    Tk, Hkv, _ = k.shape
    out = dict(o=np.zeros((Tq, Hq, D)), dq=np.zeros((Tq, Hq, D)), lse=np.zeros((Hq, Tq)),
               delta=np.zeros((Hq, Tq)), dk=np.zeros((Tk, Hkv, D)), dv=np.zeros((Tk, Hkv, D)))
    if magnitudes_too:
        for key, shape in (("o_abs", (Tq, Hq, D)), ("dq_abs", (Tq, Hq, D)),
                           ("dk_abs", (Tk, Hkv, D)), ("dv_abs", (Tk, Hkv, D))):
            out[key] = np.zeros(shape)
    for b in range(len(cu_q) - 1):
        qs, qe, ks, ke = cu_q[b], cu_q[b + 1], cu_k[b], cu_k[b + 1]
        if qe == qs and ke == ks:
            continue
        seq = lambda t, s, e: np.ascontiguousarray(t[s:e].transpose(1, 0, 2)[None])
        qb, dob = seq(q, qs, qe), seq(do, qs, qe)
        kb, vb = seq(k, ks, ke), seq(v, ks, ke)
        dr = dropout_params(p, seed, offset, bh0=b * Hq)
        if qe > qs:
            r = fwd_bwd(qb, kb, vb, dob, causal, scale, dr)
            m = magnitudes(qb, kb, vb, dob, causal, scale, dr) if magnitudes_too else None
        else:
            continue     # no query: dK = dV = 0 for these keys
        unseq = lambda a: a[0].transpose(1, 0, 2)
        out["o"][qs:qe] = unseq(r["o"]); out["dq"][qs:qe] = unseq(r["dq"])
        out["lse"][:, qs:qe] = r["lse"][0]; out["delta"][:, qs:qe] = r["delta"][0]
        out["dk"][ks:ke] = unseq(r["dk"]); out["dv"][ks:ke] = unseq(r["dv"])
        if m is not None:
            out["o_abs"][qs:qe] = unseq(m["o"]); out["dq_abs"][qs:qe] = unseq(m["dq"])
            out["dk_abs"][ks:ke] = unseq(m["dk"]); out["dv_abs"][ks:ke] = unseq(m["dv"])
    return out


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
