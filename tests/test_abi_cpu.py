"""C ABI checks that need no GPU: the library builds and loads, exports every
function include/fa.h declares, and rejects invalid arguments with the
documented status codes before touching any device (no compute call is made;
the pointers below are never dereferenced)."""

from __future__ import annotations

import ctypes
import os
import re

import pytest

from exact_attention_83_gb300 import build as fabuild
from exact_attention_83_gb300 import fa

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADERS = [os.path.join(ROOT, "include", f) for f in os.listdir(os.path.join(ROOT, "include"))
           if f.endswith(".h")]

FAKE = 0x100000          # 16-byte aligned, never dereferenced
S = (ctypes.c_int64 * 4)


@pytest.fixture(scope="module")
def lib():
    fabuild.build()
    return fa.load_library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = open(h).read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        names |= set(re.findall(r"\b(fa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_exports_every_declared_symbol(lib):
    names = declared_functions()
    assert "fa_fwd" in names and "fa_bwd" in names and "fa_bwd_preprocess" in names
    for n in names:
        assert hasattr(lib, n), f"libfa.so does not export {n}"
    assert set(fa.EXPORTED) <= set(names)


def test_status_strings(lib):
    for code, name in fa.STATUS_NAMES.items():
        assert lib.fa_status_string(code).decode().startswith(name)
    assert lib.fa_version() >= 0x000100


def _fwd(lib, q=FAKE, lse=FAKE, B=1, H=2, N=64, D=64, strides=None, scale=0.125, dtype=2):
    st = strides or (2 * 64 * 64, 64 * 64, 64, 1)
    return lib.fa_fwd(q, FAKE, FAKE, FAKE, lse, B, H, N, D, S(*st), S(*st), S(*st), S(*st),
                      0, scale, dtype, None)


def test_validation_codes(lib):
    assert _fwd(lib, q=None) == 1                       # FA_ERR_NULL
    assert _fwd(lib, lse=None) == 1
    assert _fwd(lib, N=0) == 2                          # FA_ERR_SHAPE
    assert _fwd(lib, B=-1) == 2
    assert _fwd(lib, B=1 << 40, H=1 << 40) == 2         # overflow
    assert _fwd(lib, D=48) == 3                         # FA_ERR_HEADDIM
    assert _fwd(lib, D=256) == 3
    assert _fwd(lib, dtype=7) == 4                      # FA_ERR_DTYPE
    assert _fwd(lib, strides=(8192, 4096, 64, 2)) == 5  # FA_ERR_STRIDE
    assert _fwd(lib, strides=(8192, -4096, 64, 1)) == 5
    assert _fwd(lib, q=FAKE + 2) == 6                   # FA_ERR_ALIGN
    assert _fwd(lib, strides=(8192, 4096, 68, 1), dtype=2) == 6
    assert _fwd(lib, scale=0.0) == 10                   # FA_ERR_SCALE
    assert _fwd(lib, scale=float("nan")) == 10
    assert lib.fa_set_path(5) == 11                     # FA_ERR_ARG


def test_extent_one_dims_ignore_their_stride(lib):
    # B == 1: the b-stride is never used, so an unaligned value passes the
    # alignment check; the invalid scale then stops the call before any device
    # work (a launch with these fake pointers must never happen).
    code = _fwd(lib, B=1, strides=(3, 4096, 64, 1), scale=0.0)
    assert code == 10


def test_valid_call_without_device_reports_launch_or_arch(lib):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a device is present")
    assert _fwd(lib) in (7, 9)


def test_preprocess_and_bwd_validation(lib):
    st = S(64 * 64 * 2, 64 * 64, 64, 1)
    assert lib.fa_bwd_preprocess(FAKE, None, FAKE, 1, 2, 64, 64, st, st, 2, None) == 1
    assert lib.fa_bwd_preprocess(FAKE, FAKE, FAKE, 1, 2, 64, 24, st, st, 2, None) == 3
    bad = S(64 * 64 * 2, 64 * 64, 64, 3)
    assert lib.fa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, FAKE, 1, 2, 64, 64,
                      st, st, st, st, st, st, bad, 1, 0.125, 2, None) == 5
    assert lib.fa_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, None, FAKE, FAKE, FAKE, 1, 2, 64, 64,
                      st, st, st, st, st, st, st, 1, 0.125, 2, None) == 1


def _problem(B=2, Hq=4, Hkv=2, Nq=300, Nk=200, D=64, dtype=2):
    pr = fa.Problem()
    pr.B, pr.Hq, pr.Hkv, pr.Nq, pr.Nk, pr.D = B, Hq, Hkv, Nq, Nk, D
    pr.scale, pr.dtype = 0.125, dtype
    return pr


def test_fused_workspace_size_and_validation(lib):
    """fa_bwd_fused_workspace_bytes: fp32 rows of 64 (D <= 64) or 128 floats
    per query row of every query head; 0 for an invalid problem.  fa_bwd_fused
    rejects fp32 inputs, a NULL / unaligned / short workspace before any
    device work."""
    pr = _problem()
    assert lib.fa_bwd_fused_workspace_bytes(ctypes.byref(pr)) == 2 * 4 * 300 * 64 * 4
    for D, w in ((16, 64), (32, 64), (64, 64), (128, 128)):
        pr = _problem(D=D)
        assert lib.fa_bwd_fused_workspace_bytes(ctypes.byref(pr)) == 2 * 4 * 300 * w * 4
    pr = _problem(Hkv=3)                                  # Hq % Hkv != 0
    assert lib.fa_bwd_fused_workspace_bytes(ctypes.byref(pr)) == 0
    assert lib.fa_bwd_fused_workspace_bytes(None) == 0

    def call(pr, ws=FAKE, nbytes=1 << 30):
        st = S(0, 0, 64, 1)
        return lib.fa_bwd_fused(ctypes.byref(pr), FAKE, st, FAKE, st, FAKE, st, FAKE, st,
                                FAKE, FAKE, FAKE, st, FAKE, st, FAKE, st, ws, nbytes, None)

    assert call(_problem(dtype=0)) == 4                   # FA_ERR_DTYPE: fp32
    assert call(_problem(), ws=None) == 1                 # FA_ERR_NULL
    assert call(_problem(), ws=FAKE + 4) == 6             # FA_ERR_ALIGN
    need = 2 * 4 * 300 * 64 * 4
    assert call(_problem(), nbytes=need - 16) == 12       # FA_ERR_SCRATCH


def test_general_problem_validation_codes(lib):
    """fa_fwd_ex / fa_bwd_ex reject invalid problems before any device work."""
    st = S(0, 300 * 64, 64, 1)        # [1, H, N, D] strides, B = 1

    def fwd(pr, strides=None):
        s4 = strides or st
        return lib.fa_fwd_ex(ctypes.byref(pr) if pr is not None else None, FAKE, s4, FAKE, s4,
                             FAKE, s4, FAKE, s4, FAKE, None)

    def bwd(pr, delta=FAKE):
        return lib.fa_bwd_ex(ctypes.byref(pr), FAKE, st, FAKE, st, FAKE, st, FAKE, st, FAKE,
                             delta, FAKE, st, FAKE, st, FAKE, st, None)

    assert fwd(None) == 1                                        # FA_ERR_NULL
    assert fwd(_problem(B=1, dtype=7)) == 4                      # FA_ERR_DTYPE
    assert fwd(_problem(B=0)) == 2                               # FA_ERR_SHAPE
    assert fwd(_problem(B=1, Hq=4, Hkv=3)) == 2                  # Hq % Hkv
    assert fwd(_problem(B=1, D=48)) == 3                         # FA_ERR_HEADDIM
    pr = _problem(B=1)
    pr.scale = 0.0
    assert fwd(pr) == 10                                         # FA_ERR_SCALE
    for p in (1.0, -0.1, float("nan")):
        pr = _problem(B=1)
        pr.dropout_p = p
        assert fwd(pr) == 11, p                                  # FA_ERR_ARG
    pr = _problem(B=1)
    pr.cu_seqlens_q = FAKE                                        # only one offset array
    assert fwd(pr) == 2
    pr = _problem(B=1)
    pr.cu_seqlens_q = pr.cu_seqlens_k = FAKE
    pr.total_q, pr.total_k = 0, 100                               # packed totals >= 1
    assert fwd(pr) == 2
    pr.total_q = 100
    pr.cu_seqlens_k = FAKE + 2                                    # int32 offsets, 4-byte aligned
    assert fwd(pr) == 6
    pr = _problem(B=1, Nq=(1 << 31) - 1000, Nk=10)                # TMA rows are int32
    assert fwd(pr) == 2
    assert fwd(_problem(B=1), strides=S(0, 300 * 64, 64, 2)) == 5     # FA_ERR_STRIDE
    assert bwd(_problem(B=1), delta=None) == 1


def test_dropout_mask_size_and_validation(lib):
    """fa_dropout_mask_bytes: 16 bytes per (flat head, key tile of 128, query
    row), 0 without dropout or for an invalid problem.  fa_dropout_mask and a
    problem's dropout_mask field are checked before any device work."""
    pr = _problem(B=2, Hq=4, Nq=300, Nk=333)
    assert lib.fa_dropout_mask_bytes(ctypes.byref(pr)) == 0          # dropout_p = 0
    pr.dropout_p = 0.1
    assert lib.fa_dropout_mask_bytes(ctypes.byref(pr)) == 2 * 4 * 3 * 300 * 16
    pr.Nk = 256
    assert lib.fa_dropout_mask_bytes(ctypes.byref(pr)) == 2 * 4 * 2 * 300 * 16
    pk = _problem(B=3, Hq=4, Nq=500, Nk=129)                          # packed: total_q rows
    pk.cu_seqlens_q, pk.cu_seqlens_k, pk.total_q, pk.total_k = FAKE, FAKE, 700, 300
    pk.dropout_p = 0.5
    assert lib.fa_dropout_mask_bytes(ctypes.byref(pk)) == 1 * 4 * 2 * 700 * 16
    bad = _problem(Hkv=3)
    bad.dropout_p = 0.1
    assert lib.fa_dropout_mask_bytes(ctypes.byref(bad)) == 0
    assert lib.fa_dropout_mask_bytes(None) == 0

    need = lib.fa_dropout_mask_bytes(ctypes.byref(pr))
    assert lib.fa_dropout_mask(None, FAKE, need, None) == 1             # FA_ERR_NULL
    assert lib.fa_dropout_mask(ctypes.byref(pr), None, need, None) == 1
    assert lib.fa_dropout_mask(ctypes.byref(pr), FAKE + 8, need, None) == 6   # FA_ERR_ALIGN
    assert lib.fa_dropout_mask(ctypes.byref(pr), FAKE, need - 1, None) == 12  # FA_ERR_SCRATCH
    nodrop = _problem()
    assert lib.fa_dropout_mask(ctypes.byref(nodrop), FAKE, need, None) == 11  # FA_ERR_ARG
    assert lib.fa_dropout_mask(ctypes.byref(bad), FAKE, need, None) == 2      # FA_ERR_SHAPE

    # A misaligned keep-mask pointer in the problem is refused by the passes.
    st = S(0, 0, 64, 1)
    pr.dropout_mask = FAKE + 4
    assert lib.fa_fwd_ex(ctypes.byref(pr), FAKE, st, FAKE, st, FAKE, st, FAKE, st, FAKE,
                         None) == 6
    assert lib.fa_bwd_ex(ctypes.byref(pr), FAKE, st, FAKE, st, FAKE, st, FAKE, st, FAKE, FAKE,
                         FAKE, st, FAKE, st, FAKE, st, None) == 6
