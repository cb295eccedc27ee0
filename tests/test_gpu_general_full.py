"""General problems at the size the benchmark times them, split and single-pass
backward, against the oracle on sampled rows.

Grouped (Hq 32 / Hkv 8) and multi-query (Hkv 1) heads, dropout p = 0.1
(decisions drawn again by the backward, and read by it from the keep mask
the forward stored: bitwise the same),
65536 packed tokens in sequences of 512-8192 rows, and Nq 4096 / Nk 16384
cross lengths, all D = 128 bf16 with 32 query heads: exactly the inputs and
launch configuration of `bench.py --workload <name>`.  The oracle computes
sampled query rows (O, L, dQ: tile edges, sequence ends and random rows of
three query heads) and sampled key rows (dK, dV of one key/value head, which
needs every query head of its group) one by one; packed sequences are checked
per sequence on the longest and the shortest one.  Tolerance: that of the
general workloads (tests/general.py): the unit-normal max-abs term, plus the
final rounding of each output to bf16 (u |ref|), plus u times the oracle's
magnitude sum of the element's product terms.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import BENCH_GENERAL, Workload, make_general_inputs
from general import DEV, _kw
from parity import TOL, UNIT_ROUNDOFF, check, sample_rows

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.set_path(fa.FA_PATH_AUTO)
    yield


def _run(w, inputs, fused, keep_mask=False):
    q, k, v, do, cu_q, cu_k = inputs
    qd, kd, vd, dod = (t.to(DEV) for t in (q, k, v, do))
    cq = cu_q.to(DEV) if cu_q is not None else None
    ck = cu_k.to(DEV) if cu_k is not None else None
    kw = _kw(w, cq, ck)
    if keep_mask:
        kw["dropout_mask"] = torch.full((fa.dropout_mask_bytes(qd, kd, w.causal, w.scale, **kw),),
                                        0xA5, dtype=torch.uint8, device=DEV)
    o = torch.full_like(qd, float("nan"))
    lse_shape = (w.Hq, q.shape[0]) if w.packed else (w.B, w.Hq, w.Nq)
    lse = torch.full(lse_shape, float("nan"), dtype=torch.float32, device=DEV)
    delta = torch.full_like(lse, float("nan"))
    dq = torch.full_like(qd, float("nan"))
    dk, dv = torch.full_like(kd, float("nan")), torch.full_like(vd, float("nan"))
    fa.fwd_ex(qd, kd, vd, o, lse, w.causal, w.scale, **kw)
    fa.bwd_preprocess(fa._as4(o, w.packed), fa._as4(dod, w.packed), delta)
    if fused:
        ws = torch.empty(fa.workspace_bytes(qd, kd, w.causal, w.scale, **kw) // 4,
                         dtype=torch.float32, device=DEV)
        fa.bwd_fused(qd, kd, vd, dod, lse, delta, dq, dk, dv, w.causal, w.scale, workspace=ws,
                     **kw)
    else:
        fa.bwd_ex(qd, kd, vd, dod, lse, delta, dq, dk, dv, w.causal, w.scale, **kw)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    out = dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)
    return {key: t.float().cpu() for key, t in out.items()}


def _tol(w, key, ref_abs=None):
    u = UNIT_ROUNDOFF[w.dtype]
    if key == "lse":
        return TOL[w.dtype]
    return (TOL[w.dtype] + u * ref_abs, u)


def _refs(w, q, k, v, do, bh_base=0):
    """Oracle values of sampled rows of a fixed-length problem
    [B, Hq, Nq, D] / [B, Hkv, Nk, D]: (query rows, their O/L/dQ, key rows,
    their dK/dV), magnitude sums included."""
    B, Hq, Nq = q.shape[0], q.shape[1], q.shape[2]
    Hkv, Nk = k.shape[1], k.shape[2]
    dr = oracle.dropout_params(w.dropout_p, w.drop_seed, w.drop_offset, bh0=bh_base)
    qw = Workload(w.name, B, Hq, Nq, w.D, w.dtype, w.causal)
    qheads = sorted({(0, 0), (B - 1, Hq - 1), (B // 2, Hq // 2)})
    qrows = sample_rows(qw, qheads, n_random=6)
    qref = oracle.query_rows(q, k, v, do, w.causal, qrows, w.scale, magnitudes=True, dropout=dr)
    kw_ = Workload(w.name, B, Hkv, Nk, w.D, w.dtype, w.causal)
    krows = sample_rows(kw_, [(B - 1, Hkv - 1)], n_random=6, seed=2)
    kref = oracle.key_rows(q, k, v, do, w.causal, krows, w.scale, magnitudes=True, dropout=dr)
    return (Hq, qrows, qref), (Hkv, krows, kref)


def _compare(w, got, refs, name):
    """got: CPU float tensors [B, Hq, Nq, D] (o, dq), [B, Hq, Nq] (lse),
    [B, Hkv, Nk, D] (dk, dv)."""
    (Hq, qrows, qref), (Hkv, krows, kref) = refs
    b, h, i = qrows[:, 0] // Hq, qrows[:, 0] % Hq, qrows[:, 1]
    for key in ("o", "lse", "dq"):
        g = got[key][b, h, i].double().numpy()
        check(f"{name}:{key}", g, qref[key], _tol(w, key, qref.get(key + "_abs")))
    b, h, j = krows[:, 0] // Hkv, krows[:, 0] % Hkv, krows[:, 1]
    for key in ("dk", "dv"):
        g = got[key][b, h, j].double().numpy()
        check(f"{name}:{key}", g, kref[key], _tol(w, key, kref[key + "_abs"]))


def _seq(t, c0, c1):
    """Rows c0..c1-1 of a packed [total, H, D] tensor as [1, H, n, D]."""
    return t[c0:c1].permute(1, 0, 2).unsqueeze(0)


@pytest.mark.parametrize("w", BENCH_GENERAL, ids=[w.name for w in BENCH_GENERAL])
def test_general_workload_at_bench_size(w):
    inputs = make_general_inputs(w)
    q, k, v, do, cu_q, cu_k = inputs
    runs = {name: _run(w, inputs, fused)
            for name, fused in ((w.name, False), (w.name + "-single-pass", True))}
    if w.dropout_p > 0:
        # the benchmark's dropout step: the forward stores its decisions in
        # the keep mask, the backward reads them; bitwise the same as drawing
        # them again
        read = _run(w, inputs, False, keep_mask=True)
        for key in ("o", "lse", "dq", "dk", "dv"):
            assert torch.equal(read[key], runs[w.name][key]), key
    if not w.packed:
        refs = _refs(w, q, k, v, do)
        for name, got in runs.items():
            _compare(w, got, refs, name)
        return
    lens = np.diff(cu_q.numpy())
    for s in sorted({int(np.argmax(lens)), int(np.argmin(lens))}):
        a0, a1 = int(cu_q[s]), int(cu_q[s + 1])
        k0, k1 = int(cu_k[s]), int(cu_k[s + 1])
        refs = _refs(w, _seq(q, a0, a1), _seq(k, k0, k1), _seq(v, k0, k1), _seq(do, a0, a1),
                     bh_base=s * w.Hq)
        for name, got in runs.items():
            sub = {"o": _seq(got["o"], a0, a1), "dq": _seq(got["dq"], a0, a1),
                   "dk": _seq(got["dk"], k0, k1), "dv": _seq(got["dv"], k0, k1),
                   "lse": got["lse"][:, a0:a1].unsqueeze(0)}
            _compare(w, sub, refs, f"{name}-seq{s}")
