"""The reduced-precision emulation that sizes the bound of the inputs scaled by
4 (tests/emulate.py), checked on the CPU.

  * At unit-normal inputs it meets the spec's own tolerances against the
    oracle: it is a correct computation, not a loose one.
  * At inputs scaled by 4 its error is far below the values: the derived
    bound max(tol, 4 * e_ind) stays below 1e-4 of the largest value in fp32
    and within four times a few bf16 roundings of it in bf16.
  * Mistakes a kernel could plausibly make (a dropped scale, an off-by-one
    causal mask, Delta of the wrong row, P not rounded where the model rounds
    it before a product, a transposed operand) exceed that bound.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

import oracle
from emulate import emulate_head
from exact_attention_83_gb300.inputs import Workload, make_inputs
from parity import C_EMU, TOL

KEYS = ("o", "lse", "delta", "dq", "dk", "dv")


def _ref(w, q, k, v, do):
    r = oracle.fwd_bwd(q[:1, :1], k[:1, :1], v[:1, :1], do[:1, :1], w.causal, w.scale)
    return {key: r[key][0, 0] for key in KEYS}


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp32", "bf16", "fp16"])
def test_emulation_meets_the_spec_tolerance_at_unit_normal_inputs(dtype, causal):
    w = Workload(f"emu-{dtype}", 1, 1, 300, 64, dtype, causal, seed=5)
    q, k, v, do = make_inputs(w)
    ref = _ref(w, q, k, v, do)
    e = emulate_head(q[0, 0], k[0, 0], v[0, 0], do[0, 0], causal, w.scale)
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert np.abs(e[key] - ref[key]).max() <= TOL[dtype], key


def _x4(dtype, causal, N=257, D=64):
    w = Workload(f"emu-x4-{dtype}", 1, 1, N, D, dtype, causal, layout="bnhd", qkv_scale=4.0,
                 seed=9)
    q, k, v, do = make_inputs(w)
    return w, (q[0, 0], k[0, 0], v[0, 0], do[0, 0]), _ref(w, q, k, v, do)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
def test_derived_bound_is_small_against_the_values(dtype, causal):
    w, (q, k, v, do), ref = _x4(dtype, causal)
    e = emulate_head(q, k, v, do, causal, w.scale)
    for key in KEYS:
        bound = max(TOL[dtype], C_EMU * np.abs(e[key] - ref[key]).max())
        peak = float(np.abs(ref[key]).max())
        # fp32: below the spec's fp32 tolerance relative to the largest value;
        # bf16: C_EMU times a few roundings (u = 2^-8) of the largest value
        limit = TOL["fp32"] * peak if dtype == "fp32" else C_EMU * 4 * 2.0 ** -8 * peak
        assert bound <= limit, (key, bound, peak)


def _planted(q, k, v, do, causal, scale, mistake):
    """A fp32 computation with one deliberate mistake (P and dS rounded to the
    input type as the library does, so only the planted mistake differs)."""
    dt = q.dtype
    low = dt != torch.float32
    rnd = (lambda x: x.to(dt).float()) if low else (lambda x: x)
    qf, kf, vf, dof = (t.float() for t in (q, k, v, do))
    n = qf.shape[0]
    s = (qf @ kf.T) * scale
    if causal:
        diag = 1 if mistake == "causal_off_by_one" else 0
        keep = torch.ones(n, n, dtype=torch.bool).tril(diagonal=diag)
        s = s.masked_fill(~keep, float("-inf"))
    lse = torch.logsumexp(s, dim=1)
    p = torch.exp(s - lse[:, None])
    pv = p if mistake == "p_unrounded_then_v_transposed" else rnd(p)
    vv = vf.flip(0) if mistake == "p_unrounded_then_v_transposed" else vf
    o = (pv @ vv).to(dt)
    delta = (dof * o.float()).sum(dim=1)
    if mistake == "delta_wrong_row":
        delta = delta.roll(1)
    dp = dof @ vf.T
    ds = p * (dp - delta[:, None])
    dv = (rnd(p).T @ dof).to(dt)
    dq = ((rnd(ds) @ kf) * scale).to(dt)
    dk_scale = 1.0 if mistake == "dk_unscaled" else scale
    dk = ((rnd(ds).T @ qf) * dk_scale).to(dt)
    out = dict(o=o, lse=lse, delta=delta, dq=dq, dk=dk, dv=dv)
    return {key: t.double().numpy() for key, t in out.items()}


@pytest.mark.parametrize("dtype", ["fp32", "bf16"])
@pytest.mark.parametrize("mistake,key", [("causal_off_by_one", "o"),
                                         ("causal_off_by_one", "dk"),
                                         ("delta_wrong_row", "dq"),
                                         ("dk_unscaled", "dk"),
                                         ("p_unrounded_then_v_transposed", "o")])
def test_derived_bound_rejects_planted_mistakes(dtype, mistake, key):
    causal = mistake == "causal_off_by_one"
    w, (q, k, v, do), ref = _x4(dtype, causal)
    e = emulate_head(q, k, v, do, causal, w.scale)
    bound = max(TOL[dtype], C_EMU * np.abs(e[key] - ref[key]).max())
    bad = _planted(q, k, v, do, causal, w.scale, mistake)
    assert np.abs(bad[key] - ref[key]).max() > 3 * bound, (mistake, key)
