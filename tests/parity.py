"""Helpers for the GPU parity tests: run the CUDA path through the C ABI on
seeded inputs and compare with the fp64 oracle.

Tolerances (stated in the attention spec this library follows): max-abs error
1e-4 for fp32 and 2e-2 for fp16/bf16, for O, L, dQ, dK and dV at unit-normal
inputs.

For inputs scaled by 4 the spec states no tolerance; it is derived here.
Every intermediate grows with the inputs: raw scores q.k reach ~16*sqrt(D)
standard deviations (exponents ~80 in log2 units), O grows to ~4 and dQ, dK
to tens.  A correct implementation's absolute error then scales with the
largest magnitudes, not with the RMS:
  * fp32: the fp32 dot products behind S carry ~1e-7 * |q||k| * sqrt(D) of
    rounding, i.e. a relative error of ~1e-4 in P, which multiplies
    dP - Delta (~|dO||V| sqrt(D));
  * fp16/bf16: Delta = rowsum(dO o O) is formed from the stored O (as in
    FlashAttention-2), whose rounding (|O| * 2^-9 for bf16) enters every
    dS_ij = P_ij (dP_ij - Delta_i).
Measured on the FFMA kernels, these give max errors of 2-10x the spec
tolerance times RMS(ref).  The bound used for these cases is therefore
    max |got - ref| <= tol * max(1, max |ref|)      per tensor,
which still fails on any structural mistake (those give errors of the order
of max |ref| itself).

The 16-bit tensor-core kernels also round P (before P V) and dS (before
dS K and dS^T Q) to the input type, as FlashAttention-2 does for its second
GEMM of each pair.  A sum of products with one factor rounded to relative
precision u is off by at most u times the sum of the products' magnitudes
(the standard componentwise bound), so for x4 inputs in fp16/bf16 each
element of O, dQ, dK, dV gets, on top of the per-tensor term above,
    u * (sum P|V|, scale sum |dS||K|, scale sum |dS||Q|, sum P|dO|)
with u = 2^-8 (bf16) or 2^-11 (fp16), the sums computed by the oracle.  At
unit-normal inputs the spec's tolerance is used as stated.
"""

from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import Workload, make_inputs, make_inputs_device

TOL = {"fp32": 1e-4, "fp16": 2e-2, "bf16": 2e-2}
UNIT_ROUNDOFF = {"fp16": 2.0 ** -11, "bf16": 2.0 ** -8}
KEYS = ("o", "lse", "dq", "dk", "dv")
MAG_KEYS = ("o", "dq", "dk", "dv")


def wants_magnitudes(w: Workload) -> bool:
    return w.qkv_scale != 1.0 and w.dtype in UNIT_ROUNDOFF


def tolerance(w: Workload, key: str, ref: np.ndarray, mag: np.ndarray | None = None):
    """(atol, rtol) for tensor `key` of workload `w`; atol is an array when
    the componentwise term applies (mag: the oracle's magnitude sums)."""
    t = TOL[w.dtype]
    if w.qkv_scale == 1.0:
        return t, 0.0
    peak = float(np.abs(ref).max()) if ref.size else 0.0
    atol = t * max(1.0, peak)
    if mag is not None and wants_magnitudes(w):
        atol = atol + UNIT_ROUNDOFF[w.dtype] * mag
    return atol, 0.0


def run_gpu(w: Workload, inputs=None, backward: bool = True, fused: bool = False):
    """Runs fa_fwd (+ fa_bwd_preprocess + fa_bwd, or fa_bwd_fused when `fused`)
    on cuda:0 with NaN-filled outputs; returns (inputs on CPU, dict of CPU
    float64 numpy outputs)."""
    if inputs is None:
        inputs = make_inputs(w, "cpu", with_grad_out=backward)
    q, k, v, do = inputs
    dev = torch.device("cuda", 0)

    def to_dev(x):
        # keep the generated storage order: permute back to storage, copy, re-permute
        if w.layout == "bnhd":
            return x.permute(0, 2, 1, 3).contiguous().to(dev).permute(0, 2, 1, 3)
        return x.contiguous().to(dev)

    qd, kd, vd = to_dev(q), to_dev(k), to_dev(v)
    B, H, N, D = w.B, w.H, w.N, w.D
    dt = qd.dtype
    o = torch.full((B, H, N, D), float("nan"), dtype=dt, device=dev)
    lse = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
    fa.fwd(qd, kd, vd, o, lse, w.causal, w.scale)
    out = {"o": o, "lse": lse}
    if backward:
        dod = to_dev(do)
        delta = torch.full((B, H, N), float("nan"), dtype=torch.float32, device=dev)
        fa.bwd_preprocess(o, dod, delta)
        dq = torch.full((B, H, N, D), float("nan"), dtype=dt, device=dev)
        dk = torch.full_like(dq, float("nan"))
        dv = torch.full_like(dq, float("nan"))
        if fused:
            nbytes = fa.workspace_bytes(qd, kd, w.causal, w.scale)
            ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device=dev)
            fa.bwd_fused(qd, kd, vd, dod, lse, delta, dq, dk, dv, w.causal, w.scale,
                         workspace=ws)
        else:
            fa.bwd(qd, kd, vd, dod, lse, delta, dq, dk, dv, w.causal, w.scale)
        out.update(delta=delta, dq=dq, dk=dk, dv=dv)
    torch.cuda.synchronize()
    status = fa.device_status()
    assert status == 0, f"device status {fa.STATUS_NAMES.get(status, status)}"
    return inputs, {k_: t.float().cpu().double().numpy() for k_, t in out.items()}


def check(name: str, got: np.ndarray, ref: np.ndarray, tol):
    """Per element |got - ref| <= atol + rtol * |ref|; returns the max abs error."""
    atol, rtol = tol if isinstance(tol, tuple) else (tol, 0.0)
    assert got.shape == ref.shape, (name, got.shape, ref.shape)
    assert np.isfinite(got).all(), f"{name}: non-finite values (unwritten output?)"
    if not ref.size:
        return 0.0
    diff = np.abs(got - ref)
    allow = atol + rtol * np.abs(ref)
    err = float(diff.max())
    over = diff - allow
    worst = np.unravel_index(int(np.argmax(over)), over.shape)
    assert over[worst] <= 0, (f"{name}: max abs error {err:.3e}; at {worst} error "
                              f"{diff[worst]:.3e} > allowance {np.broadcast_to(allow, diff.shape)[worst]:.3e}")
    return err


def compare_full(w: Workload, inputs, got, heads=None):
    """Compare every element of the selected heads (list of (b, h); all heads
    when None) with the oracle run on those heads alone."""
    q, k, v, do = inputs
    if heads is None:
        sel = (slice(None), slice(None))
        ref = oracle.fwd_bwd(q, k, v, do, w.causal, w.scale) if do is not None else None
        if ref is not None and wants_magnitudes(w):
            m = oracle.magnitudes(q, k, v, do, w.causal, w.scale)
            ref.update({key + "_abs": m[key] for key in MAG_KEYS})
        if ref is None:
            o, L = oracle.fwd(q, k, v, w.causal, w.scale)
            ref = {"o": o, "lse": L}
        pairs = [(ref, sel)]
    else:
        pairs = []
        for b, h in heads:
            sl = (slice(b, b + 1), slice(h, h + 1))
            qs, ks, vs = q[sl], k[sl], v[sl]
            if do is not None:
                r = oracle.fwd_bwd(qs, ks, vs, do[sl], w.causal, w.scale)
                if wants_magnitudes(w):
                    m = oracle.magnitudes(qs, ks, vs, do[sl], w.causal, w.scale)
                    r.update({key + "_abs": m[key] for key in MAG_KEYS})
            else:
                o, L = oracle.fwd(qs, ks, vs, w.causal, w.scale)
                r = {"o": o, "lse": L}
            pairs.append((r, sl))
    errs = {}
    for ref, sl in pairs:
        for key in KEYS + ("delta",):
            if key not in ref or key not in got:
                continue
            g = got[key][sl]
            tol = tolerance(w, key, ref[key], ref.get(key + "_abs"))
            if key == "delta":
                # Delta is a D-term sum of dO * O, O read back in the input type
                atol_o, r_o = tolerance(w, "o", ref["o"])
                tol = (atol_o * max(1.0, float(np.abs(ref[key]).max())), r_o)
            errs[key] = max(errs.get(key, 0.0), check(f"{w.name}:{key}", g, ref[key], tol))
    return errs


def sample_rows(w: Workload, heads, n_random: int = 8, seed: int = 1):
    """(b*H+h, i) pairs: tile edges, the ends of the sequence and random rows."""
    N = w.N
    fixed = {0, 1, 63, 64, 65, 127, 128, 129, 255, 256, N // 2, N - 129, N - 128,
             N - 65, N - 2, N - 1}
    fixed = sorted(i for i in fixed if 0 <= i < N)
    rng = np.random.default_rng(seed)
    rows = []
    for b, h in heads:
        bh = b * w.H + h
        idx = fixed + list(rng.integers(0, N, size=n_random))
        rows += [(bh, int(i)) for i in idx]
    return np.array(rows, dtype=np.int64)


def compare_sampled(w: Workload, inputs, got, q_heads, k_heads):
    """Sampled query rows (O, L, Delta, dQ) over q_heads and sampled key rows
    (dK, dV) over k_heads, against the oracle's row entry points."""
    q, k, v, do = inputs
    errs = {}
    qrows = sample_rows(w, q_heads)
    mags = wants_magnitudes(w)
    ref = oracle.query_rows(q, k, v, do, w.causal, qrows, w.scale, magnitudes=mags)
    bh, i = qrows[:, 0], qrows[:, 1]
    b, h = bh // w.H, bh % w.H
    for key in ("o", "lse", "dq"):
        g = got[key][b, h, i]
        tol = tolerance(w, key, ref[key], ref.get(key + "_abs"))
        errs[key] = check(f"{w.name}:{key}", g, ref[key], tol)
    krows = sample_rows(w, k_heads, seed=2)
    ref = oracle.key_rows(q, k, v, do, w.causal, krows, w.scale, magnitudes=mags)
    bh, j = krows[:, 0], krows[:, 1]
    b, h = bh // w.H, bh % w.H
    for key in ("dk", "dv"):
        g = got[key][b, h, j]
        tol = tolerance(w, key, ref[key], ref.get(key + "_abs"))
        errs[key] = check(f"{w.name}:{key}", g, ref[key], tol)
    return errs


def run_huge(w, fused: bool):
    """Forward and backward of a workload whose tensors hold more than 2^31
    elements, inputs generated on the device; returns the device tensors."""
    dev = torch.device("cuda", 0)
    q, k, v, do = make_inputs_device(w, dev)
    o = torch.full_like(q, float("nan"))
    lse = torch.full((w.B, w.H, w.N), float("nan"), dtype=torch.float32, device=dev)
    delta = torch.full_like(lse, float("nan"))
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    fa.fwd(q, k, v, o, lse, w.causal, w.scale)
    fa.bwd_preprocess(o, do, delta)
    if fused:
        ws = torch.empty(fa.workspace_bytes(q, k, w.causal, w.scale) // 4, dtype=torch.float32,
                         device=dev)
        fa.bwd_fused(q, k, v, do, lse, delta, dq, dk, dv, w.causal, w.scale, workspace=ws)
        del ws
    else:
        fa.bwd(q, k, v, do, lse, delta, dq, dk, dv, w.causal, w.scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    return (q, k, v, do), dict(o=o, lse=lse, dq=dq, dk=dk, dv=dv)


def check_huge_heads(w, inputs, out, heads):
    """Sampled rows of the given heads against the oracle, one head at a time
    (the head's inputs copied to the host)."""
    one = Workload(w.name + "-head", 1, 1, w.N, w.D, w.dtype, w.causal, seed=w.seed)
    for b, h in heads:
        sub = tuple(t[b:b + 1, h:h + 1].cpu() for t in inputs)
        got = {key: t[b:b + 1, h:h + 1].float().cpu().double().numpy() for key, t in out.items()}
        compare_sampled(one, sub, got, q_heads=[(0, 0)], k_heads=[(0, 0)])


# B=1, H=256, N=65793 (a ragged tail), D=128: 2.16e9 elements per tensor, so
# element offsets pass 2^31 in the last heads; ~35 GB on the device.
HUGE = Workload("huge-bf16-B1-H256-N65793-D128-causal", 1, 256, 65793, 128, "bf16", True, seed=3)
