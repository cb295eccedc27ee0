"""Shared helpers of the GPU tests for general problems (fa_fwd_ex /
fa_bwd_ex / fa_bwd_fused): running a GeneralWorkload through the C ABI, the
oracle reference and the comparison with its tolerance, the page's test
shapes and the seeded random problem generator."""

from __future__ import annotations

import numpy as np
import torch

import oracle
from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import GeneralWorkload, make_general_inputs
from parity import TOL, UNIT_ROUNDOFF, check

DEV = torch.device("cuda", 0)


def _kw(w: GeneralWorkload, cu_q, cu_k):
    kw = dict(dropout_p=w.dropout_p, seed=w.drop_seed, offset=w.drop_offset)
    if w.packed:
        kw.update(cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=w.Nq, max_seqlen_k=w.Nk)
    return kw


def run_general(w: GeneralWorkload, fused: bool = False, keep_mask: bool = False):
    """Forward, preprocess and backward (fa_bwd_ex, or fa_bwd_fused when
    `fused`) through the C ABI; outputs start as NaN so any element left
    unwritten fails the comparison.  keep_mask: the forward stores its
    dropout decisions in a keep-mask buffer (which starts as 0xA5 bytes) that
    the backward reads."""
    q, k, v, do, cu_q, cu_k = make_general_inputs(w)
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
    fa.fwd_ex(qd, kd, vd, o, lse, w.causal, w.scale, **kw)
    delta = torch.full(lse_shape, float("nan"), dtype=torch.float32, device=DEV)
    fa.bwd_preprocess(fa._as4(o, w.packed), fa._as4(dod, w.packed), delta)
    dq = torch.full_like(qd, float("nan"))
    dk = torch.full_like(kd, float("nan"))
    dv = torch.full_like(vd, float("nan"))
    if fused:
        nbytes = fa.workspace_bytes(qd, kd, w.causal, w.scale, **kw)
        ws = torch.full((nbytes // 4,), float("nan"), dtype=torch.float32, device=DEV)
        fa.bwd_fused(qd, kd, vd, dod, lse, delta, dq, dk, dv, w.causal, w.scale, workspace=ws,
                     **kw)
    else:
        fa.bwd_ex(qd, kd, vd, dod, lse, delta, dq, dk, dv, w.causal, w.scale, **kw)
    torch.cuda.synchronize()
    status = fa.device_status()
    assert status == 0, fa.STATUS_NAMES.get(status, status)
    got = {n: t.float().cpu().double().numpy() for n, t in
           dict(o=o, lse=lse, delta=delta, dq=dq, dk=dk, dv=dv).items()}
    return (q, k, v, do, cu_q, cu_k), got


def reference(w: GeneralWorkload, inputs, magnitudes: bool = False):
    q, k, v, do, cu_q, cu_k = inputs
    if w.packed:
        return oracle.varlen_fwd_bwd(q, k, v, do, cu_q.numpy(), cu_k.numpy(), w.causal, w.scale,
                                     p=w.dropout_p, seed=w.drop_seed, offset=w.drop_offset,
                                     magnitudes_too=magnitudes)
    dr = oracle.dropout_params(w.dropout_p, w.drop_seed, w.drop_offset)
    ref = oracle.fwd_bwd(q, k, v, do, w.causal, w.scale, dr)
    if magnitudes:
        m = oracle.magnitudes(q, k, v, do, w.causal, w.scale, dr)
        ref.update({key + "_abs": val for key, val in m.items()})
    return ref


def compare(w: GeneralWorkload, inputs, got):
    """Max-abs tolerance of the unit-normal workloads, plus the final rounding
    of each output to the input type (half an ulp: u * |ref|).  A sum over many
    rows (e.g. dV of a key that every query attends to with weight 1) grows
    past 1, where that rounding alone exceeds the absolute term.  For fp16 and
    bf16 each element also gets u * m, m the oracle's magnitude sum of the
    terms of its product (the componentwise bound for rounding P or dS to the
    input type before the product): a key attended by hundreds of
    (query, head) pairs, as with multi-query heads, sums that many rounded
    terms."""
    u = UNIT_ROUNDOFF.get(w.dtype, 0.0)
    ref = reference(w, inputs, magnitudes=u > 0)
    for key in ("o", "lse", "dq", "dk", "dv"):
        g, r = got[key], ref[key]
        if key == "lse":
            # rows with no key at all: L = -inf on both sides; L is fp32
            inf = np.isneginf(r)
            assert (np.isneginf(g) == inf).all(), f"{w.name}: lse -inf pattern"
            g, r = np.where(inf, 0.0, g), np.where(inf, 0.0, r)
            check(f"{w.name}:{key}", g, r, TOL[w.dtype])
            continue
        atol = TOL[w.dtype] + u * ref[key + "_abs"] if u > 0 else TOL[w.dtype]
        check(f"{w.name}:{key}", g, r, (atol, u))


# The Triton page's test shapes (batch, n_queries, n_keys, head_dim), two heads.
PAGE_SHAPES = [(4, 128, 128, 64), (2, 1024, 1024, 64), (2, 100, 100, 64), (1, 37, 53, 32),
               (1, 200, 96, 128)]


def random_general(seed: int) -> GeneralWorkload:
    """A seeded random general problem: any combination of grouped heads,
    packed or fixed lengths (empty sequences included), Nq != Nk, causal,
    dropout, head dimension and dtype, at sizes the oracle runs in well under a
    second."""
    r = np.random.default_rng(seed)
    D = int(r.choice([16, 32, 64, 128]))
    dtype = str(r.choice(["bf16", "fp16", "fp32"]))
    Hkv = int(r.choice([1, 2]))
    Hq = Hkv * int(r.choice([1, 2, 4]))
    B = int(r.integers(1, 4))
    causal = bool(r.integers(0, 2))
    p = float(r.choice([0.0, 0.0, 0.25]))
    if r.integers(0, 2):
        lq = tuple(int(x) for x in r.integers(0, 300, size=B))
        lk = tuple(int(x) for x in r.integers(0, 300, size=B))
        if sum(lq) == 0:
            lq = (1,) + lq[1:]
        if sum(lk) == 0:
            lk = (1,) + lk[1:]
        return GeneralWorkload(f"fuzz{seed}", B, Hq, Hkv, max(max(lq), 1), max(max(lk), 1), D,
                               dtype, causal, seqlens_q=lq, seqlens_k=lk, dropout_p=p,
                               seed=seed, drop_seed=seed * 7919, drop_offset=seed)
    Nq, Nk = int(r.integers(1, 400)), int(r.integers(1, 400))
    return GeneralWorkload(f"fuzz{seed}", B, Hq, Hkv, Nq, Nk, D, dtype, causal, dropout_p=p,
                           seed=seed, drop_seed=seed * 7919, drop_offset=seed)
