"""An independent reduced-precision attention, used only to size tolerances.

The fp64 oracle gives the exact result; this module gives what an honest
implementation in the kernels' own arithmetic gets: products and sums in IEEE
fp32 (torch CPU matmuls, no TF32), the probabilities P rounded to the input
type before P V and P^T dO, dS rounded to the input type before dS K and
dS^T Q, Delta formed from the stored (rounded) O, and every output rounded to
the input type -- the rounding model the library documents for fp16/bf16
(fp32 inputs: nothing is rounded but the fp32 arithmetic itself).  It is
written from the definitions (S = scale Q K^T, L = logsumexp S, P = exp(S - L),
O = P V, Delta = rowsum(dO o O), dV = P^T dO, dP = dO V^T, dS = P o (dP -
Delta), dQ = scale dS K, dK = scale dS^T Q) with whole N x N matrices per head
and shares nothing with the CUDA kernels or the oracle.

Its error against the oracle is the error a correct computation of that
precision makes on the same inputs; the parity tests for inputs outside the
unit-normal range the tolerances are stated for bound the kernels' error by a
fixed multiple of it.
"""

from __future__ import annotations

import torch

_LOW = {torch.float16, torch.bfloat16}


def emulate_head(q, k, v, do, causal: bool, scale: float):
    """One head: q, k, v, do [N, D] CPU tensors of the input type (do may be
    None: forward only).  Returns a dict of float64 numpy arrays o, lse and,
    with do, delta, dq, dk, dv (outputs rounded to the input type; lse and
    delta fp32)."""
    dt = q.dtype
    low = dt in _LOW

    def rnd(x):
        return x.to(dt).float() if low else x

    qf, kf, vf = (t.float() for t in (q, k, v))
    n, nk = qf.shape[0], kf.shape[0]
    s = (qf @ kf.T) * scale
    if causal:
        keep = torch.ones(n, nk, dtype=torch.bool).tril()
        s = s.masked_fill(~keep, float("-inf"))
    lse = torch.logsumexp(s, dim=1)
    p = torch.exp(s - lse[:, None])
    o = (rnd(p) @ vf).to(dt)
    if do is None:
        return {"o": o.double().numpy(), "lse": lse.double().numpy()}
    dof = do.float()
    delta = (dof * o.float()).sum(dim=1)
    dp = dof @ vf.T
    ds = p * (dp - delta[:, None])
    dv = (rnd(p).T @ dof).to(dt)
    dq = ((rnd(ds) @ kf) * scale).to(dt)
    dk = ((rnd(ds).T @ qf) * scale).to(dt)
    out = dict(o=o, lse=lse, delta=delta, dq=dq, dk=dk, dv=dv)
    return {key: t.double().numpy() for key, t in out.items()}


def emulate(q, k, v, do, causal: bool, scale: float, heads):
    """emulate_head over the listed (b, h) heads of [B, H, N, D] tensors;
    returns {(b, h): dict}."""
    with torch.no_grad():
        return {(b, h): emulate_head(q[b, h], k[b, h], v[b, h],
                                     None if do is None else do[b, h], causal, scale)
                for b, h in heads}
