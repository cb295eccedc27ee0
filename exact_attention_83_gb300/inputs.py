"""Seeded synthetic inputs, shared by the tests, the benchmark and the oracle checks.

This module holds no attention arithmetic: it only draws i.i.d. N(0, 1) values
from a seeded CPU generator, scales them where a workload asks for it, rounds
them to the device dtype, and lays them out.  Both the CUDA path and the fp64
oracle read exactly the tensors returned here (the oracle converts the rounded
values to float64, which is exact).

Recipe (every workload):
  * ``torch.Generator('cpu').manual_seed(seed)``;
  * ``randn`` in float32 in the order Q, K, V, dO;
  * Q, K, V multiplied by ``qkv_scale`` (4 for the shape-coverage workload,
    1 elsewhere; dO is never scaled);
  * rounded to the dtype on the host (round-to-nearest-even, torch's cast);
  * layout ``bhnd`` = contiguous [B, H, N, D], or ``bnhd`` = generated as
    contiguous [B, N, H, D] and returned as the permuted [B, H, N, D] view
    (strides b = N*H*D, h = D, n = H*D, d = 1).
"""

from __future__ import annotations

import dataclasses
import math

import torch

DTYPES = {"fp32": torch.float32, "fp16": torch.float16, "bf16": torch.bfloat16}


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    B: int
    H: int
    N: int
    D: int
    dtype: str
    causal: bool
    layout: str = "bhnd"
    qkv_scale: float = 1.0
    seed: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    def fwd_flops(self) -> float:
        """Algorithmic forward flops: two N x N x D matmuls per head, 2 flops per
        multiply-add, halved when causal."""
        f = 4.0 * self.B * self.H * self.N * self.N * self.D
        return f / 2 if self.causal else f

    def fwd_bwd_flops(self) -> float:
        """Forward plus backward, the backward credited at 2.5x the forward."""
        return 3.5 * self.fwd_flops()


def make_inputs(w: Workload, device="cpu", with_grad_out: bool = True):
    """Return (q, k, v, do) for workload ``w`` on ``device`` (do is None when
    with_grad_out is False).  Generation always happens on the CPU."""
    g = torch.Generator("cpu")
    g.manual_seed(w.seed)
    if w.layout == "bhnd":
        shape = (w.B, w.H, w.N, w.D)
    elif w.layout == "bnhd":
        shape = (w.B, w.N, w.H, w.D)
    else:
        raise ValueError(w.layout)
    dt = DTYPES[w.dtype]
    out = []
    names = ("q", "k", "v", "do") if with_grad_out else ("q", "k", "v")
    for name in names:
        x = torch.randn(shape, generator=g, dtype=torch.float32)
        if name != "do" and w.qkv_scale != 1.0:
            x = x * w.qkv_scale
        x = x.to(dt)
        if device != "cpu":
            x = x.to(device)
        if w.layout == "bnhd":
            x = x.permute(0, 2, 1, 3)
        out.append(x)
    if not with_grad_out:
        out.append(None)
    return tuple(out)


# The workloads the tests and the benchmark run.
TINY_FP32 = Workload("tiny-fp32-B1-H2-N128-D64", 1, 2, 128, 64, "fp32", False)


def bf16_n1024(causal: bool) -> Workload:
    return Workload(f"bf16-B4-H16-N1024-D64-{'causal' if causal else 'full'}",
                    4, 16, 1024, 64, "bf16", causal)


SWEEP_N = (512, 1024, 2048, 4096, 8192, 16384)


def sweep(N: int, dtype: str, causal: bool) -> Workload:
    """Sequence-length sweep: D=64, H=16, B*H*N = 262144."""
    B = 262144 // (16 * N)
    return Workload(f"sweep-{dtype}-B{B}-H16-N{N}-D64-{'causal' if causal else 'full'}",
                    B, 16, N, 64, dtype, causal)


def coverage(D: int, N: int, dtype: str, causal: bool) -> Workload:
    """Shape coverage: B=2, H=8, ragged N, permuted [B,N,H,D] storage, inputs x4."""
    return Workload(f"coverage-{dtype}-B2-H8-N{N}-D{D}-{'causal' if causal else 'full'}-bnhd-x4",
                    2, 8, N, D, dtype, causal, layout="bnhd", qkv_scale=4.0)


LONG_CAUSAL = Workload("long-bf16-B1-H32-N16384-D128-causal", 1, 32, 16384, 128,
                       "bf16", True)
