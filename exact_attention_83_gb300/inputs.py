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
import itertools
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


def make_inputs_device(w: Workload, device):
    """(q, k, v, do) for workload ``w`` generated on ``device`` by torch's
    seeded CUDA generator (i.i.d. N(0,1) in fp32, then cast): for sizes whose
    host generation would take minutes.  Callers compare against the oracle on
    slices copied back to the host, so both sides see the same values."""
    if w.layout != "bhnd":
        raise ValueError("device generation takes [B, H, N, D] workloads")
    g = torch.Generator(device)
    g.manual_seed(w.seed)
    dt = DTYPES[w.dtype]
    out = []
    for name in ("q", "k", "v", "do"):
        x = torch.randn((w.B, w.H, w.N, w.D), generator=g, dtype=torch.float32, device=device)
        if name != "do" and w.qkv_scale != 1.0:
            x.mul_(w.qkv_scale)
        out.append(x.to(dt))
        del x
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


# ---------------------------------------------------------------- general problems
@dataclasses.dataclass(frozen=True)
class GeneralWorkload:
    """Query and key lengths that differ, grouped key/value heads, packed
    variable lengths (seqlens_q / seqlens_k set) and dropout of the weights.
    Fixed lengths: q, do [B, Hq, Nq, D], k, v [B, Hkv, Nk, D].  Packed:
    q, do [sum(seqlens_q), Hq, D], k, v [sum(seqlens_k), Hkv, D]; B is the
    number of sequences, Nq / Nk their maxima."""
    name: str
    B: int
    Hq: int
    Hkv: int
    Nq: int
    Nk: int
    D: int
    dtype: str
    causal: bool
    seqlens_q: tuple | None = None
    seqlens_k: tuple | None = None
    dropout_p: float = 0.0
    seed: int = 0
    drop_seed: int = 0x5EED
    drop_offset: int = 0

    @property
    def scale(self) -> float:
        return 1.0 / math.sqrt(self.D)

    @property
    def packed(self) -> bool:
        return self.seqlens_q is not None

    def pairs(self) -> int:
        """(query, key) pairs attended per query head: sum over sequences of
        Nq*Nk, or of sum_i min(i + 1, Nk) when causal (top-left mask)."""
        lens = (list(zip(self.seqlens_q, self.seqlens_k)) if self.packed
                else [(self.Nq, self.Nk)] * self.B)
        tot = 0
        for nq, nk in lens:
            if not self.causal:
                tot += nq * nk
            else:
                m = min(nq, nk)          # rows 0..m-1 see i+1 keys, the rest all nk
                tot += m * (m + 1) // 2 + (nq - m) * nk
        return tot

    def fwd_flops(self) -> float:
        """Two matmuls over the attended pairs, 2 flops per multiply-add."""
        return 4.0 * self.Hq * self.D * self.pairs()

    def fwd_bwd_flops(self) -> float:
        return 3.5 * self.fwd_flops()


def make_general_inputs(w: GeneralWorkload, device="cpu"):
    """(q, k, v, do, cu_q, cu_k): randn in float32 in the order Q, K, V, dO from
    the seeded CPU generator, rounded to the dtype; cu_* are int32 offsets
    (None for fixed lengths)."""
    g = torch.Generator("cpu")
    g.manual_seed(w.seed)
    dt = DTYPES[w.dtype]
    if w.packed:
        tq, tk = sum(w.seqlens_q), sum(w.seqlens_k)
        shapes = [(tq, w.Hq, w.D), (tk, w.Hkv, w.D), (tk, w.Hkv, w.D), (tq, w.Hq, w.D)]
    else:
        shapes = [(w.B, w.Hq, w.Nq, w.D), (w.B, w.Hkv, w.Nk, w.D), (w.B, w.Hkv, w.Nk, w.D),
                  (w.B, w.Hq, w.Nq, w.D)]
    out = [torch.randn(s, generator=g, dtype=torch.float32).to(dt) for s in shapes]
    cu_q = cu_k = None
    if w.packed:
        cu_q = torch.tensor([0] + list(itertools.accumulate(w.seqlens_q)), dtype=torch.int32)
        cu_k = torch.tensor([0] + list(itertools.accumulate(w.seqlens_k)), dtype=torch.int32)
    if device != "cpu":
        out = [t.to(device) for t in out]
        if cu_q is not None:
            cu_q, cu_k = cu_q.to(device), cu_k.to(device)
    return (*out, cu_q, cu_k)


def seqlen_mix(total: int, lo: int, hi: int, seed: int) -> tuple:
    """Sequence lengths drawn uniformly from [lo, hi] (seeded) until they sum
    to `total` (the last one is cut to fit)."""
    g = torch.Generator("cpu")
    g.manual_seed(seed)
    lens, acc = [], 0
    while acc < total:
        n = int(torch.randint(lo, hi + 1, (1,), generator=g))
        n = min(n, total - acc)
        lens.append(n)
        acc += n
    return tuple(lens)


# General problems at the size of the long causal shape (32 query heads of
# 16384 rows, D = 128, bf16): grouped and multi-query heads, packed sequences,
# dropout, and cross-attention-like lengths.  The benchmark times them and the
# GPU tests check sampled rows of each against the oracle at this size.
_MIX = seqlen_mix(65536, 512, 8192, seed=1)
BENCH_GENERAL = [
    GeneralWorkload("gqa-bf16-B1-Hq32-Hkv8-N16384-D128-causal", 1, 32, 8, 16384, 16384, 128,
                    "bf16", True),
    GeneralWorkload("mqa-bf16-B1-Hq32-Hkv1-N16384-D128-causal", 1, 32, 1, 16384, 16384, 128,
                    "bf16", True),
    GeneralWorkload("dropout0.1-bf16-B1-H32-N16384-D128-causal", 1, 32, 32, 16384, 16384, 128,
                    "bf16", True, dropout_p=0.1),
    GeneralWorkload("varlen-bf16-64k-tokens-len512-8192-Hq32-Hkv8-D128-causal", len(_MIX), 32, 8,
                    max(_MIX), max(_MIX), 128, "bf16", True, seqlens_q=_MIX, seqlens_k=_MIX),
    GeneralWorkload("cross-bf16-B4-H32-Nq4096-Nk16384-D128-full", 4, 32, 32, 4096, 16384, 128,
                    "bf16", False),
]
