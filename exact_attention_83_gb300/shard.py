"""Host-side helpers for running the attention path on several GPUs.

Every (batch, head) pair is independent in both the forward and the backward,
so several GPUs need no exchange step: a job either gives each rank its own
workload (weak scaling, as the benchmark does) or splits the B*H heads into
contiguous ranges (head_shard).  The only collectives are host bookkeeping:
a barrier and the maximum of the per-rank timings.
"""

from __future__ import annotations

import dataclasses

import torch


def head_shard(num_heads: int, world: int, rank: int) -> range:
    """Contiguous range of flat head indices (b*H + h) owned by `rank`; the
    first num_heads % world ranks get one extra head."""
    if world < 1 or not 0 <= rank < world or num_heads < 0:
        raise ValueError("invalid shard request")
    base, extra = divmod(num_heads, world)
    start = rank * base + min(rank, extra)
    return range(start, start + base + (1 if rank < extra else 0))


def rank_workload(w, rank: int):
    """The workload rank `rank` runs under weak scaling: the same shape, its
    own seed (independent problems)."""
    return dataclasses.replace(w, seed=w.seed + rank)


def max_over_ranks(x: float, device=None) -> float:
    """Maximum of a per-rank scalar over the default process group (x itself
    when torch.distributed is not initialised)."""
    if not (torch.distributed.is_available() and torch.distributed.is_initialized()):
        return float(x)
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())
