"""Multi-rank host logic on CPU with the gloo backend (world size 2).

The attention path shards by independent heads, so several ranks never
exchange data; these tests check the head partition (every head owned by
exactly one rank, results assembled from the ranks' shards equal the
single-process result, computed here with the fp64 oracle on CPU), the
per-rank workload of weak scaling, and the max-over-ranks timing reduction.
"""

from __future__ import annotations

import os
import socket

import numpy as np
import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

import oracle
from exact_attention_83_gb300 import shard
from exact_attention_83_gb300.inputs import Workload, make_inputs


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank: int, world: int, port: int, out_dir: str):
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        w = Workload("gloo-shard", 2, 3, 40, 8, "fp32", True)
        q, k, v, do = make_inputs(w)
        heads = shard.head_shard(w.B * w.H, world, rank)
        flat = lambda t: t.reshape(w.B * w.H, 1, w.N, w.D)[heads.start:heads.stop]
        g = oracle.fwd_bwd(*(flat(t).permute(1, 0, 2, 3) for t in (q, k, v, do)), w.causal, w.scale)
        mine = torch.from_numpy(np.concatenate([g["o"], g["dq"], g["dk"], g["dv"]], axis=0))
        # gather every rank's shard (variable size: pad to the largest)
        n_max = -(-w.B * w.H // world)
        pad = torch.zeros(4, 1, n_max, w.N, w.D, dtype=torch.float64)
        pad[:, :, :len(heads)] = mine.reshape(4, 1, len(heads), w.N, w.D)
        parts = [torch.zeros_like(pad) for _ in range(world)]
        dist.all_gather(parts, pad)
        t = shard.max_over_ranks(float(rank + 1))
        if rank == 0:
            full = []
            for r, p in enumerate(parts):
                n = len(shard.head_shard(w.B * w.H, world, r))
                full.append(p[:, :, :n])
            full = torch.cat(full, dim=2).numpy()
            np.save(os.path.join(out_dir, "sharded.npy"), full)
            with open(os.path.join(out_dir, "max.txt"), "w") as f:
                f.write(repr(t))
    finally:
        dist.destroy_process_group()


def test_head_shard_partitions_every_head_once():
    for n in (1, 2, 7, 64, 65):
        for world in (1, 2, 3, 8):
            owned = [h for r in range(world) for h in shard.head_shard(n, world, r)]
            assert owned == list(range(n))
    with pytest.raises(ValueError):
        shard.head_shard(4, 2, 2)


def test_rank_workload_changes_only_the_seed():
    w = Workload("x", 1, 2, 16, 8, "bf16", True, seed=5)
    w1 = shard.rank_workload(w, 1)
    assert (w1.B, w1.H, w1.N, w1.D, w1.causal, w1.dtype) == (w.B, w.H, w.N, w.D, w.causal, w.dtype)
    assert w1.seed == 6 and shard.rank_workload(w, 0) == w


def test_two_gloo_ranks_assemble_the_single_process_result(tmp_path):
    world = 2
    mp.start_processes(_worker, args=(world, _free_port(), str(tmp_path)), nprocs=world,
                       join=True, start_method="spawn")
    got = np.load(tmp_path / "sharded.npy")
    w = Workload("gloo-shard", 2, 3, 40, 8, "fp32", True)
    q, k, v, do = make_inputs(w)
    ref = oracle.fwd_bwd(q, k, v, do, w.causal, w.scale)
    for i, key in enumerate(("o", "dq", "dk", "dv")):
        np.testing.assert_array_equal(got[i, 0], ref[key].reshape(w.B * w.H, w.N, w.D), err_msg=key)
    assert float((tmp_path / "max.txt").read_text()) == 2.0
