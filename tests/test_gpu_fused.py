"""GPU parity for the single-pass backward (fa_bwd_fused): one kernel per key
tile produces dK, dV and each tile's share of dQ, summed by fp32 bulk
reductions into a workspace and converted by a second kernel.

The same oracle and tolerances as the split backward, over the same workloads:
the long causal training shape (sampled rows), bf16 N=1024, the D=64 sequence
sweep, the shape-coverage set (fp16/bf16), edge lengths, and the general
problems (Nq != Nk, grouped heads, packed sequences, dropout, seeded random
problems).  dK and dV must equal the split backward's bit for bit (same
products in the same order); dQ, summed in an order that is not fixed, within
the tolerance.
"""

from __future__ import annotations

import dataclasses

import numpy as np
import pytest
import torch

from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import (LONG_CAUSAL, SWEEP_N, GeneralWorkload, Workload,
                                             bf16_n1024, coverage, make_inputs, sweep)
from parity import HUGE, check_huge_heads, compare_full, compare_sampled, run_gpu, run_huge
from general import PAGE_SHAPES, compare, random_general, run_general

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.set_path(fa.FA_PATH_AUTO)
    yield
    fa.set_path(fa.FA_PATH_AUTO)


# --------------------------------------------------------------- square problems
def test_long_causal_step_fused():
    w = LONG_CAUSAL
    inputs, got = run_gpu(w, fused=True)
    compare_sampled(w, inputs, got, q_heads=[(0, h) for h in range(32)],
                    k_heads=[(0, 0), (0, 31)])


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_n1024_fused(causal):
    w = bf16_n1024(causal)
    inputs, got = run_gpu(w, fused=True)
    compare_full(w, inputs, got, heads=[(0, 0), (1, 7), (3, 15)])
    compare_sampled(w, inputs, got, q_heads=[(b, h) for b in range(4) for h in (0, 5, 15)],
                    k_heads=[(2, 3)])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("N", SWEEP_N)
def test_sweep_fused(N, dtype, causal):
    w = sweep(N, dtype, causal)
    inputs, got = run_gpu(w, fused=True)
    heads = [(0, 0), (w.B - 1, 15), (w.B // 2, 7)]
    compare_sampled(w, inputs, got, q_heads=heads, k_heads=[(w.B - 1, 15)])
    if N <= 1024:
        compare_full(w, inputs, got, heads=[(0, 3)])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("N", [1000, 3001])
@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_coverage_permuted_x4_fused(D, N, dtype, causal):
    w = coverage(D, N, dtype, causal)
    inputs, got = run_gpu(w, fused=True)
    compare_full(w, inputs, got, heads=[(0, 0), (1, 5)])
    compare_sampled(w, inputs, got, q_heads=[(b, h) for b in range(2) for h in range(8)],
                    k_heads=[(1, 2)])


@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 63, 127, 128, 129, 255, 257, 383])
@pytest.mark.parametrize("D", [16, 64, 128])
def test_edge_lengths_fused(D, N, causal, dtype):
    w = Workload(f"edge-fused-{dtype}-N{N}-D{D}", 1, 3, N, D, dtype, causal, seed=N)
    inputs, got = run_gpu(w, fused=True)
    compare_full(w, inputs, got)


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("D", [64, 128])
def test_dk_dv_equal_split_backward_bitwise(D, causal):
    """The single-pass kernel forms dK and dV with the same products in the
    same order as the split dK/dV kernel: identical bits.  dQ agrees within
    the fp32 rounding of a different summation order, far inside the
    tolerance."""
    w = Workload(f"fused-vs-split-D{D}", 2, 4, 777, D, "bf16", causal)
    inputs, split = run_gpu(w)
    _, fused = run_gpu(w, inputs, fused=True)
    for key in ("o", "lse", "delta", "dk", "dv"):
        np.testing.assert_array_equal(fused[key], split[key], err_msg=key)
    assert np.abs(fused["dq"] - split["dq"]).max() <= 2e-2


def test_runs_repeat_dk_dv_exactly_and_dq_closely():
    w = Workload("fused-repeat", 2, 4, 1000, 128, "bf16", True)
    inputs, a = run_gpu(w, fused=True)
    _, b = run_gpu(w, inputs, fused=True)
    for key in ("dk", "dv"):
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)
    assert np.abs(a["dq"] - b["dq"]).max() <= 1e-2


def test_outputs_stay_inside_their_buffers_fused():
    """Guard regions around dQ, dK, dV and the workspace stay untouched
    (ragged N, permuted dQ view)."""
    B, H, N, D = 2, 3, 333, 64
    w = Workload("guard-fused-bf16", B, H, N, D, "bf16", True)
    q, k, v, do = (t.to(DEV) for t in make_inputs(w))
    o, lse = fa.attention_fwd(q, k, v, True)
    delta = torch.empty(B, H, N, dtype=torch.float32, device=DEV)
    fa.bwd_preprocess(o, do, delta)
    pad, sentinel = 4096, 12345.0

    def guarded(n, dtype):
        buf = torch.full((pad + n + pad,), sentinel, dtype=dtype, device=DEV)
        return buf, buf[pad:pad + n]

    numel = B * H * N * D
    bq, dq = guarded(numel, torch.bfloat16)
    dq = dq.view(B, N, H, D).permute(0, 2, 1, 3)
    bk, dk = guarded(numel, torch.bfloat16)
    bv, dv = guarded(numel, torch.bfloat16)
    nws = fa.workspace_bytes(q, k, True) // 4
    bw, ws = guarded(nws, torch.float32)
    fa.bwd_fused(q, k, v, do, lse, delta, dq, dk.view(B, H, N, D), dv.view(B, H, N, D), True,
                 workspace=ws)
    torch.cuda.synchronize()
    for buf, n in ((bq, numel), (bk, numel), (bv, numel), (bw, nws)):
        assert (buf[:pad] == sentinel).all() and (buf[pad + n:] == sentinel).all()
    assert fa.device_status() == 0
    dq2, dk2, dv2 = fa.attention_bwd(q, k, v, o, lse, do, True)
    assert torch.equal(dk.view(B, H, N, D), dk2) and torch.equal(dv.view(B, H, N, D), dv2)
    assert (dq.float() - dq2.float()).abs().max().item() <= 2e-2


def test_workspace_is_zeroed_by_the_call():
    """A workspace full of garbage gives the same result as a clean one."""
    w = Workload("fused-ws-garbage", 1, 2, 300, 64, "fp16", False)
    q, k, v, do = (t.to(DEV) for t in make_inputs(w))
    o, lse = fa.attention_fwd(q, k, v, False)
    delta = torch.empty(1, 2, 300, dtype=torch.float32, device=DEV)
    fa.bwd_preprocess(o, do, delta)
    outs = []
    for fill in (0.0, 1e30):
        ws = torch.full((fa.workspace_bytes(q, k) // 4,), fill, dtype=torch.float32, device=DEV)
        g = [torch.empty_like(q) for _ in range(3)]
        fa.bwd_fused(q, k, v, do, lse, delta, *g, False, workspace=ws)
        outs.append(g)
    for a, b in zip(*outs):
        assert (a.float() - b.float()).abs().max().item() <= 1e-3


def test_fused_backward_replays_from_a_cuda_graph():
    """The call allocates nothing (the workspace is the caller's), so it can be
    captured into a CUDA graph and replayed."""
    w = Workload("graph-fused-bf16", 1, 4, 1000, 128, "bf16", True, seed=13)
    q, k, v, do = (t.to(DEV) for t in make_inputs(w))
    o, lse = fa.attention_fwd(q, k, v, True)
    delta = torch.empty(1, 4, 1000, dtype=torch.float32, device=DEV)
    ws = torch.empty(fa.workspace_bytes(q, k, True) // 4, dtype=torch.float32, device=DEV)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fa.bwd_preprocess(o, do, delta)
        fa.bwd_fused(q, k, v, do, lse, delta, dq, dk, dv, True, workspace=ws)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (dq, dk, dv)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.bwd_preprocess(o, do, delta)
        fa.bwd_fused(q, k, v, do, lse, delta, dq, dk, dv, True, workspace=ws)
    for t in (dq, dk, dv):
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(dk, ref[1]) and torch.equal(dv, ref[2])
    assert (dq.float() - ref[0].float()).abs().max().item() <= 1e-2
    assert fa.device_status() == 0


# --------------------------------------------------------------- general problems
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("shape", PAGE_SHAPES, ids=lambda s: "x".join(map(str, s)))
def test_page_shapes_fused(shape, dtype, causal):
    B, Nq, Nk, D = shape
    w = GeneralWorkload(f"shape-fused-{dtype}-{B}x{Nq}x{Nk}x{D}-{causal}", B, 2, 2, Nq, Nk, D,
                        dtype, causal, seed=Nq + Nk)
    compare(w, *run_general(w, fused=True))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("Nq,Nk", [(300, 1000), (1000, 300), (129, 1), (1, 257), (640, 641)])
def test_non_square_lengths_fused(Nq, Nk, causal):
    w = GeneralWorkload(f"nonsq-fused-{Nq}x{Nk}-{causal}", 2, 4, 4, Nq, Nk, 128, "bf16", causal,
                        seed=7)
    compare(w, *run_general(w, fused=True))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["bf16", "fp16"])
@pytest.mark.parametrize("Hq,Hkv,D", [(8, 2, 128), (8, 1, 64), (6, 3, 32), (4, 4, 16),
                                      (16, 2, 128)])
def test_grouped_heads_fused(Hq, Hkv, D, dtype, causal):
    """Few key/value heads leave the grid short, so clusters of CTAs split each
    key tile's query heads (dK, dV summed through distributed shared memory)."""
    w = GeneralWorkload(f"gqa-fused-{dtype}-Hq{Hq}-Hkv{Hkv}-D{D}-{causal}", 2, Hq, Hkv, 777, 901,
                        D, dtype, causal, seed=Hq * 10 + Hkv)
    compare(w, *run_general(w, fused=True))


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("lens", [(1, 127, 128, 129, 700, 0, 1500, 3), (256, 1, 511)],
                         ids=["mix", "short"])
def test_packed_sequences_fused(lens, causal):
    """Packed rows past a sequence's end belong to the next sequence: its keys
    must not leak into this sequence's dQ, and the exact zeros this sequence's
    tail rows add to the next one change nothing."""
    lk = tuple(reversed(lens))
    w = GeneralWorkload(f"varlen-fused-{len(lens)}seq-{causal}", len(lens), 8, 2, max(lens),
                        max(lk), 128, "bf16", causal, seqlens_q=lens, seqlens_k=lk, seed=3)
    compare(w, *run_general(w, fused=True))


def test_packed_sequence_with_no_keys_fused():
    w = GeneralWorkload("varlen-nokeys-fused", 3, 4, 4, 200, 130, 64, "bf16", False,
                        seqlens_q=(200, 5, 0), seqlens_k=(0, 9, 130), seed=4)
    inputs, got = run_general(w, fused=True)
    assert (got["dq"][:200] == 0).all()
    assert (got["dk"][9:] == 0).all() and (got["dv"][9:] == 0).all()
    compare(w, inputs, got)


def test_packed_rows_outside_every_sequence_untouched():
    """Rows before cu_seqlens_q[0] and after cu_seqlens_q[B] keep their dQ."""
    H, D = 2, 64
    total = 400
    cu = torch.tensor([50, 150, 330], dtype=torch.int32, device=DEV)
    gen = torch.Generator().manual_seed(21)
    q, k, v, do = (torch.randn(total, H, D, generator=gen).to(torch.bfloat16).to(DEV)
                   for _ in range(4))
    kw = dict(cu_seqlens_q=cu, cu_seqlens_k=cu, max_seqlen_q=180, max_seqlen_k=180)
    o, lse = fa.attention_ex_fwd(q, k, v, True, None, **kw)
    delta = torch.empty(H, total, dtype=torch.float32, device=DEV)
    fa.bwd_preprocess(fa._as4(o, True), fa._as4(do, True), delta)
    dq = torch.full_like(q, 7.0)
    dk, dv = torch.empty_like(k), torch.empty_like(v)
    ws = torch.empty(fa.workspace_bytes(q, k, True, None, **kw) // 4, dtype=torch.float32,
                     device=DEV)
    fa.bwd_fused(q, k, v, do, lse, delta, dq, dk, dv, True, None, workspace=ws, **kw)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert (dq[:50] == 7.0).all() and (dq[330:] == 7.0).all()
    assert not (dq[50:330] == 7.0).all()


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype,D", [("bf16", 128), ("fp16", 64), ("bf16", 32)])
def test_dropout_fused(dtype, D, causal):
    w = GeneralWorkload(f"drop-fused-{dtype}-D{D}-{causal}", 2, 4, 2, 333, 517, D, dtype, causal,
                        dropout_p=0.17, seed=5, drop_seed=0xDEADBEEF12345, drop_offset=3)
    compare(w, *run_general(w, fused=True))


def test_dropout_packed_fused():
    lens = (100, 1, 260, 0, 64)
    w = GeneralWorkload("drop-varlen-fused", 5, 4, 1, 260, 260, 64, "bf16", True,
                        seqlens_q=lens, seqlens_k=lens, dropout_p=0.3, seed=6, drop_offset=11)
    compare(w, *run_general(w, fused=True))


@pytest.mark.parametrize("seed", range(40))
def test_random_general_problems_fused(seed):
    w = random_general(seed)
    if w.dtype == "fp32":           # the single-pass backward takes 16-bit inputs only
        w = dataclasses.replace(w, dtype="bf16")
    compare(w, *run_general(w, fused=True))


def test_autograd_single_pass_backward():
    w = GeneralWorkload("autograd-fused", 1, 4, 2, 200, 260, 64, "bf16", True, dropout_p=0.1,
                        seed=9)
    from exact_attention_83_gb300.inputs import make_general_inputs
    q, k, v, do, _, _ = make_general_inputs(w, DEV)
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = fa.attention_gqa(qa, ka, va, True, None, 0.1, w.drop_seed, 0, deterministic=False)
    o.backward(do)
    o2, lse = fa.attention_ex_fwd(q, k, v, True, None, dropout_p=0.1, seed=w.drop_seed)
    dq, dk, dv = fa.attention_ex_bwd(q, k, v, o2, lse, do, True, None, dropout_p=0.1,
                                     seed=w.drop_seed)
    assert torch.equal(ka.grad, dk) and torch.equal(va.grad, dv)
    assert (qa.grad.float() - dq.float()).abs().max().item() <= 2e-2


def test_fused_rejects_fp32_and_short_workspace():
    q = torch.zeros(1, 2, 64, 64, dtype=torch.float32, device=DEV)
    ws = torch.zeros(1 << 16, dtype=torch.float32, device=DEV)
    with pytest.raises(fa.FAError) as e:
        fa.bwd_fused(q, q, q, q, q[0, :, :, 0], q[0, :, :, 0], q, q, q, False, workspace=ws)
    assert e.value.code == 4
    qb = q.to(torch.bfloat16)
    lse = torch.zeros(1, 2, 64, dtype=torch.float32, device=DEV)
    need = fa.workspace_bytes(qb, qb)
    assert need == 1 * 2 * 64 * 64 * 4
    with pytest.raises(fa.FAError) as e:
        fa.bwd_fused(qb, qb, qb, qb, lse, lse, qb, qb, qb, False, workspace=ws[: need // 4 - 4])
    assert e.value.code == 12
    with pytest.raises(fa.FAError) as e:
        fa.bwd_fused(qb, qb, qb, qb, lse, lse, qb, qb, qb, False, workspace=ws[1:])
    assert e.value.code == 6
    assert fa.device_status() == 0


def test_offsets_beyond_2_31_elements_fused():
    """The single-pass backward and its workspace (8.6 GB) on tensors of more
    than 2^31 elements; sampled rows of the last head, wholly past element
    2^31."""
    inputs, out = run_huge(HUGE, fused=True)
    check_huge_heads(HUGE, inputs, out, heads=[(0, 255)])
    del inputs, out
    torch.cuda.empty_cache()
