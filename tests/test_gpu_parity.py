"""GPU parity: the CUDA path (through the C ABI) against the fp64 oracle.

Workloads: the tiny fp32 case, bf16 B=4 H=16 N=1024 D=64, the D=64 sequence
sweep N=512..16384 (fp16, bf16) at its full launch size, the shape-coverage
set (D 16..128, ragged N, permuted views, inputs x4, fp16/bf16/fp32), the long
causal B=1 H=32 N=16384 D=128 bf16 step, and edge cases (N = 1, tile +- 1).
Full-size launches are checked on sampled rows the oracle computes one by one.
"""

from __future__ import annotations

import numpy as np
import pytest
import torch

from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import (LONG_CAUSAL, SWEEP_N, TINY_FP32, Workload,
                                             bf16_n1024, coverage, make_inputs, sweep)
from parity import HUGE, check_huge_heads, compare_full, compare_sampled, run_gpu, run_huge

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.set_path(fa.FA_PATH_AUTO)
    yield
    fa.set_path(fa.FA_PATH_AUTO)


def test_tiny_fp32():
    inputs, got = run_gpu(TINY_FP32)
    compare_full(TINY_FP32, inputs, got)


@pytest.mark.parametrize("causal", [False, True])
def test_bf16_n1024(causal):
    w = bf16_n1024(causal)
    inputs, got = run_gpu(w)
    compare_full(w, inputs, got, heads=[(0, 0), (1, 7), (3, 15)])
    compare_sampled(w, inputs, got, q_heads=[(b, h) for b in range(4) for h in (0, 5, 15)],
                    k_heads=[(2, 3)])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16"])
@pytest.mark.parametrize("N", SWEEP_N)
def test_sweep(N, dtype, causal):
    w = sweep(N, dtype, causal)
    inputs, got = run_gpu(w)
    heads = [(0, 0), (w.B - 1, 15), (w.B // 2, 7)]
    compare_sampled(w, inputs, got, q_heads=heads, k_heads=[(w.B - 1, 15)])
    if N <= 1024:
        compare_full(w, inputs, got, heads=[(0, 3)])


@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("dtype", ["fp16", "bf16", "fp32"])
@pytest.mark.parametrize("N", [1000, 3001])
@pytest.mark.parametrize("D", [16, 32, 64, 128])
def test_coverage_permuted_x4(D, N, dtype, causal):
    w = coverage(D, N, dtype, causal)
    inputs, got = run_gpu(w)
    compare_full(w, inputs, got, heads=[(0, 0), (1, 5)])
    compare_sampled(w, inputs, got, q_heads=[(b, h) for b in range(2) for h in range(8)],
                    k_heads=[(1, 2)])


def test_long_causal_step():
    w = LONG_CAUSAL
    inputs, got = run_gpu(w)
    compare_sampled(w, inputs, got, q_heads=[(0, h) for h in range(32)],
                    k_heads=[(0, 0), (0, 31)])


@pytest.mark.parametrize("dtype", ["bf16", "fp16", "fp32"])
@pytest.mark.parametrize("causal", [False, True])
@pytest.mark.parametrize("N", [1, 2, 63, 127, 128, 129, 255, 256, 257, 383])
@pytest.mark.parametrize("D", [16, 64, 128])
def test_edge_lengths(D, N, causal, dtype):
    w = Workload(f"edge-{dtype}-N{N}-D{D}", 1, 3, N, D, dtype, causal, seed=N)
    inputs, got = run_gpu(w)
    compare_full(w, inputs, got)


@pytest.mark.parametrize("causal", [False, True])
def test_deterministic(causal):
    """No atomics anywhere: two runs give bit-identical outputs."""
    w = Workload("det-bf16", 2, 4, 777, 128, "bf16", causal)
    inputs, a = run_gpu(w)
    _, b = run_gpu(w, inputs)
    for key in a:
        np.testing.assert_array_equal(a[key], b[key], err_msg=key)


def test_outputs_stay_inside_their_buffers():
    """Guard regions around every output stay untouched (ragged N, permuted
    output views)."""
    B, H, N, D = 2, 3, 333, 64
    dev = torch.device("cuda", 0)
    w = Workload("guard-bf16", B, H, N, D, "bf16", True)
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    pad = 4096
    numel = B * H * N * D
    sentinel = 12345.0

    def guarded(shape, dtype):
        buf = torch.full((pad + int(np.prod(shape)) + pad,), sentinel, dtype=dtype, device=dev)
        return buf, buf[pad:pad + int(np.prod(shape))].view(shape)

    bo, o = guarded((B, N, H, D), torch.bfloat16)
    o = o.permute(0, 2, 1, 3)
    bl, lse = guarded((B, H, N), torch.float32)
    bd, delta = guarded((B, H, N), torch.float32)
    bq, dq = guarded((B, H, N, D), torch.bfloat16)
    bk, dk = guarded((B, H, N, D), torch.bfloat16)
    bv, dv = guarded((B, H, N, D), torch.bfloat16)
    fa.fwd(q, k, v, o, lse, True, w.scale)
    fa.bwd_preprocess(o, do, delta)
    fa.bwd(q, k, v, do, lse, delta, dq, dk, dv, True, w.scale)
    torch.cuda.synchronize()
    for buf, n in ((bo, numel), (bl, B * H * N), (bd, B * H * N), (bq, numel), (bk, numel), (bv, numel)):
        assert (buf[:pad] == sentinel).all()
        assert (buf[pad + n:] == sentinel).all()
    assert fa.device_status() == 0


@pytest.mark.parametrize("D", [64, 128])
def test_ffma_path_and_default_path_both_match_oracle(D):
    """The FFMA kernels (forced for bf16) and the default tensor-core kernels
    each match the oracle; so they agree with each other within twice the
    tolerance on O, L, dQ, dK and dV."""
    w = Workload(f"paths-bf16-D{D}", 2, 4, 1000, D, "bf16", True)
    inputs, a = run_gpu(w)
    fa.set_path(fa.FA_PATH_FFMA)
    try:
        _, b = run_gpu(w, inputs)
    finally:
        fa.set_path(fa.FA_PATH_AUTO)
    heads = [(0, 0), (1, 3)]
    compare_full(w, inputs, a, heads=heads)
    compare_full(w, inputs, b, heads=heads)
    for key in ("o", "lse", "dq", "dk", "dv"):
        assert np.abs(a[key] - b[key]).max() <= 2 * 2e-2, key


def test_autograd_wrapper_and_double_backward_refused():
    dev = torch.device("cuda", 0)
    w = Workload("autograd-bf16", 1, 2, 300, 64, "bf16", True)
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    qa, ka, va = (t.clone().requires_grad_(True) for t in (q, k, v))
    o = fa.attention(qa, ka, va, causal=True)
    o.backward(do)
    o2, lse = fa.attention_fwd(q, k, v, True)
    dq, dk, dv = fa.attention_bwd(q, k, v, o2, lse, do, True)
    assert torch.equal(o, o2)
    assert torch.equal(qa.grad, dq) and torch.equal(ka.grad, dk) and torch.equal(va.grad, dv)
    qb = q.clone().requires_grad_(True)
    ob = fa.attention(qb, k, v, causal=True)
    (g,) = torch.autograd.grad(ob, qb, do, create_graph=True)
    with pytest.raises(RuntimeError):
        g.sum().backward()


def test_invalid_arguments_return_codes_without_launch():
    dev = torch.device("cuda", 0)
    q = torch.zeros(1, 1, 64, 64, dtype=torch.bfloat16, device=dev)
    o = torch.empty_like(q)
    lse = torch.empty(1, 1, 64, dtype=torch.float32, device=dev)
    with pytest.raises(fa.FAError) as e:
        fa.fwd(q, q, q, o, lse, False, -1.0)
    assert e.value.code == 10
    qs = q[..., ::2]
    with pytest.raises(fa.FAError) as e:
        fa.fwd(qs, qs, qs, o[..., ::2], lse, False, 0.1)
    assert e.value.code == 5
    assert fa.device_status() == 0


def test_offsets_beyond_2_31_elements():
    """64-bit offsets ("Triton FlashAttention", lessons): every kernel of the
    split path addresses tensors of more than 2^31 elements; sampled rows of
    the last head, which lies wholly past element 2^31, match the oracle."""
    inputs, out = run_huge(HUGE, fused=False)
    check_huge_heads(HUGE, inputs, out, heads=[(0, 255)])
    del inputs, out
    torch.cuda.empty_cache()
