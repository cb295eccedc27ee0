"""Device-side failure detection without a GPU fault.

Every mbarrier wait in the tensor-core kernels is bounded.  A test hook
withholds one arrival in the next forward or single-pass backward launch (a
flag nothing else sets); the waiting warps run out their bound, the kernel
records FA_ERR_TIMEOUT, drains what it has in flight, frees its tensor memory
and returns.  The host reads the status, and the same context then runs
forward and backward correctly.
"""

import numpy as np
import pytest
import torch

from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import Workload, make_inputs
from parity import compare_full, run_gpu

pytestmark = pytest.mark.gpu


def test_withheld_arrival_times_out_and_context_stays_usable():
    lib = fa.load_library()
    dev = torch.device("cuda", 0)
    w = Workload("timeout-bf16", 1, 2, 600, 128, "bf16", True)
    q, k, v, _ = (t.to(dev) if t is not None else None for t in make_inputs(w))
    assert fa.device_status() == 0
    fa.set_wait_timeout_ns(50_000_000)          # 50 ms bound for this test
    try:
        lib.fa_test_withhold_next_arrival()
        o, lse = fa.attention_fwd(q, k, v, True, w.scale)
        torch.cuda.synchronize()
        assert fa.device_status() == 8          # FA_ERR_TIMEOUT, read and cleared
        assert fa.device_status() == 0          # the word was cleared
    finally:
        fa.set_wait_timeout_ns(0)               # back to the default bound
    # the context is usable: a full forward + backward matches the oracle
    inputs, got = run_gpu(w)
    compare_full(w, inputs, got)


def test_single_pass_backward_times_out_and_context_stays_usable():
    """The same hook on the single-pass backward: the MMA warp of CTA 0 gives
    up waiting for the first P^T, every role of that CTA ends its loop, the
    reductions already issued complete, and the next calls run correctly."""
    lib = fa.load_library()
    dev = torch.device("cuda", 0)
    w = Workload("timeout-fused-bf16", 1, 2, 600, 128, "bf16", True)
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    o, lse = fa.attention_fwd(q, k, v, True, w.scale)
    delta = torch.empty(1, 2, 600, dtype=torch.float32, device=dev)
    fa.bwd_preprocess(o, do, delta)
    ws = torch.empty(fa.workspace_bytes(q, k, True, w.scale) // 4, dtype=torch.float32,
                     device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    fa.set_wait_timeout_ns(50_000_000)
    try:
        lib.fa_test_withhold_next_arrival()
        fa.bwd_fused(q, k, v, do, lse, delta, dq, dk, dv, True, w.scale, workspace=ws)
        torch.cuda.synchronize()
        assert fa.device_status() == 8          # FA_ERR_TIMEOUT
        assert fa.device_status() == 0
    finally:
        fa.set_wait_timeout_ns(0)
    fa.bwd_fused(q, k, v, do, lse, delta, dq, dk, dv, True, w.scale, workspace=ws)
    dq2, dk2, dv2 = fa.attention_bwd(q, k, v, o, lse, do, True, w.scale)
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    assert torch.equal(dk, dk2) and torch.equal(dv, dv2)
    assert (dq.float() - dq2.float()).abs().max().item() <= 2e-2
