"""Device-side failure detection without a GPU fault.

Every mbarrier wait in the tensor-core kernels is bounded.  A test hook
withholds one arrival in the next forward launch (a flag nothing else sets);
the waiting warps run out their bound, the kernel records FA_ERR_TIMEOUT,
drains what it has in flight, frees its tensor memory and returns.  The host
reads the status, and the same context then runs forward and backward
correctly.
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
