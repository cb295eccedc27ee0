"""fa_bwd_noalloc: the backward for callers that cannot allocate device memory.

Callers that run the backward while a CUDA graph is being captured, inside a
framework that hands them fixed buffers and no allocator, or on a path that
must not take cudaMalloc's implicit synchronisation cannot allocate the
per-row Delta buffer that fa_bwd_preprocess / fa_bwd ask for.  The entry point
under test keeps Delta in a fixed buffer inside the library.  These tests call
it through the C ABI and check it against the regular entry points.

This file is named so that pytest collects it last.
"""

from __future__ import annotations

import ctypes

import pytest
import torch

from exact_attention_83_gb300 import build as fabuild
from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import Workload, make_inputs


@pytest.mark.gpu
def test_noalloc_backward_matches_regular_backward_on_two_calls_in_a_row():
    """Same preprocess, dK/dV and dQ kernels on the same inputs as the regular
    entry points, only Delta lives elsewhere: the outputs must be bit-identical
    (a stale Delta row or a race on the shared array would show here)."""
    dev = torch.device("cuda", 0)
    fa.load_library()
    fa.set_path(fa.FA_PATH_AUTO)
    # Two calls in a row with different shapes and masks: the second must not
    # see anything the first left in the library's buffer.
    cases = [Workload("noalloc-bf16-causal", 2, 8, 1500, 128, "bf16", True, seed=11),
             Workload("noalloc-fp16-full", 1, 4, 700, 64, "fp16", False, seed=12)]
    for w in cases:
        q, k, v, do = (t.to(dev) for t in make_inputs(w))
        o, lse = fa.attention_fwd(q, k, v, w.causal, w.scale)
        ref = fa.attention_bwd(q, k, v, o, lse, do, w.causal, w.scale)
        got = [torch.full_like(q, float("nan")) for _ in range(3)]
        fa.bwd_noalloc(q, k, v, o, do, lse, *got, w.causal, w.scale)
        torch.cuda.synchronize()
        assert fa.device_status() == 0
        for name, g, r in zip(("dq", "dk", "dv"), got, ref):
            assert torch.equal(g, r), (w.name, name)


_FAKE = 0x100000          # a 16-byte aligned address no kernel ever receives


def _call(lib, B, H, N, D, scale=0.088, dq=_FAKE, dtype=2):
    st = (ctypes.c_int64 * 4)(0, 0, D, 1)
    f = _FAKE
    return lib.fa_bwd_noalloc(f, f, f, f, f, f, dq, f, f, B, H, N, D, st, st, st, st, st, st, st,
                              st, 1, ctypes.c_float(scale), dtype, None)


def test_noalloc_rejects_sizes_beyond_its_buffer():
    """The size and argument checks come before any device work: without a
    GPU (here) a call that reached the device would return FA_ERR_LAUNCH, so
    the exact validation codes show that nothing was touched."""
    fabuild.build()
    lib = fa.load_library()
    rows_ok = 1 << 22
    # Exactly at the limit the size is accepted; D = 48 then stops the call at
    # argument validation, so no kernel ever sees the fake pointers.
    assert _call(lib, 1, 1, rows_ok, 48) == 3                  # FA_ERR_HEADDIM
    assert _call(lib, 1, 2, rows_ok // 2 + 1, 128) == 12       # FA_ERR_SCRATCH
    assert lib.fa_status_string(12).decode().startswith("FA_ERR_SCRATCH")


def test_noalloc_validates_every_argument_before_device_work():
    fabuild.build()
    lib = fa.load_library()
    assert _call(lib, 1, 2, 256, 128, scale=0.0) == 10          # FA_ERR_SCALE
    assert _call(lib, 1, 2, 256, 128, scale=float("inf")) == 10
    assert _call(lib, 1, 2, 256, 128, dq=0) == 1                # FA_ERR_NULL
    assert _call(lib, 1, 2, 256, 128, dq=_FAKE + 8) == 6        # FA_ERR_ALIGN
    assert _call(lib, 1, 2, 256, 128, dtype=7) == 4             # FA_ERR_DTYPE
    assert _call(lib, 0, 2, 256, 128) == 2                      # FA_ERR_SHAPE


@pytest.mark.gpu
def test_forward_and_noalloc_backward_replay_from_a_cuda_graph():
    """The use the entry point exists for: the forward and fa_bwd_noalloc
    captured into a CUDA graph (no allocation may happen during capture) and
    replayed; the replay gives bit-identical results to eager calls."""
    dev = torch.device("cuda", 0)
    fa.load_library()
    fa.set_path(fa.FA_PATH_AUTO)
    w = Workload("graph-bf16-causal", 1, 4, 1000, 128, "bf16", True, seed=13)
    q, k, v, do = (t.to(dev) for t in make_inputs(w))
    o = torch.empty_like(q)
    lse = torch.empty(w.B, w.H, w.N, dtype=torch.float32, device=dev)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))

    def step():
        fa.fwd(q, k, v, o, lse, w.causal, w.scale)
        fa.bwd_noalloc(q, k, v, o, do, lse, dq, dk, dv, w.causal, w.scale)

    s = torch.cuda.Stream(dev)
    s.wait_stream(torch.cuda.current_stream(dev))
    with torch.cuda.stream(s):
        step()                       # first call on the device: looks up the buffer
    torch.cuda.current_stream(dev).wait_stream(s)
    torch.cuda.synchronize()
    ref = [t.clone() for t in (o, lse, dq, dk, dv)]
    for t in (o, lse, dq, dk, dv):
        t.fill_(float("nan"))
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        step()
    for _ in range(2):
        graph.replay()
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for name, got, want in zip(("o", "lse", "dq", "dk", "dv"), (o, lse, dq, dk, dv), ref):
        assert torch.equal(got, want), name
