"""The backward's two kernels running at the same time.

For sequences of at most 4096 keys and queries, fa_bwd runs the dQ kernel on
a stream of the library's own, concurrently with the dK/dV kernel on the
caller's stream, and joins it back before returning (include/fa.h,
"Ordering").  The kernels are deterministic, so every path must give the same
bits as the in-sequence one:

* a backward captured into a CUDA graph (the library then keeps both kernels
  on the caller's stream) and replayed equals the eager call;
* two host threads, each running backwards on its own stream, get exactly what
  one thread gets (the side stream's fork and join are serialised per device);
* the profiling events still bracket the whole backward.
"""

from __future__ import annotations

import threading

import pytest
import torch

from exact_attention_83_gb300 import fa
from exact_attention_83_gb300.inputs import Workload, make_inputs

pytestmark = pytest.mark.gpu
DEV = torch.device("cuda", 0)


@pytest.fixture(scope="module", autouse=True)
def _lib():
    fa.load_library()
    fa.set_path(fa.FA_PATH_AUTO)
    yield


def _problem(w):
    q, k, v, do = (t.to(DEV) for t in make_inputs(w))
    o, lse = fa.attention_fwd(q, k, v, w.causal, w.scale)
    delta = torch.empty_like(lse)
    fa.bwd_preprocess(o, do, delta)
    return q, k, v, do, lse, delta


def _bwd(w, q, k, v, do, lse, delta):
    dq, dk, dv = (torch.full_like(q, float("nan")) for _ in range(3))
    fa.bwd(q, k, v, do, lse, delta, dq, dk, dv, w.causal, w.scale)
    return dq, dk, dv


CASES = [Workload("conc-bf16-causal-512", 4, 8, 512, 64, "bf16", True, seed=21),
         Workload("conc-fp16-full-1000-d128", 2, 4, 1000, 128, "fp16", False, seed=22)]


@pytest.mark.parametrize("w", CASES, ids=[w.name for w in CASES])
def test_graph_captured_backward_equals_eager(w):
    args = _problem(w)
    eager = _bwd(w, *args)
    q = args[0]
    outs = [torch.full_like(q, float("nan")) for _ in range(3)]
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        fa.bwd(*args[:6], *outs, w.causal, w.scale)
    for t in outs:
        t.fill_(float("nan"))
    g.replay()
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for name, a, b in zip(("dq", "dk", "dv"), outs, eager):
        assert torch.equal(a, b), (w.name, name)


def test_two_host_threads_on_their_own_streams():
    problems = [(w, _problem(w)) for w in CASES]
    ref = [_bwd(w, *args) for w, args in problems]
    torch.cuda.synchronize()
    results = [[None] * 3 for _ in problems]
    errors = []

    def worker(i):
        try:
            w, args = problems[i]
            s = torch.cuda.Stream(DEV)
            s.wait_stream(torch.cuda.current_stream(DEV))
            with torch.cuda.stream(s):
                for rep in range(3):
                    results[i][rep] = _bwd(w, *args)
            s.synchronize()
        except Exception as e:          # reported by the main thread
            errors.append(e)

    threads = [threading.Thread(target=worker, args=(i,)) for i in range(len(problems))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    torch.cuda.synchronize()
    assert fa.device_status() == 0
    for i, (w, _) in enumerate(problems):
        for rep in range(3):
            for name, a, b in zip(("dq", "dk", "dv"), results[i][rep], ref[i]):
                assert torch.equal(a, b), (w.name, rep, name)


def test_profile_events_bracket_the_overlapped_backward():
    w = CASES[0]
    args = _problem(w)
    ev = [torch.cuda.Event(enable_timing=True) for _ in range(3)]
    for e in ev:
        e.record()
    torch.cuda.synchronize()
    fa.set_profile_events(ev)
    try:
        out = _bwd(w, *args)
    finally:
        fa.set_profile_events(None)
    end = torch.cuda.Event(enable_timing=True)
    end.record()
    torch.cuda.synchronize()
    assert 0 <= ev[0].elapsed_time(ev[1]) <= ev[0].elapsed_time(ev[2])
    assert ev[2].elapsed_time(end) >= 0
    assert all(bool(torch.isfinite(t).all()) for t in out)
