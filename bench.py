"""Benchmark: exact attention forward + backward on GB300, one JSON line.

A step is one pass of the whole path on one batch: fa_fwd, fa_bwd_preprocess
and fa_bwd (dK/dV kernel then dQ kernel) on the long causal training shape
B=1, H=32, N=16384, D=128, bf16.  `value` is forward+backward TFLOP/s over all
ranks (forward 4*B*H*N^2*D flops halved for causal, backward credited at 2.5x
the forward), timed with CUDA events on the launching stream, inputs resident
in HBM.  The inputs (4 x 128 MiB) are larger than the 129 MB L2, so L2 is not
flushed between steps.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]
                  [--workload NAME] [--bwd split|fused]

The default run also adds a `sweep` record: the sequence-length sweep over the
metric's range (D = 64, H = 16, B*N = 16384, N = 512 .. 16384, bf16 and fp16,
causal and full), forward and forward+backward TFLOP/s per point with L2
flushed before every timed step; and `e2e.link`: the host link's rates for
the step's copies alone and the compute alone, so that the end-to-end time
can be set against max(compute, host-to-device, device-to-host).

`--bwd fused` times the single-pass backward (fa_bwd_fused: one kernel per key
tile, dQ summed by fp32 bulk reductions into a workspace, then converted)
instead of the split one.

Under torchrun each rank runs its own copy of the workload (independent heads,
no collective on the data path; weak scaling) and rank 0 prints the line.
`--impl reference` times the fp64 CPU oracle on a bounded sample (one head) of
the same workload on the host cores (rank 0 only).
"""

from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import torch  # noqa: E402

from exact_attention_83_gb300 import shard  # noqa: E402
from exact_attention_83_gb300.inputs import (BENCH_GENERAL, LONG_CAUSAL, SWEEP_N,  # noqa: E402
                                             TINY_FP32, GeneralWorkload, Workload, bf16_n1024,
                                             coverage, make_general_inputs, make_inputs, sweep)

METRIC = "attention TFLOP/s fwd & fwd+bwd, bf16 N=1k-16k, % of GB300 dense BF16 peak"

# ncu DRAM traffic (dram__bytes_read.sum + dram__bytes_write.sum) per launch of
# the dominant kernel, keyed by the sha256 of the source file it was measured
# on; a changed source gives null.  Figures come from the summaries under
# profiles/.
MEASURED_TRAFFIC = {
    # bwd_dkdv_tc_kernel<bf16,128>: 393.8 MB per launch measured on 16 heads,
    # scaled by heads to the 32-head launch (captured on source 06b6ebce...;
    # the file has changed since only in a comment)
    ("dkdv", "18895767631bca8a5cc47774cca7d10a7d5df65cee57a74897e0cc0d0d05f17c",
     "long-bf16-B1-H32-N16384-D128-causal"): 787.6e6,
    # bwd_fused_tc_kernel<bf16,128>: 2929.2 MB per launch measured on 16 heads,
    # scaled by heads to the 32-head launch
    ("fused", "7a40ac2fd235fad28a6a7f44662e8e368ab7a4b4121be356c5b381d64da86cd1",
     "long-bf16-B1-H32-N16384-D128-causal"): 5858.5e6,
}


# The long causal shape with half the heads: inputs (4 x 64 MiB) still exceed
# L2, device footprint ~0.5 GB; used for counter captures.
PROFILE_CASE = Workload("long-bf16-B1-H16-N16384-D128-causal", 1, 16, 16384, 128, "bf16", True)
# The dropout workload at the profiling size (16 heads: inputs, outputs and the
# 0.5 GB keep mask stay a few GB on the device under ncu).
PROFILE_DROPOUT = GeneralWorkload("dropout0.1-bf16-B1-H16-N16384-D128-causal", 1, 16, 16, 16384,
                                  16384, 128, "bf16", True, dropout_p=0.1)


def workloads():
    ws = {LONG_CAUSAL.name: LONG_CAUSAL, PROFILE_CASE.name: PROFILE_CASE,
          TINY_FP32.name: TINY_FP32, PROFILE_DROPOUT.name: PROFILE_DROPOUT}
    ws.update({g.name: g for g in BENCH_GENERAL})
    for c in (False, True):
        w = bf16_n1024(c)
        ws[w.name] = w
        for N in SWEEP_N:
            for dt in ("bf16", "fp16"):
                s = sweep(N, dt, c)
                ws[s.name] = s
        for D in (16, 32, 64, 128):
            for N in (1000, 3001):
                for dt in ("fp16", "bf16", "fp32"):
                    cv = coverage(D, N, dt, c)
                    ws[cv.name] = cv
    return ws


def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            p = json.load(f)
        return {"hbm_gbs": p["hbm_gbs"], "bf16_tflops": p["bf16_tflops"],
                "bf16_tflops_sustained": p.get("bf16_tflops_sustained", p["bf16_tflops"]),
                "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0,
            "source": "fallback"}


class ClockSampler:
    """nvidia-smi samples of SM clock and throttle reasons during the timed region.

    nvidia-smi's start-up (NVML initialisation) stalls the GPU for tens of
    milliseconds, so __enter__ returns only once the first sample has been
    printed: the stall then lies before the timed region, not inside it.  A
    reader thread drains the pipe so that a long region cannot fill it."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    START_TIMEOUT_S = 10.0
    SETTLE_S = 0.2

    def __init__(self, device_index: int):
        self.dev = device_index
        self.proc = None
        self.lines = []

    def _read(self, first):
        for ln in self.proc.stdout:
            if ln.strip():
                self.lines.append(ln)
                first.set()
        first.set()

    def __enter__(self):
        self.lines = []
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.dev), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "50"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return self
        first = threading.Event()
        self.reader = threading.Thread(target=self._read, args=(first,), daemon=True)
        self.reader.start()
        first.wait(self.START_TIMEOUT_S)
        time.sleep(self.SETTLE_S)
        self.lines.clear()          # samples from before the region
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.proc.wait()
            self.reader.join(timeout=5)
        return False

    def summary(self):
        sm, mx, reasons = [], [], set()
        names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
        for ln in getattr(self, "lines", []):
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                mx.append(float(parts[2]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() in ("active", "1", "yes"):
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["unsampled"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


def kernel_source_sha(name: str) -> str:
    path = os.path.join(ROOT, "exact_attention_83_gb300", "csrc", name)
    with open(path, "rb") as f:
        return hashlib.sha256(f.read()).hexdigest()


def run_reference(args, w: Workload):
    """The fp64 oracle on the host cores, one head of the workload per step."""
    import oracle
    sample = Workload(w.name + "-one-head", w.B, 1, w.N, w.D, w.dtype, w.causal, w.layout,
                      w.qkv_scale, w.seed)
    q, k, v, do = make_inputs(sample)
    qn, kn, vn, dn = (t.float().double().numpy() for t in (q, k, v, do))
    for _ in range(args.warmup):
        oracle.fwd_bwd(qn, kn, vn, dn, w.causal, w.scale)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.fwd_bwd(qn, kn, vn, dn, w.causal, w.scale)
    dt = (time.perf_counter() - t0) / max(args.steps, 1)
    tflops = sample.fwd_bwd_flops() / dt / 1e12
    cores = oracle.num_threads()
    line = {
        "metric": METRIC, "impl": "reference", "value": tflops, "unit": "TFLOP/s",
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": dt * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": w.name, "sample": "one head (B=1, H=1) per step",
                   "B": w.B, "H": w.H, "N": w.N, "D": w.D, "causal": w.causal},
        "cpu_baseline": {"value": tflops, "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"fp64 oracle fwd+bwd on 1 of {w.B * w.H} heads per step"},
        "e2e": {"value": tflops, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def cpu_baseline(w: Workload):
    """The oracle as it stands, on one head of the workload (bounded sample)."""
    import oracle
    sample = Workload(w.name + "-one-head", w.B, 1, w.N, w.D, w.dtype, w.causal, w.layout,
                      w.qkv_scale, w.seed)
    q, k, v, do = make_inputs(sample)
    qn, kn, vn, dn = (t.float().double().numpy() for t in (q, k, v, do))
    t0 = time.perf_counter()
    oracle.fwd_bwd(qn, kn, vn, dn, w.causal, w.scale)
    dt = time.perf_counter() - t0
    out = {"value": sample.fwd_bwd_flops() / dt / 1e12, "unit": "TFLOP/s",
           "cores": oracle.num_threads(), "kind": "oracle",
           "sample": f"fp64 oracle fwd+bwd on 1 of {w.B * w.H} heads ({dt:.1f} s)"}
    # the same on one core, on one head of a quarter of the length (the
    # oracle's work per flop does not depend on N)
    small = Workload(w.name + "-one-head-quarter", 1, 1, max(w.N // 4, 1), w.D, w.dtype,
                     w.causal, w.layout, w.qkv_scale, w.seed)
    q, k, v, do = make_inputs(small)
    qn, kn, vn, dn = (t.float().double().numpy() for t in (q, k, v, do))
    threads = oracle.num_threads()
    oracle.set_num_threads(1)
    try:
        t0 = time.perf_counter()
        oracle.fwd_bwd(qn, kn, vn, dn, w.causal, w.scale)
        dt1 = time.perf_counter() - t0
    finally:
        oracle.set_num_threads(threads)
    out["single_core"] = {"value": small.fwd_bwd_flops() / dt1 / 1e12, "unit": "TFLOP/s",
                          "cores": 1,
                          "sample": f"one head, N={small.N} ({dt1:.1f} s)"}
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=LONG_CAUSAL.name)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-sweep", action="store_true",
                    help="skip the sequence-length sweep record of the default run")
    ap.add_argument("--bwd", default="split", choices=["split", "fused"])
    ap.add_argument("--dropout-in-kernels", action="store_true",
                    help="dropout workloads: the backward kernels draw the keep decisions "
                         "again instead of reading the keep mask the forward stored")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3
    w = workloads()[args.workload]
    world, rank, local = dist_env()

    if isinstance(w, GeneralWorkload):
        if args.impl == "reference":
            if rank == 0:
                print(json.dumps({"impl": "reference", "unavailable":
                                  "the reference arm is timed on the long causal workload"}))
            return
        run_general(args, w, world, rank, local)
        return

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, w)
        return

    from exact_attention_83_gb300 import fa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    fa.load_library()

    # weak scaling: each rank runs its own independent copy of the workload
    q, k, v, do = (t.to(dev) for t in make_inputs(shard.rank_workload(w, rank)))
    B, H, N, D = w.B, w.H, w.N, w.D
    o = torch.empty((B, H, N, D), dtype=q.dtype, device=dev)
    lse = torch.empty((B, H, N), dtype=torch.float32, device=dev)
    delta = torch.empty_like(lse)
    dq, dk, dv = (torch.empty_like(q) for _ in range(3))
    stream = torch.cuda.current_stream(dev)
    fused = args.bwd == "fused"
    ws = (torch.empty(fa.workspace_bytes(q, k, w.causal, w.scale) // 4, dtype=torch.float32,
                      device=dev) if fused else None)

    def bwd():
        if fused:
            fa.bwd_fused(q, k, v, do, lse, delta, dq, dk, dv, w.causal, w.scale, workspace=ws)
        else:
            fa.bwd(q, k, v, do, lse, delta, dq, dk, dv, w.causal, w.scale)

    def step():
        fa.fwd(q, k, v, o, lse, w.causal, w.scale)
        fa.bwd_preprocess(o, do, delta)
        bwd()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    def max_over_ranks(x: float) -> float:
        return shard.max_over_ranks(x, dev)

    for _ in range(args.warmup):
        step()
    barrier()
    if fa.device_status() != 0:
        raise RuntimeError("device status not OK after warm-up")

    # Inputs smaller than twice the L2 are flushed from it before every timed
    # step (a 2 x L2 write, outside the events), and steps are timed one by one.
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    in_bytes = 4 * B * H * N * D * q.element_size()
    flush_buf = (torch.empty(2 * l2, dtype=torch.uint8, device=dev) if in_bytes < 2 * l2
                 else None)

    # ---- forward + backward step, with per-kernel events on the stream
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for e in ev:        # create the events (torch creates them lazily on first record)
        for x in e:
            x.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        start.record(stream)
        for i in range(args.steps):
            e = ev[i]
            if flush_buf is not None:
                flush_buf.zero_()
            e[0].record(stream)
            fa.fwd(q, k, v, o, lse, w.causal, w.scale)
            e[1].record(stream)
            fa.bwd_preprocess(o, do, delta)
            fa.set_profile_events(e[2:5])
            bwd()
        end.record(stream)
        barrier()
    fa.set_profile_events(None)
    if flush_buf is None:
        ms_step = max_over_ranks(start.elapsed_time(end)) / args.steps
    else:
        ms_step = max_over_ranks(statistics.median(e[0].elapsed_time(e[4]) for e in ev))
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    pre_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    dkdv_ms = statistics.median(e[2].elapsed_time(e[3]) for e in ev)
    dq_ms = statistics.median(e[3].elapsed_time(e[4]) for e in ev)
    if fa.device_status() != 0:
        raise RuntimeError("device status not OK after the timed region")

    # ---- forward alone
    barrier()
    if flush_buf is None:
        fs, fe = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        fs.record(stream)
        for _ in range(args.steps):
            fa.fwd(q, k, v, o, lse, w.causal, w.scale)
        fe.record(stream)
        barrier()
        fwd_only_ms = max_over_ranks(fs.elapsed_time(fe)) / args.steps
    else:
        fev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
               for _ in range(args.steps)]
        for a_, b_ in fev:
            flush_buf.zero_()
            a_.record(stream)
            fa.fwd(q, k, v, o, lse, w.causal, w.scale)
            b_.record(stream)
        barrier()
        fwd_only_ms = max_over_ranks(statistics.median(a_.elapsed_time(b_) for a_, b_ in fev))

    flops_fwd = w.fwd_flops()
    flops_step = w.fwd_bwd_flops()
    value = world * flops_step / (ms_step * 1e-3) / 1e12
    pk = peaks()
    # The timed region lasts tens of milliseconds and the sampled SM clock stays
    # at its maximum, so the burst cuBLAS rate is the denominator (the more
    # demanding of the two); the sustained-rate fraction is reported beside it.
    peak_dense = pk["bf16_tflops"]
    peak_sustained = pk["bf16_tflops_sustained"]

    # dominant kernel: the dK/dV kernel (4 of the 7 N x N x D products of the
    # split backward), or the single-pass kernel (5 products); algorithmic
    # flops are 2*N^2*D per product and head, halved when causal.
    nprod = 5 if fused else 4
    dkdv_flops = nprod * 2.0 * B * H * N * N * D * (0.5 if w.causal else 1.0)
    achieved = dkdv_flops / (dkdv_ms * 1e-3) / 1e12
    sha = kernel_source_sha("fa_bwd_fused.cu" if fused else "fa_bwd_tc.cu")
    traffic = MEASURED_TRAFFIC.get(("fused" if fused else "dkdv", sha, w.name))

    e2e = None
    if not args.no_e2e:
        e2e = measure_e2e(args, w, dev, fa, fused)

    sweep_rec = None
    if not args.no_sweep and w.name == LONG_CAUSAL.name and world == 1:
        sweep_rec = run_sweep(fa, dev, stream, args.steps, args.warmup, pk["bf16_tflops"])

    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(w)

    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": "bf16" if w.dtype == "bf16" else w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": B, "H": H, "N": N, "D": D,
                       "causal": w.causal, "parallelism": f"replicas{world}",
                       "backward": BWD_NAMES[args.bwd],
                       "l2": ("inputs 4 x %d MiB > L2, no flush" % (B * H * N * D * q.element_size() >> 20)
                              if flush_buf is None else
                              "L2 flushed (%d MiB write) before each step; steps timed one by one"
                              % (2 * l2 >> 20))},
            "fwd_tflops": world * flops_fwd / (fwd_only_ms * 1e-3) / 1e12,
            "fwd_ms": fwd_only_ms,
            "fwd_frac_of_peak": flops_fwd / (fwd_only_ms * 1e-3) / 1e12 / peak_dense,
            "fwd_bwd_frac_of_peak": value / world / peak_dense,
            "fwd_bwd_frac_of_sustained_peak": value / world / peak_sustained,
            "peak_tflops": peak_dense, "peak_source": pk["source"] + " burst bf16 (cuBLAS)",
            "kernel_ms": kernel_ms(fused, fwd_ms, pre_ms, dkdv_ms, dq_ms),
            "roofline": {"kernel": "bwd_fused" if fused else "bwd_dkdv", "bound": "tensor",
                         "achieved": achieved, "peak": peak_dense, "unit": "TFLOP/s",
                         "frac": achieved / peak_dense, "traffic": traffic},
            "clocks": clocks.summary(),
            "gpu_launches": 4 * args.steps,
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        if sweep_rec is not None:
            line["sweep"] = sweep_rec
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


BWD_NAMES = {"split": "split: dK/dV kernel + dQ kernel (deterministic)",
             "fused": "single pass: dQ by fp32 bulk reduce-add + convert"}


def kernel_ms(fused, fwd_ms, pre_ms, k1_ms, k2_ms):
    if fused:
        return {"fwd": fwd_ms, "preprocess+workspace_zero": pre_ms, "bwd_fused": k1_ms,
                "dq_convert": k2_ms}
    return {"fwd": fwd_ms, "preprocess": pre_ms, "bwd_dkdv": k1_ms, "bwd_dq": k2_ms}


def run_general(args, w: GeneralWorkload, world: int, rank: int, local: int):
    """fa_fwd_ex + fa_bwd_preprocess + fa_bwd_ex on a general problem; the same
    JSON line as the main workload (no e2e or CPU-baseline leg).  FLOPs count
    the attended (query, key) pairs exactly (causal: sum_i min(i + 1, Nk))."""
    from exact_attention_83_gb300 import fa
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl", device_id=dev)
    fa.load_library()
    q, k, v, do, cu_q, cu_k = make_general_inputs(w, dev)
    kw = dict(dropout_p=w.dropout_p, seed=w.drop_seed, offset=w.drop_offset)
    if w.packed:
        kw.update(cu_seqlens_q=cu_q, cu_seqlens_k=cu_k, max_seqlen_q=w.Nq, max_seqlen_k=w.Nk)
    o = torch.empty_like(q)
    lse_shape = (w.Hq, q.shape[0]) if w.packed else (w.B, w.Hq, w.Nq)
    lse = torch.empty(lse_shape, dtype=torch.float32, device=dev)
    delta = torch.empty_like(lse)
    dq, dk, dv = torch.empty_like(q), torch.empty_like(k), torch.empty_like(v)
    o4, do4 = fa._as4(o, w.packed), fa._as4(do, w.packed)
    stream = torch.cuda.current_stream(dev)
    fused = args.bwd == "fused"
    ws = (torch.empty(fa.workspace_bytes(q, k, w.causal, w.scale, **kw) // 4,
                      dtype=torch.float32, device=dev) if fused else None)
    # Dropout: by default the forward stores the keep decisions it draws in a
    # keep mask that the backward reads; with --dropout-in-kernels the
    # backward kernels draw them again.
    mask = None
    if w.dropout_p > 0 and not args.dropout_in_kernels:
        mask = torch.empty(fa.dropout_mask_bytes(q, k, w.causal, w.scale, **kw),
                           dtype=torch.uint8, device=dev)
        kw["dropout_mask"] = mask

    def bwd():
        if fused:
            fa.bwd_fused(q, k, v, do, lse, delta, dq, dk, dv, w.causal, w.scale, workspace=ws,
                         **kw)
        else:
            fa.bwd_ex(q, k, v, do, lse, delta, dq, dk, dv, w.causal, w.scale, **kw)

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize(dev)

    for _ in range(args.warmup):
        fa.fwd_ex(q, k, v, o, lse, w.causal, w.scale, **kw)
        fa.bwd_preprocess(o4, do4, delta)
        bwd()
    barrier()
    if fa.device_status() != 0:
        raise RuntimeError("device status not OK after warm-up")
    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(6)] for _ in range(args.steps)]
    for e in ev:
        for x in e:
            x.record(stream)
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clocks:
        barrier()
        start.record(stream)
        for i in range(args.steps):
            e = ev[i]
            e[0].record(stream)
            fa.fwd_ex(q, k, v, o, lse, w.causal, w.scale, **kw)
            e[1].record(stream)
            fa.bwd_preprocess(o4, do4, delta)
            fa.set_profile_events(e[2:5])
            bwd()
        end.record(stream)
        barrier()
    fa.set_profile_events(None)
    if fa.device_status() != 0:
        raise RuntimeError("device status not OK after the timed region")
    ms_step = shard.max_over_ranks(start.elapsed_time(end), dev) / args.steps
    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
    pre_ms = statistics.median(e[1].elapsed_time(e[2]) for e in ev)
    dkdv_ms = statistics.median(e[2].elapsed_time(e[3]) for e in ev)
    dq_ms = statistics.median(e[3].elapsed_time(e[4]) for e in ev)
    value = world * w.fwd_bwd_flops() / (ms_step * 1e-3) / 1e12
    pk = peaks()
    peak = pk["bf16_tflops"]
    dkdv_flops = (5 if fused else 4) * 2.0 * w.D * w.Hq * w.pairs()
    achieved = dkdv_flops / (dkdv_ms * 1e-3) / 1e12
    if rank == 0:
        line = {
            "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_step,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
            "dtype": w.dtype, "data": "synthetic",
            "config": {"workload": w.name, "B": w.B, "Hq": w.Hq, "Hkv": w.Hkv, "Nq": w.Nq,
                       "Nk": w.Nk, "D": w.D, "causal": w.causal, "packed": w.packed,
                       "dropout_p": w.dropout_p, "parallelism": f"replicas{world}",
                       "backward": BWD_NAMES[args.bwd],
                       "dropout_decisions": (None if w.dropout_p == 0 else
                                             "drawn by the forward and again by the backward"
                                             if mask is None else
                                             "drawn by the forward, stored in a keep mask the "
                                             "backward reads"),
                       "flops": "4*D*Hq*(attended pairs), backward credited 2.5x"},
            "fwd_tflops": w.fwd_flops() / (fwd_ms * 1e-3) / 1e12, "fwd_ms": fwd_ms,
            "fwd_frac_of_peak": w.fwd_flops() / (fwd_ms * 1e-3) / 1e12 / peak,
            "fwd_bwd_frac_of_peak": value / world / peak,
            "peak_tflops": peak, "peak_source": pk["source"] + " burst bf16 (cuBLAS)",
            "kernel_ms": kernel_ms(fused, fwd_ms, pre_ms, dkdv_ms, dq_ms),
            "roofline": {"kernel": "bwd_fused" if fused else "bwd_dkdv", "bound": "tensor",
                         "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                         "frac": achieved / peak, "traffic": None},
            "clocks": clocks.summary(),
            "gpu_launches": 4 * args.steps,
            "e2e": None,
            "cpu_baseline": None,
        }
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()


def run_sweep(fa, dev, stream, steps: int, warmup: int, peak: float):
    """The sequence-length sweep over the metric's range: D = 64, H = 16,
    B*N = 16384, N = 512 .. 16384, bf16 and fp16, causal and full.  Inputs
    (4 x 32 MiB) are smaller than twice the L2, so L2 is flushed (2 x L2
    write) before every timed step and steps are timed one by one; each point
    reports the median forward and forward+backward TFLOP/s (forward 4*B*H*N^2*D
    halved when causal, backward credited 2.5x) and their fractions of the
    burst bf16 peak."""
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    flush = torch.empty(2 * l2, dtype=torch.uint8, device=dev)
    points = []
    with ClockSampler(dev.index) as clocks:
        for dt in ("bf16", "fp16"):
            for N in SWEEP_N:
                # causal and full share the seed, hence the inputs
                q, k, v, do = (t.to(dev) for t in make_inputs(sweep(N, dt, False)))
                o, dq, dk, dv = (torch.empty_like(q) for _ in range(4))
                lse = torch.empty(q.shape[:3], dtype=torch.float32, device=dev)
                delta = torch.empty_like(lse)
                for causal in (True, False):
                    w = sweep(N, dt, causal)

                    def step(ev=None):
                        if ev is not None:
                            ev[0].record(stream)
                        fa.fwd(q, k, v, o, lse, causal, w.scale)
                        if ev is not None:
                            ev[1].record(stream)
                        fa.bwd_preprocess(o, do, delta)
                        fa.bwd(q, k, v, do, lse, delta, dq, dk, dv, causal, w.scale)
                        if ev is not None:
                            ev[2].record(stream)

                    for _ in range(warmup):
                        step()
                    ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)]
                          for _ in range(steps)]
                    for e in ev:
                        flush.zero_()
                        step(e)
                    torch.cuda.synchronize(dev)
                    fwd_ms = statistics.median(e[0].elapsed_time(e[1]) for e in ev)
                    step_ms = statistics.median(e[0].elapsed_time(e[2]) for e in ev)
                    f = w.fwd_flops() / (fwd_ms * 1e-3) / 1e12
                    fb = w.fwd_bwd_flops() / (step_ms * 1e-3) / 1e12
                    points.append({"N": N, "B": w.B, "dtype": dt, "causal": causal,
                                   "fwd_tflops": f, "fwd_bwd_tflops": fb,
                                   "fwd_frac": f / peak, "fwd_bwd_frac": fb / peak,
                                   "fwd_ms": fwd_ms, "fwd_bwd_ms": step_ms})
                del q, k, v, do, o, dq, dk, dv, lse, delta
    if fa.device_status() != 0:
        raise RuntimeError("device status not OK after the sweep")
    return {"workload": "D=64 H=16 B*N=16384 (B*H*N=262144), N 512..16384, bf16 and fp16, "
                        "causal and full; inputs i.i.d. N(0,1) seed 0",
            "l2": "flushed (%d MiB write) before each timed step; median of %d steps"
                  % (2 * l2 >> 20, steps),
            "unit": "TFLOP/s", "peak_tflops": peak, "points": points,
            "clocks": clocks.summary()}


E2E_REPS = 3     # repetitions of the end-to-end loop; the median one is reported


def measure_e2e(args, w, dev, fa, fused=False):
    """Same metric through the public API with host buffers.  Every step copies
    Q, K, V, dO from pinned host memory to the device, runs the forward and
    the backward, and copies O, dQ, dK, dV back to pinned host memory.  The
    copies run on their own streams and overlap the neighbouring steps'
    compute (device tensors double-buffered, ordered by events); the timed
    region spans all K steps including every copy."""
    hq, hk, hv, hdo = (t.contiguous().pin_memory() for t in make_inputs(w))
    hin = (hq, hk, hv, hdo)
    hout = [[torch.empty(hq.shape, dtype=hq.dtype).pin_memory() for _ in range(4)] for _ in range(2)]
    din = [[torch.empty(hq.shape, dtype=hq.dtype, device=dev) for _ in range(4)] for _ in range(2)]
    dout = [[torch.empty(hq.shape, dtype=hq.dtype, device=dev) for _ in range(4)] for _ in range(2)]
    lse = [torch.empty(hq.shape[:3], dtype=torch.float32, device=dev) for _ in range(2)]
    delta = [torch.empty(hq.shape[:3], dtype=torch.float32, device=dev) for _ in range(2)]
    ws = ([torch.empty(fa.workspace_bytes(din[b][0], din[b][1], w.causal, w.scale) // 4,
                       dtype=torch.float32, device=dev) for b in range(2)] if fused else None)
    s_in, s_comp, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev = lambda: torch.cuda.Event()
    in_ready, comp_done, out_done = {}, {}, {}
    comp_ev = {}        # timed steps: events around each step's compute

    def step(i):
        b = i % 2
        with torch.cuda.stream(s_in):
            if i - 2 in comp_done:                 # compute of step i-2 read din[b]
                s_in.wait_event(comp_done[i - 2])
            if i in comp_ev:
                comp_ev[i][2].record(s_in)
            for d, h in zip(din[b], hin):
                d.copy_(h, non_blocking=True)
            if i in comp_ev:
                comp_ev[i][3].record(s_in)
            in_ready[i] = ev(); in_ready[i].record(s_in)
        with torch.cuda.stream(s_comp):
            s_comp.wait_event(in_ready[i])
            if i - 2 in out_done:                  # D2H of step i-2 read dout[b]
                s_comp.wait_event(out_done[i - 2])
            if i in comp_ev:
                comp_ev[i][0].record(s_comp)
            q, k, v, do = din[b]
            o, dq, dk, dv = dout[b]
            fa.fwd(q, k, v, o, lse[b], w.causal, w.scale)
            fa.bwd_preprocess(o, do, delta[b])
            if fused:
                fa.bwd_fused(q, k, v, do, lse[b], delta[b], dq, dk, dv, w.causal, w.scale,
                             workspace=ws[b])
            else:
                fa.bwd(q, k, v, do, lse[b], delta[b], dq, dk, dv, w.causal, w.scale)
            if i in comp_ev:
                comp_ev[i][1].record(s_comp)
            comp_done[i] = ev(); comp_done[i].record(s_comp)
        with torch.cuda.stream(s_out):
            s_out.wait_event(comp_done[i])
            if i in comp_ev:
                comp_ev[i][4].record(s_out)
            for h, d in zip(hout[b], dout[b]):
                h.copy_(d, non_blocking=True)
            if i in comp_ev:
                comp_ev[i][5].record(s_out)
            out_done[i] = ev(); out_done[i].record(s_out)

    for i in range(args.warmup):
        step(i)
    torch.cuda.synchronize(dev)
    in_ready.clear(); comp_done.clear(); out_done.clear()

    # The link alone: one step's host->device and device->host copies on the
    # same pinned buffers, nothing else running (median of five).
    def copy_ms(stream, pairs):
        a_, b_ = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a_.record(stream)
        with torch.cuda.stream(stream):
            for dst, src in pairs:
                dst.copy_(src, non_blocking=True)
        b_.record(stream)
        torch.cuda.synchronize(dev)
        return a_.elapsed_time(b_)

    h2d_ms = statistics.median(copy_ms(s_in, list(zip(din[0], hin))) for _ in range(5))
    d2h_ms = statistics.median(copy_ms(s_out, list(zip(hout[0], dout[0]))) for _ in range(5))
    # The compute alone on the same device buffers (no copy in flight).
    ca, cb = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    ca.record(s_comp)
    with torch.cuda.stream(s_comp):
        for _ in range(args.steps):
            q, k, v, do = din[0]
            o, dq, dk, dv = dout[0]
            fa.fwd(q, k, v, o, lse[0], w.causal, w.scale)
            fa.bwd_preprocess(o, do, delta[0])
            if fused:
                fa.bwd_fused(q, k, v, do, lse[0], delta[0], dq, dk, dv, w.causal, w.scale,
                             workspace=ws[0])
            else:
                fa.bwd(q, k, v, do, lse[0], delta[0], dq, dk, dv, w.causal, w.scale)
    cb.record(s_comp)
    torch.cuda.synchronize(dev)
    comp_ms = ca.elapsed_time(cb) / args.steps
    # No clock sampler here: nvidia-smi's queries stall this copy-heavy loop for
    # milliseconds at a time (measured: with 50 ms polling the compute spans
    # showed gaps of 0.8-4.6 ms and the first step started 1-6 ms late; without
    # it, no gap), so its clocks would cost the number they describe.  The
    # device-timed region, which has no copies, carries the clock record.
    # The loop runs E2E_REPS times and the median repetition is reported, with
    # every repetition's time and longest compute gap: on a machine shared with
    # other jobs a single repetition has shown one gap of ~29 ms while the host
    # had long since enqueued every step.
    reps = []
    for _ in range(E2E_REPS):
        in_ready.clear(); comp_done.clear(); out_done.clear(); comp_ev.clear()
        comp_ev.update({i: [torch.cuda.Event(enable_timing=True) for _ in range(6)]
                        for i in range(args.steps)})
        torch.cuda.synchronize(dev)
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(s_in)
        h0 = time.perf_counter()
        for i in range(args.steps):
            step(i)
        host_issue_ms = (time.perf_counter() - h0) * 1e3
        # the end event follows the last copy of every stream
        s_in.wait_stream(s_comp); s_in.wait_stream(s_out)
        end.record(s_in)
        torch.cuda.synchronize(dev)
        # compute idle between consecutive steps (0 when the copies are hidden)
        idle = [comp_ev[i][1].elapsed_time(comp_ev[i + 1][0]) for i in range(args.steps - 1)]
        reps.append({
            "ms": start.elapsed_time(end) / args.steps,
            "idle_med": statistics.median(idle) if idle else 0.0,
            "idle_max": max(idle) if idle else 0.0,
            "fill": start.elapsed_time(comp_ev[0][0]),
            "drain": comp_ev[args.steps - 1][1].elapsed_time(end),
            "host": host_issue_ms,
            "comp": statistics.median(e[0].elapsed_time(e[1]) for e in comp_ev.values()),
            "h2d": statistics.median(e[2].elapsed_time(e[3]) for e in comp_ev.values()),
            "d2h": statistics.median(e[4].elapsed_time(e[5]) for e in comp_ev.values()),
        })
    rep = sorted(reps, key=lambda r: r["ms"])[len(reps) // 2]
    ms = rep["ms"]
    world = int(os.environ.get("WORLD_SIZE", "1"))
    nbytes = hq.numel() * hq.element_size()
    return {"value": world * w.fwd_bwd_flops() / (ms * 1e-3) / 1e12, "unit": "TFLOP/s",
            "ms_per_step": ms, "h2d_bytes_per_step": 4 * nbytes, "d2h_bytes_per_step": 4 * nbytes,
            "overlap": "copies on separate streams, double-buffered",
            "link": {"h2d_ms": h2d_ms, "d2h_ms": d2h_ms,
                     "h2d_gbs": 4 * nbytes / (h2d_ms * 1e-3) / 1e9,
                     "d2h_gbs": 4 * nbytes / (d2h_ms * 1e-3) / 1e9,
                     "compute_alone_ms": comp_ms,
                     "compute_during_copies_ms": rep["comp"],
                     "h2d_during_compute_ms": rep["h2d"],
                     "d2h_during_compute_ms": rep["d2h"],
                     "compute_idle_between_steps_ms": rep["idle_med"],
                     "compute_idle_max_ms": rep["idle_max"],
                     "fill_ms": rep["fill"],
                     "drain_ms": rep["drain"],
                     "host_issue_ms": rep["host"],
                     "repetitions_ms_per_step": [r["ms"] for r in reps],
                     "repetitions_compute_idle_max_ms": [r["idle_max"] for r in reps],
                     "clocks": "not sampled in this region (nvidia-smi polling stalls its "
                               "copies); see the line's clocks",
                     "bound_ms": max(comp_ms, h2d_ms, d2h_ms),
                     "note": "each direction's copies alone on the step's pinned buffers; "
                             "compute alone on the same device buffers; with full overlap "
                             "a step takes max of the three; the *_during_* times and the compute "
                             "idle between steps are medians over the timed end-to-end steps "
                             "(compute_idle_max_ms the longest gap) of the median repetition of "
                             "E2E_REPS, whose times are listed; fill_ms / drain_ms: start to "
                             "the first step's compute, last step's compute to the end; "
                             "host_issue_ms is the host time to enqueue all timed steps"}}


if __name__ == "__main__":
    main()
