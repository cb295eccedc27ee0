"""bench.py on the CPU: the reference arm (the fp64 oracle timed on the host
cores) prints one JSON line with the contract's keys, general workloads have
no reference arm, and the workload catalogue names every configuration."""

from __future__ import annotations

import json
import os
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402


def _run(*args):
    r = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), *args],
                       capture_output=True, text=True, timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [ln for ln in r.stdout.splitlines() if ln.startswith("{")]
    assert len(lines) == 1, r.stdout
    return json.loads(lines[0])


def test_reference_arm_line():
    d = _run("--impl", "reference", "--workload", "tiny-fp32-B1-H2-N128-D64",
             "--steps", "2", "--warmup", "1")
    for key in ("metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config",
                "cpu_baseline", "e2e"):
        assert key in d, key
    assert d["impl"] == "reference" and d["unit"] == "TFLOP/s" and d["value"] > 0
    assert d["warmup"] >= 3                      # the contract's minimum is enforced
    assert d["config"]["workload"] == "tiny-fp32-B1-H2-N128-D64"
    assert d["cpu_baseline"]["kind"] == "oracle" and d["cpu_baseline"]["cores"] >= 1
    assert d["cpu_baseline"]["value"] == d["value"]
    assert d["e2e"]["h2d_bytes_per_step"] == 0 and d["e2e"]["d2h_bytes_per_step"] == 0
    assert d["vs_baseline"] is None and d["higher_is_better"] is True


def test_general_workloads_have_no_reference_arm():
    d = _run("--impl", "reference", "--workload", "gqa-bf16-B1-Hq32-Hkv8-N16384-D128-causal",
             "--steps", "1", "--warmup", "3")
    assert d["impl"] == "reference" and "unavailable" in d


def test_workload_catalogue():
    ws = bench.workloads()
    assert bench.LONG_CAUSAL.name in ws and "tiny-fp32-B1-H2-N128-D64" in ws
    for causal in ("causal", "full"):
        assert f"bf16-B4-H16-N1024-D64-{causal}" in ws
        for N in (512, 1024, 2048, 4096, 8192, 16384):
            for dt in ("bf16", "fp16"):
                assert f"sweep-{dt}-B{16384 // N}-H16-N{N}-D64-{causal}" in ws
    cover = [n for n in ws if n.startswith("cover")]
    assert len(cover) == 48
    for g in bench.BENCH_GENERAL:
        assert g.name in ws


@pytest.mark.parametrize("fused", [False, True])
def test_kernel_time_names(fused):
    k = bench.kernel_ms(fused, 1.0, 2.0, 3.0, 4.0)
    assert list(k.values()) == [1.0, 2.0, 3.0, 4.0]
    assert ("bwd_fused" in k) == fused and ("bwd_dkdv" in k) == (not fused)
