import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running case")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Error against the derived bound for every comparison of the inputs
    scaled by 4 (recorded by parity.py), worst ratio first."""
    mod = sys.modules.get("parity")
    rows = getattr(mod, "REPORT", None) if mod is not None else None
    if not rows:
        return
    worst = {}
    for case, key, err, bound, ratio, plain in rows:
        if (case, key) not in worst or ratio > worst[(case, key)][2]:
            worst[(case, key)] = (err, bound, ratio, plain)
    tr = terminalreporter
    tr.section("x4 inputs: max error / derived bound (bound = max(spec tol, 4 x emulation error))")
    n_plain = sum(1 for v in worst.values() if v[3])
    tr.write_line(f"{len(worst)} (case, tensor) pairs; {n_plain} also within the plain spec "
                  f"tolerance; worst ratio {max(v[2] for v in worst.values()):.3f}")
    for (case, key), (err, bound, ratio, plain) in sorted(worst.items(), key=lambda x: -x[1][2]):
        tr.write_line(f"  {case:52s} {key:5s} err {err:.3e}  bound {bound:.3e}  "
                      f"ratio {ratio:.3f}  plain-tol {'pass' if plain else 'fail'}")
