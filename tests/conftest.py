import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter):
    """Worst |gpu - ref| / bound of each GPU parity check against the oracle
    (bound = 2^-7 |ref| + 1e-3 rms(ref)); 1.0 is the tolerance's edge."""
    mod = sys.modules.get("gpu_util")
    ratios = getattr(mod, "RATIOS", None) if mod else None
    if not ratios:
        return
    worst = {}
    for test, r, n in ratios:
        w, m = worst.get(test, (0.0, 0))
        worst[test] = (max(w, r), m + n)
    tr = terminalreporter
    tr.write_sep("-", "parity against the oracle: worst |err|/bound per test")
    for test, (r, n) in sorted(worst.items(), key=lambda kv: -kv[1][0]):
        tr.write_line(f"{r:6.3f}  {n:>9d} elements  {test}")
    tr.write_line(f"overall worst {max(r for r, _ in worst.values()):.3f} over "
                  f"{sum(n for _, n in worst.values())} elements in {len(worst)} tests")
