import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")
    config.addinivalue_line("markers", "slow: long-running check (full-size workloads)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA GPU on this machine")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Raw errors of every tolerance comparison made in this run (passing ones
    included): test, tensor, raw max-abs, max-abs beyond the output's bf16
    rounding, relative L2, and the exact value and the result at the worst
    entry."""
    try:
        from msa_testutil import RECORD
    except Exception:  # pragma: no cover
        return
    if not RECORD:
        return
    tr = terminalreporter
    tr.section("parity errors (raw)")
    for test, name, ma, ma_arith, rl, w_at, g_at in RECORD:
        tr.write_line(f"{test} | {name} | max-abs {ma:.3e} | beyond-rounding {ma_arith:.3e} | rel-L2 {rl:.3e} | "
                      f"worst entry exact {w_at:.6g} got {g_at:.6g}")
