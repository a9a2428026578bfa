import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a device: skip them (they are run on a B300 with -m gpu).
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    # the measured parity errors closest to their bars (error / bar), so that a run's log shows the
    # margin and which case sits nearest the bar
    try:
        from helpers import RECORD
    except Exception:  # pragma: no cover
        return
    if not RECORD:
        return
    worst = {}
    for test, what, err, tol in RECORD:
        key = (test, what.split(" ")[0])
        if key not in worst or err / tol > worst[key][0] / worst[key][1]:
            worst[key] = (err, tol)
    rows = sorted(worst.items(), key=lambda kv: -kv[1][0] / kv[1][1])
    tr = terminalreporter
    tr.write_sep("-", f"parity margins: {len(RECORD)} checked comparisons, the closest to the bar last")
    for (test, what), (err, tol) in reversed(rows[:15]):
        tr.write_line(f"{err / tol:6.3f} of bar  err {err:.3e}  bar {tol:.0e}  {what:2s} {test}")
