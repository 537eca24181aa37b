import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Accuracy of every Y comparison made against the oracle: the normwise
    ratios the tolerance bounds, and the elementwise diagnostic."""
    try:
        from tests import _gpu
    except Exception:  # pragma: no cover
        return
    if not _gpu.DIAGNOSTICS:
        return
    tr = terminalreporter
    tr.section("Y against the oracle (normwise max / mean, elementwise over |Y_ref| >= 0.1 mean)")
    worst = [0.0, 0.0, 0.0]
    for what, mx, mean, el in _gpu.DIAGNOSTICS:
        tr.write_line(f"{what:60s} max {mx:.2e} mean {mean:.2e} elem {el:.2e}")
        worst = [max(worst[0], mx), max(worst[1], mean), max(worst[2], el)]
    tr.write_line(f"{len(_gpu.DIAGNOSTICS)} comparisons; worst max {worst[0]:.2e} "
                  f"mean {worst[1]:.2e} elem {worst[2]:.2e}")
