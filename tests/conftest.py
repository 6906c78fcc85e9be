import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built extension")
    config.addinivalue_line("markers", "slow: large workload, minutes of host CPU for the oracle")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device visible")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the worst error / bound of every parity check that ran."""
    try:
        import parity_util
    except Exception:  # pragma: no cover
        return
    lines = parity_util.margin_report()
    if lines:
        terminalreporter.write_sep("-", "parity margins (error, bound, fraction of the bound)")
        for ln in lines:
            terminalreporter.write_line(ln)
