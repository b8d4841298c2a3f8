import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
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
    """The tolerated deviations of every GPU-vs-oracle comparison in the run:
    accept flips (|u - p/q| < 1e-5), race near-ties and top-p boundary cases."""
    try:
        from tests import parity
    except Exception:  # pragma: no cover
        return
    t = parity.TALLY
    if t["calls"]:
        terminalreporter.write_line(
            f"parity: {t['calls']} comparisons, {t['requests']} requests, {t['exact']} exact; "
            f"tolerated: accept flips {t['accept_flips']}, race near-ties {t['race_ties']}, "
            f"top-p boundary {t['topp_boundary']}")
