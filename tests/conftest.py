import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_100/sm_103) and the built library")


def pytest_collection_modifyitems(config, items):
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Table of the parity comparisons made in this session (GPU against the oracle)."""
    try:
        from parity_utils import REPORT
    except ImportError:
        return
    if not REPORT:
        return
    tr = terminalreporter
    tr.section("parity against the fp64 oracle")
    for r in REPORT:
        stats = "  ".join(f"{k}={v:.3g}" for k, v in r.items() if k not in ("kind", "what", "n"))
        tr.write_line(f"{r['kind']:10s} | {r['what'][:60]:60s} | n {r['n']:<9d} | {stats}")
