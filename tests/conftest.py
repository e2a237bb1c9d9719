import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkda.so")


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


def pytest_terminal_summary(terminalreporter):
    """The fp32 parity checks' elementwise relative error (reported, not
    asserted; the asserted bound is the normwise one in parity.py)."""
    try:
        import parity
    except ImportError:  # pragma: no cover
        return
    if not parity.F32_ELEMENTWISE:
        return
    what, norm, elem = max(parity.F32_ELEMENTWISE, key=lambda r: r[2])
    terminalreporter.write_line(
        f"fp32 parity: {len(parity.F32_ELEMENTWISE)} checks; worst elementwise relative error "
        f"{elem:.3e} over |ref| > {parity.F32_ELEM_FLOOR:g} max|ref| ({what}; normwise "
        f"{norm:.3e}); asserted bound: normwise <= {parity.F32_REL:g}")
