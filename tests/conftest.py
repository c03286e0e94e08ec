import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Margins of the parity comparisons (achieved error against the bound)."""
    try:
        from tests import _parity
    except Exception:  # pragma: no cover
        return
    if not _parity.RECORDS:
        return
    terminalreporter.write_sep("-", "parity margins (err / bound, 1.0 = at the bound)")
    for line in _parity.margin_summary():
        terminalreporter.write_line(line)
    path = os.environ.get("ATTN_PARITY_LOG")
    if path:
        with open(path, "w") as fh:
            for name, dt, kind, mx, mtol, mn, ntol in _parity.RECORDS:
                fh.write(f"{name}\t{dt}\t{kind}\t{mx:.3e}\t{mtol:.3e}\t{mn:.3e}\t{ntol}\n")
