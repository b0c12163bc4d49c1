import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running parity case")


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
    """The literal O error of every GPU parity check: max-abs, share inside 2e-3 + half-ulp, and the count
    outside it against what an ideal kernel with the same rounding steps gives (tests/helpers.py)."""
    try:
        from helpers import O_STATS
    except Exception:  # pragma: no cover
        return
    if not O_STATS:
        return
    tr = terminalreporter
    tr.section("O parity: literal max-abs error and share inside 2e-3 + half-ulp")
    tr.write_line(f"{'check':<64} {'max_abs':>9} {'share':>10} {'outside':>8} {'ideal':>6} {'allowed':>7} {'elements':>10}")
    for what, mx, share, n_out, n_ideal, allowed, size in O_STATS:
        tr.write_line(f"{what[:64]:<64} {mx:9.2e} {share:10.7f} {n_out:8d} "
                      f"{'-' if n_ideal is None else n_ideal:>6} {'-' if allowed is None else allowed:>7} {size:10d}")
