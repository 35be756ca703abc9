import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built liblla.so")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if gpu_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the achieved parity error of every GPU comparison that recorded one (relative
    Frobenius error over the checked rows, the worst row's error, their bounds), so that the
    margin to each bound is visible in the test log."""
    from parity import RECORDS
    if not RECORDS:
        return
    tr = terminalreporter
    tr.section("parity margins (GPU vs float64 oracle)")
    tr.write_line(f"{'case':64s} {'rows':>7s} {'rel_frob':>10s} {'bound':>8s} "
                  f"{'row_max':>10s} {'bound':>8s}")
    for r in RECORDS:
        tr.write_line(f"{r['case'][:64]:64s} {r['rows']:7d} {r['rel']:10.3e} {r['tol']:8.1e} "
                      f"{r['row_max']:10.3e} {r['row_tol']:8.1e}")
