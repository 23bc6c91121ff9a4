import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_sessionstart(session):
    # On a GPU machine, make sure the CUDA library is built for this host
    # before the GPU tests import it (compiled objects are never shared
    # between machines).
    try:
        import torch
    except ImportError:
        return
    if torch.cuda.is_available():
        import __graft_entry__
        __graft_entry__.build()


def pytest_terminal_summary(terminalreporter):
    import parity_stats
    b = parity_stats.BF16
    if b["checked"]:
        terminalreporter.write_line(
            f"BF16 parity: {b['checked']} outputs checked, {b['within_1ulp']} within one ulp of "
            f"the correctly rounded exact value, {b['by_cancellation_clause']} accepted by the "
            f"cancellation clause only")
