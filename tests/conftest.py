import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """Print the argmax agreement of every parity check that recorded one."""
    try:
        from helpers import ARGMAX_LOG, format_argmax_log
    except ImportError:
        return
    if ARGMAX_LOG:
        for line in format_argmax_log(ARGMAX_LOG):
            terminalreporter.write_line(line)
