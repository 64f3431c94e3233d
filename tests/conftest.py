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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (run with -m gpu)")
    config.addinivalue_line("markers", "slow: long CPU test")


def pytest_terminal_summary(terminalreporter):
    # how many units of the step-level parity checks took the tie path (their
    # GPU selection differed inside the tie band, and the oracle's union,
    # gather and attention were re-run on the GPU's own selection)
    import dd_testlib as tl
    t = tl.TIE_TALLY
    if t["checks"]:
        terminalreporter.write_line(
            f"tie path: {t['tie_units']} of {t['units']} (request, KV head) units in {t['checks']} step checks "
            f"({t['tie_rows']} selection rows inside the tie band); every unit's union, miss list, "
            f"staging bytes and attention compared")
