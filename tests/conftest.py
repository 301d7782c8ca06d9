import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


def pytest_terminal_summary(terminalreporter):
    """Print how much of the output tolerance each kind of comparison used at worst."""
    helpers = sys.modules.get("helpers")
    MARGINS = getattr(helpers, "MARGINS", None)
    if not MARGINS:
        return
    terminalreporter.write_sep("-", "tolerance used: max |gpu - oracle| / (atol + rtol |oracle|)")
    for key in sorted(MARGINS):
        terminalreporter.write_line(f"{MARGINS[key]:8.4f}  {key}")
