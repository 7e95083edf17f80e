import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libdr.so")
    config.addinivalue_line("markers", "slow: large-size case")


def pytest_terminal_summary(terminalreporter):
    """Prints the measured errors the full-size parity tests recorded."""
    import json

    try:
        from parity import ERROR_LOG
    except ImportError:
        return
    if not ERROR_LOG:
        return
    terminalreporter.write_line("measured errors (max |gpu - oracle| / RMS(oracle) unless noted):")
    for e in ERROR_LOG:
        vals = "  ".join(f"{k}={v:.3e}" for k, v in e.items() if k not in ("case", "what"))
        terminalreporter.write_line(f"  {e['case']:<44s} {e['what']:<22s} {vals}")
    path = os.environ.get("DR_ERROR_LOG")
    if path:
        with open(path, "a") as f:
            for e in ERROR_LOG:
                f.write(json.dumps(e) + "\n")
