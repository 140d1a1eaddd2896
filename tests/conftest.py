import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """Worst relative L2 error per parity case and output (the margin to the tolerance)."""
    gu = sys.modules.get("gpu_util")
    if gu is None or not gu.WORST:
        return
    rows = sorted(gu.WORST.items())
    terminalreporter.section("worst relative L2 error per case and output")
    for (case, what), err in rows:
        terminalreporter.write_line(f"{case:48s} {what:16s} {err:.3e}")
    path = os.environ.get("TTT_PARITY_LOG")
    if path:
        import json
        with open(path, "w") as f:
            json.dump([{"case": c, "output": w, "rel_l2": e} for (c, w), e in rows], f, indent=1)
