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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter):
    """Worst errors of the GPU parity comparisons, against the fixed bar and
    against the derived rounding bound (err / bound <= 1 passes)."""
    mod = sys.modules.get("gpu_harness")
    log = getattr(mod, "PARITY_LOG", None) if mod else None
    if not log:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity: worst |gpu - oracle|, err / bound, slope / allowed")
    for label, dtype, st in log:
        tr.write_line(f"{label:60s} {dtype:4s} rows {st['rows']:5d}  max_abs {st['max_abs']:.3e}"
                      f"  err/bound {st['ratio']:.3f}  slope {st['slope_ratio']:.3f}")
