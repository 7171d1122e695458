import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (GB300, sm_103a); run with -m gpu")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """After a GPU run: per checked output set, the error-scale figure max |dy|/S (the
    acceptance bound is 1e-5) and the plain max |dy|/|y64| over outputs with |y64| >= 1e-3 S."""
    gu = sys.modules.get("gpu_util")
    rows = getattr(gu, "ERROR_REPORT", None) if gu else None
    if not rows:
        return
    tr = terminalreporter
    tr.section("output error vs the oracle (y64)")
    tr.write_line(f"{'max |dy|/S':>12} {'plain max |dy|/|y|':>19} {'outputs (|y|>=1e-3 S / all)':>28}  test")
    for label, worst, plain, counted, total in rows:
        tr.write_line(f"{worst:12.3e} {plain:19.3e} {counted:>13d} / {total:<12d}  {label}")
    tr.write_line(f"overall: max |dy|/S = {max(r[1] for r in rows):.3e}, "
                  f"plain max |dy|/|y| = {max(r[2] for r in rows):.3e} over {len(rows)} output sets")
