import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Worst margin per test: max error against its bound, for every GPU parity check."""
    try:
        from gpu_common import MARGINS
    except Exception:
        return
    if not MARGINS:
        return
    worst = {}
    for test, what, err, bound in MARGINS:
        r = err / bound if bound > 0 else 0.0
        if test not in worst or r > worst[test][0]:
            worst[test] = (r, what, err, bound)
    tr = terminalreporter
    tr.write_sep("-", f"parity margins: {len(MARGINS)} checks, worst error / bound per test")
    rows = sorted(worst.items(), key=lambda x: -x[1][0])
    # the worst 20, then every full-size workload's check (the sizes the bench times)
    shown = rows[:20] + [r for r in rows[20:] if "full" in r[0] or "every_element" in r[0]]
    for test, (r, what, err, bound) in shown:
        tr.write_line(f"{r:6.3f}  {err:.3g} <= {bound:.3g}  {test} [{what}]")
    if len(rows) > len(shown):
        rest = [r for r in rows if r not in shown]
        tr.write_line(f"... {len(rest)} more tests, each at most {rest[0][1][0]:.3f} of its bound")
