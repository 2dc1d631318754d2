import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Logit margins of the GPU parity checks: the worst max and mean
    |GPU - oracle| per check group, against the tolerance it was held to."""
    try:
        from nc_testutil import MARGINS
    except Exception:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.write_sep("-", "logit margins vs the fp64 oracle (worst over each group)")
    for group, (mx, mean, tmax, tmean, n) in sorted(MARGINS.items()):
        tr.write_line(f"{group:<44s} max {mx:.2e} (tol {tmax:g})  mean {mean:.2e} (tol {tmean:g})  checks {n}")
