import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the achieved parity errors beside their bars: every full-size
    comparison, and the tightest of the others."""
    try:
        from parity import MARGINS
    except ImportError:
        return
    if not MARGINS:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity margins (achieved error / bar)")
    full = [m for m in MARGINS if m[4]]
    for what, measure, value, bar, _ in full:
        tr.write_line(f"  {what:<48s} {measure:<26s} {value:10.3e}  bar {bar:8.1e}  ({value / bar:6.3f} of bar)")
    rest = [m for m in MARGINS if not m[4]]
    if rest:
        what, measure, value, bar, _ = max(rest, key=lambda m: m[2] / m[3])
        tr.write_line(f"  tightest of {len(rest)} other comparisons: {what} {measure} {value:.3e} "
                      f"({value / bar:.3f} of bar {bar:.1e})")
