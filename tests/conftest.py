import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
TESTS = os.path.dirname(os.path.abspath(__file__))
if TESTS not in sys.path:
    sys.path.insert(0, TESTS)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (runs through the C ABI)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints every parity comparison of the session: its size, worst and mean
    errors, and how many O elements needed the one-ulp rounding escape."""
    try:
        from parity import ESCAPES
    except ImportError:
        return
    if not ESCAPES:
        return
    tr = terminalreporter
    tr.section("parity comparisons (O elements, one-ulp escapes, max|dO|, mean|dO|, max|dlse|)")
    total = sum(r[1] for r in ESCAPES)
    esc = sum(r[2] for r in ESCAPES)
    for what, n, n_esc, o_max, o_mean, l_max in ESCAPES:
        if n >= 1_000_000 or n_esc:
            tr.write_line(f"{what[:60]:60s} {n:>11d} {n_esc:>6d} {o_max:.3e} {o_mean:.3e} "
                          f"{l_max:.3e}")
    tr.write_line(f"{len(ESCAPES)} comparisons, {total} O elements, {esc} one-ulp escapes "
                  f"({esc / max(total, 1):.2e} of the elements)")
