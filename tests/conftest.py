import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")


def pytest_runtest_setup(item):
    parity = sys.modules.get("parity")
    if parity is not None:
        parity.CURRENT = item.nodeid


def pytest_terminal_summary(terminalreporter):
    """Print the errors of every parity comparison of the run against their
    bounds (worst fraction first on each line), so the margins are visible
    even in a quiet run."""
    parity = sys.modules.get("parity")
    if parity is None or not parity.MARGINS:
        return
    lines = parity.margin_lines()
    terminalreporter.write_sep("-", "parity margins: error (fraction of bound), %d comparisons" % len(lines))
    for line in lines:
        terminalreporter.write_line(line)
    worst = max(float(line.split()[0]) for line in lines)
    terminalreporter.write_line("largest fraction of a bound: %.2f" % worst)
