import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 (sm_103a) GPU")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    import parity_report
    rows = parity_report.lines()
    if rows:
        terminalreporter.section("parity figures (GPU vs oracle)")
        for r in rows:
            terminalreporter.write_line(r)
