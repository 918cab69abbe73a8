import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


def pytest_terminal_summary(terminalreporter):
    """Error margins of the parity comparisons (relative Frobenius and max-abs against the
    bars 1e-2 and 5e-2), largest relative error last, so the end of the output shows the
    cases nearest the bar."""
    mc = sys.modules.get("tests.mla_cases")
    rows = getattr(mc, "MARGINS", None) if mc else None
    if not rows:
        return
    tr = terminalreporter
    tr.section("parity margins (bar: rel_fro 1.0e-02, max_abs 5.0e-02)")
    for test, what, rel, mx in sorted(rows, key=lambda r: r[2]):
        tr.write_line(f"rel_fro {rel:.2e} ({rel / 1e-2:5.1%} of bar)  max_abs {mx:.2e} "
                      f"({mx / 5e-2:5.1%})  {test}: {what}")
