import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def oracle():
    from oracle import oracle as _o
    _o.build()
    return _o


def pytest_addoption(parser):
    parser.addoption("--parity-report", default=None,
                     help="write the full-output parity reports (JSON) to this path")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    from parity import REPORTS
    if not REPORTS:
        return
    terminalreporter.section("full-output parity against the fp64 oracle")
    for r in REPORTS:
        terminalreporter.write_line(
            "%s: %d elements, max|dO| %.3g, mean|dO| %.3g, max|dLSE| %.3g, worst row %s, "
            "|dO| histogram %s over edges %s" % (r["workload"], r["elements"], r["max_o"],
                                                  r["mean_o"], r["max_lse"], r["worst_row"],
                                                  r["hist_counts"], r["hist_edges"]))
    path = config.getoption("--parity-report")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(REPORTS, f, indent=1)

