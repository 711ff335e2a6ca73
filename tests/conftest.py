import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built fa8 library")
    config.addinivalue_line("markers", "slow: longer-running CPU test")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the error of every GPU-vs-oracle parity check against its bars (the margin per
    case), and writes them as JSON to the file named by FA8_PARITY_LOG, if set."""
    mod = sys.modules.get("parity_util")
    rows = getattr(mod, "MARGINS", None) if mod else None
    if not rows:
        return
    tr = terminalreporter
    tr.section("parity margins (error / bar; bars: max 3e-2, mean 4e-3, LSE 2e-3)")
    for r in rows:
        b = r["bars"]
        tr.write_line(f"{r['max_abs'] / b[0]:6.3f} {r['mean_abs'] / b[1]:6.3f} {r['lse_abs'] / b[2]:6.3f}  "
                      f"{r['test']} [{r['case']}, rows {r['rows']}]")
    path = os.environ.get("FA8_PARITY_LOG")
    if path:
        import json

        with open(path, "w") as f:
            json.dump(rows, f, indent=1)
