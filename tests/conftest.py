import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Prints the strict error figures the parity tests recorded (and writes
    them as JSON to the file ATTN_PARITY_REPORT names, if set)."""
    from tests.helpers import REPORT
    if not REPORT:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity: strict errors against the fp64 oracle")
    for e in REPORT:
        tr.write_line(
            f"{e['case']:<48} {e['kind']:<4} rows {e['rows_checked']:>8}  "
            f"O max|err| {e['o_max_abs']:.3e} (floor {e['o_floor']:g}, "
            f"{e['n_over_floor']} of {e['n_elems']} over it, worst of those "
            f"{e['max_ulps_over_floor']:.2f} ulp; gate use {e['gate_use']:.2f}; "
            f"max|O| {e['max_abs_ref']:.2f})  LSE max|err| {e['lse_max_abs']:.2e}")
    path = os.environ.get("ATTN_PARITY_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(REPORT, f, indent=1)
