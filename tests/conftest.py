import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HERE = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, HERE):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(autouse=True)
def _name_parity_records(request):
    import _util
    _util.CURRENT_TEST[0] = request.node.nodeid
    yield


def pytest_terminal_summary(terminalreporter):
    """Every parity check's raw max-abs error (over RMS) against its bound."""
    import _util
    if not _util.RECORDS:
        return
    tr = terminalreporter
    tr.section("parity: raw max-abs error / RMS vs bound (storage-adjusted diagnostic)")
    worst = max(_util.RECORDS, key=lambda r: r[2] / r[4])
    for test, what, raw, adj, tol in _util.RECORDS:
        tr.write_line(f"{raw:10.3e} {adj:10.3e}  tol {tol:.0e}  {raw / tol:6.3f} of bound  "
                      f"{test.split('::', 1)[-1]} [{what}]")
    tr.write_line(f"checks: {len(_util.RECORDS)}; largest fraction of its bound: "
                  f"{worst[2] / worst[4]:.3f} ({worst[0].split('::', 1)[-1]} [{worst[1]}])")
