import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


@pytest.fixture(scope="session")
def oracle():
    from oracle import oracle as _o

    return _o.get()


@pytest.fixture(autouse=True)
def _name_band_checks(request):
    """Tags the BF16 tolerance checks of the GPU helpers with the running test."""
    g = sys.modules.get("gpu_util")
    if g is not None:
        g.CURRENT_TEST[0] = request.node.nodeid
    yield


def pytest_terminal_summary(terminalreporter):
    """How many BF16 elements of each check needed the FP32 band (beyond 1 ulp of the oracle)."""
    g = sys.modules.get("gpu_util")
    if g is None or not g.BAND_LOG:
        return
    tr = terminalreporter
    tr.section("BF16 checks: elements beyond 1 ulp of the oracle that lie in the FP32 band")
    total = sum(n for _, _, _, n in g.BAND_LOG)
    compared = sum(c for _, _, c, _ in g.BAND_LOG)
    tr.write_line(f"{len(g.BAND_LOG)} checks, {compared} elements compared, {total} took the band")
    for test, name, c, n in g.BAND_LOG:
        if n:
            tr.write_line(f"  {test} {name}: {n} of {c}")
