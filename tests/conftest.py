import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")


# q8(h) codes that came out one step away from the oracle's at a provable rounding
# ambiguity, per parity case: {case: [codes that differ, codes compared]}. Printed at the
# end of the run, and written as JSON to $COLIBRI_FLIP_REPORT when that is set.
_FLIPS = {}


@pytest.fixture
def flip_report(request):
    def record(n_diff, n_codes):
        _FLIPS[request.node.nodeid] = [int(n_diff), int(n_codes)]
        # a drift guard well above what rounding ambiguities produce; each differing code
        # is also checked to sit at an ambiguity by the caller
        assert n_diff <= 1e-2 * max(n_codes, 1), (n_diff, n_codes)
    return record


def pytest_terminal_summary(terminalreporter):
    if not _FLIPS:
        return
    terminalreporter.write_sep("-", "q8(h) codes one step from the oracle's (rounding ambiguities)")
    for k, (n, tot) in sorted(_FLIPS.items()):
        terminalreporter.write_line(f"{n:6d} of {tot:10d}  {k}")
    path = os.environ.get("COLIBRI_FLIP_REPORT")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(_FLIPS, f, indent=1, sort_keys=True)


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle
