import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


# Flips counted by the GPU parity tests (builder order swaps between near-tied
# prefixes; draws across a CDF boundary within the stated tolerance), reported
# in the terminal summary and as junit properties.
_FLIPS = []


@pytest.fixture
def flip_log(request, record_property):
    def add(kind: str, n: int):
        _FLIPS.append((request.node.nodeid, kind, int(n)))
        record_property("flips_" + kind, int(n))
    return add


def pytest_terminal_summary(terminalreporter):
    if not _FLIPS:
        return
    tr = terminalreporter
    tr.write_sep("-", "counted flips (GPU vs oracle, each within its stated tolerance)")
    tot = {}
    for nodeid, kind, n in _FLIPS:
        tot[kind] = tot.get(kind, 0) + n
        if n:
            tr.write_line("%-8s %3d  %s" % (kind, n, nodeid))
    tr.write_line("totals over %d checks: %s" % (
        len(_FLIPS), ", ".join("%s %d" % kv for kv in sorted(tot.items()))))
