import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the built libkda.so")


@pytest.fixture(scope="session")
def kda_lib():
    """Build (if stale) and load the CUDA library; GPU tests depend on it."""
    from kimi_delta_attention_08_gb300 import build, _lib
    build.build()
    return _lib.load()


def pytest_terminal_summary(terminalreporter):
    """Parity margins of the run: every full-size case and the worst case overall
    (max-rel output error and final-state rel-L2 against the fp64 oracle)."""
    try:
        from tests.kda_testutil import OUT_TOL, PARITY_LOG, STATE_TOL
    except ImportError:
        return
    if not PARITY_LOG:
        return
    tr = terminalreporter
    tr.write_sep("-", f"parity vs fp64 oracle (tolerances: out {OUT_TOL:g}, state {STATE_TOL:g})")
    fmt = lambda x: "-" if x is None else f"{x:.2e}"
    for label, eo, es in PARITY_LOG:
        if label.startswith("full:"):
            tr.write_line(f"{label[5:]}: out {fmt(eo)} state {fmt(es)}")
    wo = max(PARITY_LOG, key=lambda r: r[1])
    ws = max(PARITY_LOG, key=lambda r: -1.0 if r[2] is None else r[2])
    tr.write_line(f"worst of {len(PARITY_LOG)} cases: out {fmt(wo[1])} ({wo[0]}), "
                  f"state {fmt(ws[2])} ({ws[0]})")
