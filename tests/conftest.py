import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built CUDA library")


@pytest.fixture(scope="session", autouse=True)
def _native_libraries():
    """The CUDA library, the input generator and the oracle are built once per
    session if missing or stale (nvcc cross-compiles without a GPU)."""
    import __graft_entry__
    __graft_entry__.build()


def pytest_terminal_summary(terminalreporter):
    """The tolerance maxima every parity check recorded against the oracle (max
    abs error, and max relative error over |ref| >= 0.1), for decode and for
    multi-query attention separately."""
    lib = sys.modules.get("pa_testlib")
    log = getattr(lib, "GATE_LOG", None) if lib is not None else None
    if not log:
        return
    tr = terminalreporter
    tr.write_sep("-", "tolerance vs the oracle")
    for kind in ("decode", "prefill"):
        rows = [r for r in log if r[4] == kind]
        if not rows:
            continue
        n_el = sum(r[1] for r in rows)
        wa = max(rows, key=lambda r: r[2])
        wr = max(rows, key=lambda r: r[3])
        tr.write_line(f"{kind}: {len(rows)} checks, {n_el} outputs compared element by element")
        tr.write_line(f"  max abs err {wa[2]:.3e} (bound 2e-3 below |ref| = 4) in '{wa[0]}'")
        tr.write_line(f"  max rel err {wr[3]:.3e} (bound 1e-2, |ref| >= 0.1) in '{wr[0]}'")
    if tr.config.getoption("verbose") > 0:
        for what, n, a, r, kind in log:
            tr.write_line(f"  [{kind}] {what}: {n} outputs, max abs {a:.3e}, max rel {r:.3e}")
