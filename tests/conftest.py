import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Measured errors of the long-window GPU comparisons (rel-L2 against
    their bar: 1e-3, or the split-bf16 chunked form's tighter one), one line
    per buffer, and the smallest margin of all."""
    mod = sys.modules.get("gpu_helpers")
    rows = getattr(mod, "MEASURED", None) if mod is not None else None
    if not rows:
        return
    tr = terminalreporter
    tr.section("parity errors against the oracle (long windows: rel-L2 against its bar)")
    for test, name, measure, err, bar in rows:
        if measure == "rel-L2":
            margin = f"x{bar / err:8.1f} below" if err > 0 else "   exact"
            tr.write_line(f"{err:9.2e}  {margin} bar {bar:.0e}  {name:13s} {test}")
    worst = min(rows, key=lambda r: r[4] / max(r[3], 1e-300))
    tr.write_line(f"smallest margin: {worst[3]:.2e} against {worst[4]:.0e} ({worst[2]}, {worst[1]}, "
                  f"{worst[0]})")
