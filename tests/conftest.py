import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running full-size parity case")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


def read_golden(path):
    """Rows of a ';'-separated golden fixture, comments and blanks skipped."""
    rows = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([c.strip() for c in line.split(";")])
    return rows


def pytest_terminal_summary(terminalreporter):
    """Print the achieved error ratios of the fp32 / TF32 checks and of the
    MXFP8 parity checks (max
    |gpu - ref| / max |ref| against the oracle with the same quantization,
    relative Frobenius error against the unquantized oracle) when any were
    recorded."""
    try:
        from tests import harness
    except ImportError:
        return
    tr = terminalreporter
    if harness.TF32_RATIOS:
        tr.write_line("fp32 path on TF32 tensor cores: max|gpu-ref|/max|ref| against the fp64 "
                      "oracle (bound 1e-2 + 1e-3/max|ref|):")
        for name, r in harness.TF32_RATIOS:
            tr.write_line(f"  {name}: {r:.2e}")
        tr.write_line(f"  worst: {max(r for _, r in harness.TF32_RATIOS):.2e}")
    if not harness.MX_RATIOS:
        return
    tr.write_line("MXFP8 parity: max|gpu-ref|/max|ref| against the oracle with the same "
                  "quantization (bound 1e-2) / relative Frobenius error against the "
                  "unquantized oracle (bound 1e-1):")
    worst_m = max(r[1] for r in harness.MX_RATIOS)
    worst_u = max((r[2] for r in harness.MX_RATIOS if r[2] is not None), default=None)
    for name, r_m, r_u in harness.MX_RATIOS:
        tr.write_line(f"  {name}: {r_m:.2e}" + (f" / {r_u:.2e}" if r_u is not None else ""))
    tr.write_line(f"  worst: {worst_m:.2e}" + (f" / {worst_u:.2e}" if worst_u is not None else ""))
