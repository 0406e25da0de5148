import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")


def read_golden(name):
    """Parse a tests/golden text fixture into a list of (tag, tokens) lines."""
    path = os.path.join(ROOT, "tests", "golden", name)
    out = []
    with open(path) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            out.append(line)
    return out


# Parity figures of the GPU tests: one record per checked case (the largest
# output error relative to the largest oracle output, the oracle's near-tie
# chunks and how many of them the GPU ranked differently).  They are printed
# in the terminal summary, which `pytest -q` keeps, and written as JSON to the
# path in STILL_PARITY_JSON when that variable is set.
PARITY_RECORDS = []


def record_parity(case, **fields):
    PARITY_RECORDS.append(dict(case=case, **fields))


def pytest_terminal_summary(terminalreporter):
    if not PARITY_RECORDS:
        return
    tr = terminalreporter
    tr.write_line(f"parity records ({len(PARITY_RECORDS)} cases; err = max|y_gpu - y_ref| / max|y_ref|):")
    for r in PARITY_RECORDS:
        extra = " ".join(f"{k}={v:.3e}" if isinstance(v, float) else f"{k}={v}"
                         for k, v in r.items() if k != "case")
        tr.write_line(f"  {r['case']}: {extra}")
    path = os.environ.get("STILL_PARITY_JSON")
    if path:
        import json
        with open(path, "w") as f:
            json.dump(PARITY_RECORDS, f, indent=1)


@pytest.fixture(scope="session")
def cuda_ok():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return True
