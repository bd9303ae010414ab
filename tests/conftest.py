import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Parse a tests/golden/*.txt fixture: 'key = value' lines, '#' comments."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            k, v = (s.strip() for s in line.split("=", 1))
            parts = v.split()
            vals = [float(p) if any(c in p for c in ".e") else int(p) for p in parts]
            out[k] = vals[0] if len(vals) == 1 else vals
    return out


@pytest.fixture
def golden():
    return read_golden


@pytest.fixture(scope="session")
def qmm():
    """Build libqmm.so (no-op when current) and return the Python binding."""
    from quantized_matmul_qmm_gb300 import build as _build
    _build.build()
    import quantized_matmul_qmm_gb300.qmm as q
    return q


@pytest.fixture(scope="session")
def cuda(qmm):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a CUDA GPU is required for tests marked gpu")
    return torch.device("cuda:0")
