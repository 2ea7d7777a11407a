import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def load_golden(name: str) -> dict:
    """Parse a ``key: v1 v2 ...`` fixture; '#' starts a comment line."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, vals = line.partition(":")
            out[key.strip()] = vals.split()
    return out


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def qmm():
    """The CUDA library binding; GPU tests fail loudly if it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import quantized_matmul_gb300 as q
    q.load()  # raises if libqmm.so is missing or does not load
    return q


def rel_gate(y_gpu, y_orc, absterms, tol=1e-5):
    """The f32 parity gate: every output within tol * sum_b |sumi*dw*da|, and
    max|diff| / max|y| within tol.  Returns (ok, worst_ratio, maxrel)."""
    y_gpu = np.asarray(y_gpu, np.float64)
    y_orc = np.asarray(y_orc, np.float64)
    diff = np.abs(y_gpu - y_orc)
    bound = tol * np.asarray(absterms, np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        ratio = np.where(bound > 0, diff / bound, np.where(diff > 0, np.inf, 0.0))
    worst = float(ratio.max()) if ratio.size else 0.0
    ymax = float(np.abs(y_orc).max()) if y_orc.size else 0.0
    maxrel = float(diff.max() / ymax) if ymax > 0 else float(diff.max() if diff.size else 0.0)
    return (worst <= 1.0 and maxrel <= tol), worst, maxrel
