import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long-running full-size case")


def read_golden(name):
    """Rows of a whitespace-separated golden file, comments dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line)
    return rows


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library's binding; GPU tests only."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_mixed_precision_reduce_gb300 as fp8mp

    fp8mp.load()
    return fp8mp
