import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA library")


def read_golden(name):
    """Non-comment lines of a golden fixture, split into fields."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library's Python binding, on a GPU; skips the test without one."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import nvfp4_quantized_paged_quantize_gb300 as kv

    kv.load()
    return kv
