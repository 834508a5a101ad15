import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_runtest_setup(item):
    if item.get_closest_marker("gpu") is not None:
        import torch

        if not torch.cuda.is_available():
            pytest.fail("GPU test run without a visible CUDA device")


def read_golden(name):
    """Parse a ``key: values`` fixture under tests/golden (``#`` lines are
    citations and comments).  Values come back as a list of floats when
    they all parse, else as the raw string."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            parts = val.split()
            try:
                out[key.strip()] = [float(p) for p in parts]
            except ValueError:
                out[key.strip()] = val.strip()
    return out


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle

    return oracle.load()
