import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long CPU case")


def read_golden(name):
    """Lines of a golden fixture, comments and blank lines dropped, split on '|'."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            if line.lstrip().startswith("#") or not line.strip():
                continue
            rows.append([part.strip() for part in line.rstrip("\n").split("|")])
    return rows


ORACLE_UNDER_TEST = "W4V_ORACLE_UNDER_TEST"


@pytest.fixture(scope="session")
def oracle_mod():
    """The oracle; with W4V_ORACLE_UNDER_TEST naming a shared library, that build
    of oracle.c instead (test_oracle_mutants.py runs the pins that way)."""
    import oracle
    oracle.build()
    alt = os.environ.get(ORACLE_UNDER_TEST)
    if alt:
        oracle._use_library(alt)
    return oracle


@pytest.fixture(scope="session")
def w4v_mod():
    """The ctypes binding, with libw4v.so built for sm_103a (nvcc cross-compiles without a GPU)."""
    from speculative_decoding_verify_w4a16_gb300 import _build, w4v
    _build.build()
    w4v.load()
    return w4v


@pytest.fixture(scope="session")
def gpu(w4v_mod):
    """Skips nothing: a gpu-marked test on a machine without CUDA fails loudly."""
    import torch
    assert torch.cuda.is_available(), "gpu test needs a CUDA device"
    w4v_mod.init()
    return torch.device("cuda:0")
