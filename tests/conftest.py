import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# The mutation test (test_oracle_mutations.py) reruns the oracle's pin tests
# against a copy of the oracle with one planted mistake: this variable names
# the folder holding that copy, which then shadows the real package.
_ORACLE_UNDER_TEST = os.environ.get("RSA_ORACLE_UNDER_TEST")
if _ORACLE_UNDER_TEST:
    sys.path.insert(0, _ORACLE_UNDER_TEST)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Rows of whitespace-separated fields of a golden fixture, comments dropped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(autouse=True)
def _debug_build_bounds_checks(request):
    """Under RSA_DEBUG=1 (the library's bounds-checked build), every GPU test
    ends by reading the device error word, so that a failed bounds check
    anywhere in it fails the test."""
    yield
    if os.environ.get("RSA_DEBUG", "0") in ("", "0") or request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if torch.cuda.is_available():
        import context_attention_rsa_gb300 as rsa
        rsa.check_device_error()
