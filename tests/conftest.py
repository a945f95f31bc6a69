import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (run with -m gpu)")


def golden_lines(name):
    """Non-comment lines of a golden fixture, split on whitespace."""
    with open(os.path.join(GOLDEN, name)) as f:
        return [ln.split() for ln in f if ln.strip() and not ln.lstrip().startswith("#")]


def golden_kv(name):
    """First-token -> remaining tokens, for fixtures written as `key v1 v2 ...`."""
    return {ln[0]: ln[1:] for ln in golden_lines(name)}


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.build()
    return o
