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


@pytest.fixture(scope="session")
def hp():
    """The CUDA library binding, built in-tree for sm_103a if it is stale."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    from paged_kv_cache_hp_gb300 import build, hp as binding
    build.build()
    binding.lib()
    return binding


def guarded(nbytes, device="cuda", guard=256, fill=0xEE):
    """A byte buffer with `guard` bytes of `fill` on both sides of an nbytes window;
    returns (buffer, window)."""
    import torch
    buf = torch.full((guard + nbytes + guard,), fill, dtype=torch.uint8, device=device)
    return buf, buf[guard:guard + nbytes]


def guards_intact(buf, nbytes, guard=256, fill=0xEE):
    b = buf.cpu().numpy()
    return bool((b[:guard] == fill).all() and (b[guard + nbytes:] == fill).all())
