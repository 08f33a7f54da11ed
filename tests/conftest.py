import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_kv(name):
    """key = value lines of a golden fixture (comments start with #)."""
    out = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            k, v = (x.strip() for x in line.split("=", 1))
            out[k] = v
    return out


def read_rows(name):
    """'|'-separated rows of a golden fixture (comments start with #)."""
    rows = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([x.strip() for x in line.split("|")])
    return rows


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library, built in-tree if needed (host code only is exercised on CPU)."""
    from paged_kv_cache_51_gb300 import _build

    _build.build()
    import paged_kv_cache_51_gb300 as pkv

    return pkv
