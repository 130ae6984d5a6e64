import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def golden_lines(name):
    """Non-comment, non-empty lines of a golden fixture, split on whitespace."""
    out = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                out.append(line.split())
    return out


def golden_kv(name):
    """key -> list of values for `key v1 v2 ...` lines."""
    return {parts[0]: parts[1:] for parts in golden_lines(name)}


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle
