import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_sessionstart(session):
    # Every test module imports the package, which loads libqgemv.so, at
    # collection; a fresh checkout has not built it (nor the C oracle) yet.
    # The build is incremental: a no-op when both are up to date.
    import __graft_entry__
    __graft_entry__.build()


def load_golden(name):
    """Parse a tests/golden/*.txt fixture into a dict of strings."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, val = line.partition(":")
            out[key.strip()] = val.strip()
    return out
