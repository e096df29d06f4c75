import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: oracle runs of several seconds or more")


def golden(name):
    """Parse a tests/golden/*.txt fixture: '#' lines are the citation, other
    lines are 'key value [value ...]'.  Repeated keys accumulate."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            vals = [float(v) for v in vals]
            out.setdefault(key, []).append(vals if len(vals) != 1 else vals[0])
    return {k: (v[0] if len(v) == 1 else v) for k, v in out.items()}


@pytest.fixture
def gold():
    return golden
