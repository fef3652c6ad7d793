import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.join(ROOT, "tests")
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


def read_golden(name):
    """Parse a `key = values` fixture under tests/golden/."""
    vals = {}
    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, rhs = (s.strip() for s in line.split("=", 1))
            nums = [float(x) for x in rhs.split()]
            vals[key] = nums[0] if len(nums) == 1 else nums
    return vals


@pytest.fixture(scope="session")
def golden():
    return read_golden
