import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def load_constants():
    """Parse tests/golden/anvil_constants.txt (values typed from the page)."""
    path = os.path.join(ROOT, "tests", "golden", "anvil_constants.txt")
    maps, consts = [], {}
    with open(path) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            if parts[0] == "map":
                maps.append(tuple(float(x) for x in parts[1:]))
            else:
                consts[parts[0]] = float(parts[1])
    return maps, consts


@pytest.fixture(scope="session")
def constants():
    return load_constants()
