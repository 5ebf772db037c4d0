import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libnt.so")
    config.addinivalue_line("markers", "slow: full-size workload; minutes of CPU oracle time")


@pytest.fixture(scope="session")
def golden_blocks():
    import json
    with open(os.path.join(ROOT, "tests", "golden", "blocks.json")) as f:
        return {b["fmt"]: b for b in json.load(f)["blocks"]}
