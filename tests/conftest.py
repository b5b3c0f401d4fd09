import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_sessionfinish(session, exitstatus):
    """Write the GPU tests' per-case parity errors to $PKV_PARITY_LOG (a JSON list), when it is set."""
    path = os.environ.get("PKV_PARITY_LOG")
    if not path:
        return
    import json

    import parity_log
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "w") as f:
        json.dump(parity_log.RECORDS, f, indent=1)
