import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 (sm_103a) GPU")


def pytest_sessionfinish(session, exitstatus):
    # measured parity of every comparison the GPU tests made (see tests/harness.py)
    path = os.environ.get("LACT_PARITY_LOG")
    if not path:
        return
    from tests import harness
    import json
    with open(path, "w") as f:
        json.dump(harness.RECORDS, f, indent=0)
