import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) and the built CUDA library")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.build()
    return oracle


def pytest_sessionfinish(session, exitstatus):
    """Write every checked parity row to $Q3_PARITY_REPORT (JSON lines), if set."""
    path = os.environ.get("Q3_PARITY_REPORT")
    if not path:
        return
    try:
        import dataclasses
        import json
        from helpers import REPORT
    except ImportError:
        return
    with open(path, "w") as f:
        for tag, c in REPORT:
            f.write(json.dumps({"tag": tag, **dataclasses.asdict(c), "ambiguous": c.ambiguous}) + "\n")
