import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionfinish(session, exitstatus):
    """With MLA_PARITY_MARGINS=<file>, write the achieved parity margins of
    this session (one record per comparison) as JSON."""
    path = os.environ.get("MLA_PARITY_MARGINS")
    if not path:
        return
    import json
    from tests import parity
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "w") as f:
        json.dump(parity.MARGINS, f, indent=1)
