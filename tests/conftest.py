import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_sessionstart(session):
    """GPU runs build the CUDA library first (it is never shipped prebuilt)."""
    if session.config.getoption("-m", default="") == "gpu":
        import __graft_entry__
        __graft_entry__.build()


def pytest_sessionfinish(session, exitstatus):
    """Write the largest errors the GPU parity tests saw, if asked to."""
    path = os.environ.get("ATTN_PARITY_REPORT")
    if not path:
        return
    try:
        from gpu_common import REPORT
    except ImportError:
        return
    if REPORT:
        import json
        with open(path, "w") as f:
            json.dump(REPORT, f, indent=1, sort_keys=True)
