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
