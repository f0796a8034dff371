import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


def pytest_collection_modifyitems(config, items):
    # keep the file that must run last at the end of the collection order
    last = [it for it in items if os.path.basename(str(it.fspath)).startswith("test_zz_")]
    rest = [it for it in items if it not in last]
    items[:] = rest + last
