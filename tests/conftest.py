import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # GPU tests are selected with -m gpu; without a GPU they would fail loudly
    # on purpose (the library has no CPU fallback), so nothing is skipped here.
    pass
