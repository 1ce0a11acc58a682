import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_sessionstart(session):
    # GPU test modules import the binding at collection time; make sure the
    # in-tree library exists (nvcc cross-compiles without a GPU).
    from online_kv_cache_02_gb300 import build as b
    if not os.path.exists(b.LIB):
        b.build()
