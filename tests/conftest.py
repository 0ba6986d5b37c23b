import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (B300, sm_103a)")


def pytest_sessionstart(session):
    # Build libfa.so in-tree if it is missing or older than its sources (nvcc
    # cross-compiles without a GPU).
    from online_softmax_14_b300.build import build_library

    build_library()
