import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


def pytest_sessionstart(session):
    # rebuild the CUDA library if any source is newer than it (nvcc cross-compiles without a GPU)
    from mixture_experts_layer_96_b300 import build
    build.build()
