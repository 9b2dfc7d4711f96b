import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libmla")


def pytest_collection_modifyitems(config, items):
    # GPU tests fail loudly (not skip) when CUDA is missing on a run that selected them,
    # except when running the CPU suite, where they are deselected by `-m "not gpu"`.
    pass
