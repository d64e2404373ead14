import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    # A GPU test that runs without a GPU fails loudly rather than silently skipping;
    # the CPU suite deselects them with -m "not gpu".
    pass


@pytest.fixture(scope="session", autouse=True)
def _built_cpu_libs():
    import oracle
    import synth
    oracle.build()
    synth.build()
