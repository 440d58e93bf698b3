import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def hm():
    """The C-ABI binding, building libhm in-tree first when it is missing."""
    from head_muon_mxfp8_gb300 import _abi
    if not os.path.exists(_abi.LIB_PATH):
        from head_muon_mxfp8_gb300 import build
        build.build()
    _abi.lib()
    return _abi
