import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


@pytest.fixture(scope="session")
def oracle():
    import oracle as orc
    orc.lib()  # builds the C oracle on first use
    return orc


@pytest.fixture(scope="session")
def w8a8():
    """The CUDA library binding; built if missing, and required to load."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from w8a8_int8_linear_gb300 import build as b
    b.build()
    import w8a8_int8_linear_gb300 as w
    w.lib()
    return w
