import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 (sm_103a) GPU and the CUDA library")
    config.addinivalue_line("markers", "slow: long CPU oracle runs")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library, loaded through the product package (fails loudly if it
    cannot be built or loaded)."""
    import packed_resolution_diffusion_pack_b300 as mf
    mf.load()
    return mf
