import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU case")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library's binding; GPU tests fail loudly without it."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test collected but no CUDA device is visible")
    from video_vae_causal_gb300 import wanvae
    wanvae.load()
    return wanvae
