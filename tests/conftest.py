import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: CPU test taking more than a few seconds")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library on a GPU host; GPU tests fail (not skip) when it
    cannot be loaded, so a missing extension is never mistaken for a pass."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from gated_deltanet_prefill_gb300 import gdn2
    gdn2.load()
    return gdn2
