import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def to_f64(t) -> np.ndarray:
    """Exact widening of a (possibly bf16) torch tensor to float64 NumPy."""
    return t.detach().to("cpu").double().numpy()


def bits16(t) -> np.ndarray:
    """The raw 16-bit patterns of a bf16 tensor (for bit-exact comparisons)."""
    import torch
    return t.detach().to("cpu").contiguous().view(torch.int16).numpy()


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda:0")
