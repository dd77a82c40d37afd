"""Shared pytest configuration: the ``gpu`` marker and the repo root on sys.path."""
import sys
from pathlib import Path

ROOT = Path(__file__).resolve().parents[1]
if str(ROOT) not in sys.path:
    sys.path.insert(0, str(ROOT))


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a); compares the CUDA path with the oracle")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def cuda():
    """The CUDA device, with the library built; GPU tests fail loudly without one."""
    import torch

    from mxfp8_gemm_mailbox_gb300 import build

    assert torch.cuda.is_available(), "the -m gpu tests need a CUDA GPU (sm_103a)"
    build.build()
    return torch.device("cuda")
