"""The binding's tensor checks, on the CPU: the kernels take plain pointers
and read or write rows x columns elements from them, so the binding refuses a
tensor of the wrong element size or shape before any call, where its size is
still known (a CPU tensor of the right shape is refused for not being on the
device)."""
import pytest
import torch

from mxfp8_gemm_mailbox_gb300.api import _codes, _halves


def test_codes_checks_element_size_shape_rows_and_device():
    with pytest.raises(TypeError, match="one-byte"):
        _codes(torch.zeros((2, 64), dtype=torch.int16), "x", 64)
    for bad in (torch.zeros(64, dtype=torch.uint8), torch.zeros((2, 32), dtype=torch.uint8),
                torch.zeros((2, 64, 1), dtype=torch.uint8)):
        with pytest.raises(ValueError, match=r"x must be \[rows >= 0\]\[64\]"):
            _codes(bad, "x", 64)
    with pytest.raises(ValueError, match=r"x_scale must be \[rows >= 3\]\[2\]"):
        _codes(torch.zeros((2, 2), dtype=torch.uint8), "x_scale", 2, min_rows=3)
    with pytest.raises(ValueError, match="CUDA"):
        _codes(torch.zeros((3, 2), dtype=torch.uint8), "x_scale", 2, min_rows=3)
    with pytest.raises(ValueError, match="CUDA"):
        _codes(torch.zeros((4, 64), dtype=torch.float8_e4m3fn), "x", 64)


def test_halves_checks_element_size_shape_rows_and_device():
    with pytest.raises(TypeError, match="two-byte"):
        _halves(torch.zeros((8, 256), dtype=torch.float32), "c", 8, 256)
    with pytest.raises(ValueError, match=r"c must be \[rows >= 8\]\[256\]"):
        _halves(torch.zeros((7, 256), dtype=torch.bfloat16), "c", 8, 256)
    with pytest.raises(ValueError, match=r"out must be \[rows >= 1\]\[256\]"):
        _halves(torch.zeros((8, 128), dtype=torch.int16), "out", 1, 256)
    for ok in (torch.zeros((8, 256), dtype=torch.bfloat16), torch.zeros((9, 256), dtype=torch.int16)):
        with pytest.raises(ValueError, match="CUDA"):
            _halves(ok, "c", 8, 256)
