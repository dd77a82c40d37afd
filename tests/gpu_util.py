"""Helpers shared by the GPU parity tests: device upload, BF16 tolerance."""
from __future__ import annotations

import numpy as np
import torch

import oracle

# BF16 outputs must lie within 2 BF16 ULPs of the oracle (distance in the
# ordered BF16 encoding, +0 and -0 equal), or within 1e-3 absolute where the
# oracle's magnitude is below 2^-6.
ULP_TOL = 2
ABS_TOL = 1e-3
SMALL = 2.0 ** -6


def dev(a: np.ndarray, device="cuda") -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a)).to(device)


def bits(t: torch.Tensor) -> np.ndarray:
    """uint16 BF16 bits of a CUDA/CPU tensor (bfloat16 or int16/uint16 storage)."""
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def ordered(b: np.ndarray) -> np.ndarray:
    b = b.astype(np.int64)
    return np.where(b & 0x8000, -(b & 0x7FFF), b)


def is_nan(b: np.ndarray) -> np.ndarray:
    """BF16 NaN codes: exponent all ones, mantissa not zero."""
    b = np.asarray(b, dtype=np.uint16)
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def bf16_mismatches(got: np.ndarray, want: np.ndarray) -> np.ndarray:
    """Boolean mask of positions outside the tolerance.  A NaN on either side
    is a mismatch, even beside a NaN (two NaN codes can be 0 or 1 apart in the
    ordered encoding)."""
    got = np.asarray(got, dtype=np.uint16)
    want = np.asarray(want, dtype=np.uint16)
    ulp = np.abs(ordered(got) - ordered(want))
    gv = oracle.bf16_bits_to_float(got)
    wv = oracle.bf16_bits_to_float(want)
    small_ok = (np.abs(wv) < SMALL) & (np.abs(gv - wv) <= ABS_TOL)
    return ~((ulp <= ULP_TOL) | small_ok) | is_nan(got) | is_nan(want)


def describe(got: np.ndarray, want: np.ndarray, limit: int = 8) -> str:
    bad = bf16_mismatches(got, want)
    idx = np.argwhere(bad)[:limit]
    gv = oracle.bf16_bits_to_float(got)
    wv = oracle.bf16_bits_to_float(want)
    parts = [f"{int(bad.sum())} of {bad.size} outside tolerance"]
    for i in idx:
        i = tuple(i)
        parts.append(f"{i}: got {gv[i]!r} (0x{int(got[i]):04x}) want {wv[i]!r} (0x{int(want[i]):04x})")
    return "; ".join(parts)


def assert_bf16_close(got, want, what=""):
    bad = bf16_mismatches(got, want)
    assert not bad.any(), f"{what}: {describe(got, want)}"


def mailbox_words(mb) -> np.ndarray:
    """The mailbox as uint32 words [3][capacity][n/2]."""
    w = mb.words.cpu().numpy().view(np.uint32)
    return w.reshape(oracle.GENERATIONS, mb.capacity, mb.n // 2)


def state_words(mb) -> list:
    return [int(v) for v in mb.state.cpu()]


def sanitized(c_bits: np.ndarray) -> np.ndarray:
    return np.where(c_bits == 0x8000, 0, c_bits).astype(np.uint16)


def pack_words(c_bits: np.ndarray) -> np.ndarray:
    """[m][n] BF16 bits -> [m][n/2] words, column 2w in the low half."""
    c = np.asarray(c_bits, dtype=np.uint32)
    return (c[:, 0::2] | (c[:, 1::2] << 16)).astype(np.uint32)
