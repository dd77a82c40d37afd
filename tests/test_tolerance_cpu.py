"""The tolerance the GPU parity tests apply to BF16 outputs, checked on the
CPU: within 2 BF16 ULPs of the oracle (distance in the ordered encoding, +0
and -0 equal), or within 1e-3 absolute where the oracle's magnitude is below
2^-6; anything else, NaN included, is a mismatch."""
import numpy as np

from tests.gpu_util import bf16_mismatches


def _bad(got, want):
    return bool(bf16_mismatches(np.array([got], np.uint16), np.array([want], np.uint16))[0])


def test_ulp_distance_in_the_ordered_encoding():
    assert not _bad(0x3F80, 0x3F80)                                # 1.0
    assert not _bad(0x3F81, 0x3F80) and not _bad(0x3F82, 0x3F80)   # 1 and 2 ULPs
    assert _bad(0x3F83, 0x3F80) and _bad(0x3F7D, 0x3F80)           # 3 ULPs either side
    assert not _bad(0x3F7E, 0x3F80)                                # 2 ULPs below, across a binade
    assert not _bad(0xC382, 0xC380) and _bad(0xC383, 0xC380)       # negative values alike
    assert not _bad(0x447C, 0x447A) and _bad(0x447D, 0x447A)       # 1008 vs 1000: 2 ULPs; 1012: 3


def test_signed_zeros_are_equal_and_zero_is_crossed_by_distance():
    assert not _bad(0x8000, 0x0000) and not _bad(0x0000, 0x8000)
    assert not _bad(0x8001, 0x0001)                                # -q vs +q: 2 ULPs apart
    assert not _bad(0x7F7F, 0x7F7F) and _bad(0x7F7F, 0xFF7F)       # largest finite vs its negative


def test_absolute_tolerance_only_below_two_to_the_minus_six():
    want = 0x3C00                                                  # 2^-7 (ULP 2^-14 there)
    assert not _bad(0x3C10, want)                                  # 16 ULPs = 9.8e-4 away
    assert _bad(0x3C11, want)                                      # 17 ULPs = 1.04e-3 away
    assert not _bad(0xBC10, 0xBC00) and _bad(0xBC11, 0xBC00)       # negative alike
    # At |want| = 2^-6 the absolute rule no longer applies: 3 ULPs (3 x 2^-13) fail.
    assert _bad(0x3C83, 0x3C80)


def test_nan_never_matches():
    assert _bad(0x7FC0, 0x3F80) and _bad(0x7FC0, 0x0000) and _bad(0x3F80, 0x7FC0)
    # not even another NaN, whose code may lie 0 or 1 apart in the ordered encoding
    assert _bad(0x7FC0, 0x7FC0) and _bad(0x7FC1, 0x7FC0) and _bad(0xFFC0, 0xFFC0)
    assert _bad(0x7F81, 0x7F80)                                    # NaN beside infinity
    assert not _bad(0x7F80, 0x7F80) and not _bad(0xFF80, 0xFF80)   # infinity is a value
