"""Pins of the CPU oracle against things other than itself (CPU only).

Each test ties one oracle function to a library routine, a closed form, an
exact rational computation, an invariant of the protocol, or a worked example
under ``tests/golden`` (each fixture cites its passage).  The source pages are
"vllm.models.deepseek_v41.nvidia.specialized_decode.boundary.publishing_gemm"
(the MXFP8 product, rounding, negative-zero clearing and publish) and
"vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_gather" (sentinel,
generations, consume).
"""
from fractions import Fraction
from pathlib import Path

import numpy as np
import pytest
import torch

import oracle
import synthetic

GOLDEN = Path(__file__).resolve().parent / "golden"


def _rows(name):
    for line in (GOLDEN / name).read_text().splitlines():
        line = line.split("#", 1)[0].strip() if line.lstrip().startswith("#") else line.strip()
        if line:
            yield line.split()


def _same(a: float, b: float) -> bool:
    if np.isnan(a) or np.isnan(b):
        return bool(np.isnan(a) and np.isnan(b))
    return a == b and np.signbit(a) == np.signbit(b)


# --- decoding -------------------------------------------------------------

def test_e4m3_all_codes_match_torch():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float64)
    for code in range(256):
        assert _same(oracle.e4m3_value(code), float(ref[code])), hex(code)


def test_e8m0_all_codes_match_torch_and_closed_form():
    ref = torch.arange(256, dtype=torch.uint8).view(torch.float8_e8m0fnu).to(torch.float64)
    for code in range(255):
        v = oracle.e8m0_value(code)
        assert v == 2.0 ** (code - 127)
        assert v == float(ref[code]), hex(code)
    assert np.isnan(oracle.e8m0_value(0xFF))


def test_format_code_points_golden():
    for fmt, code, value in _rows("e4m3_e8m0_points.txt"):
        code = int(code, 16)
        expect = float("nan") if value == "nan" else (
            float.fromhex(value) if "p" in value else float(value))
        got = oracle.e4m3_value(code) if fmt == "e4m3" else oracle.e8m0_value(code)
        assert _same(got, expect), (fmt, hex(code), got, expect)


# --- rounding -------------------------------------------------------------

def _exact_bf16_rne(q: Fraction) -> int:
    """RNE of an exact rational to BF16 bits, by integer arithmetic on the
    rational (a different construction from the oracle's double code)."""
    if q == 0:
        return 0
    sign = 0x8000 if q < 0 else 0
    a = abs(q)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    while Fraction(2) ** (e + 1) <= a:
        e += 1
    e = max(e, -126)
    quantum = Fraction(2) ** (e - 7)
    units = a / quantum
    lo = units.numerator // units.denominator
    rem = units - lo
    if rem > Fraction(1, 2) or (rem == Fraction(1, 2) and lo % 2 == 1):
        lo += 1
    value = lo * quantum
    if value >= Fraction(2) ** 128:
        return sign | 0x7F80
    f = np.float32(float(value))  # exactly representable
    return sign | int(f.view(np.uint32) >> 16)


def test_bf16_rounding_golden():
    for value, expect, *_ in _rows("bf16_rounding.txt"):
        assert oracle.bf16_rne(float.fromhex(value)) == int(expect, 16), value


def test_bf16_rounding_matches_torch_on_float32_inputs():
    # Doubles that are exact float32 values: the single rounding equals
    # torch's float32 -> bfloat16 conversion (a library RNE).
    rng = np.random.default_rng(7)
    bits = rng.integers(0, 2**32, size=20000, dtype=np.uint64).astype(np.uint32)
    # Force a share of exact ties and of subnormals.
    bits[:2000] = (bits[:2000] & 0xFFFF0000) | 0x8000
    bits[2000:4000] &= 0x807FFFFF
    f = bits.view(np.float32)
    keep = np.isfinite(f)
    f = f[keep]
    ref = torch.from_numpy(f.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.bf16_rne(float(v)) for v in f], dtype=np.uint16)
    assert (got == ref).all()


def test_bf16_rounding_matches_exact_rationals():
    rng = np.random.default_rng(8)
    for _ in range(3000):
        mant = int(rng.integers(1, 2**53))
        exp = int(rng.integers(-190, 120))
        q = Fraction(mant) * Fraction(2) ** exp * (1 if rng.random() < 0.5 else -1)
        assert oracle.bf16_rne(float(q)) == _exact_bf16_rne(q)


def test_clear_negative_zero():
    assert oracle.clear_negative_zero(0x8000) == 0x0000
    for h in (0x0000, 0x0001, 0x7F80, 0x8001, 0xFFFF, 0x3F80, 0xBF80):
        assert oracle.clear_negative_zero(h) == h


# --- the product ----------------------------------------------------------

def _decoded(codes, scales):
    v = torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    s = np.ldexp(1.0, scales.astype(np.int64) - 127)
    return v * np.repeat(s, 32, axis=1)


def test_gemm_worked_examples_golden():
    for k, wc, wsc, xc, xsc, expect, *_ in _rows("gemm_worked.txt"):
        k = int(k)
        n, m = 128, 2
        w = np.full((n, k), int(wc, 16), np.uint8)
        ws = np.full((n, k // 32), int(wsc, 16), np.uint8)
        x = np.full((m, k), int(xc, 16), np.uint8)
        xs = np.full((m, k // 32), int(xsc, 16), np.uint8)
        c = oracle.gemm_bf16(w, ws, x, xs)
        assert (c == int(expect, 16)).all(), (k, wc, xc, hex(int(c[0, 0])))


def _terms_operands(k, w_scales, x_scales, terms, n=128, m=2):
    """W [n][k] and x [m][k] all zero but for the listed (k, w code, x code)
    elements, identical in every row, with the listed per-block scale codes."""
    w = np.zeros((n, k), np.uint8)
    x = np.zeros((m, k), np.uint8)
    for term in terms.split(","):
        kk, wc, xc = term.split(":")
        w[:, int(kk)] = int(wc, 16)
        x[:, int(kk)] = int(xc, 16)
    ws = np.tile(np.array([int(v, 16) for v in w_scales.split(",")], np.uint8), (n, 1))
    xs = np.tile(np.array([int(v, 16) for v in x_scales.split(",")], np.uint8), (m, 1))
    return w, ws, x, xs


def test_gemm_rounds_the_exact_sum_once_golden():
    """Sums just past a BF16 midpoint by less than half an FP32 ulp: the
    product and the scaled product round the exact sum once, not via FP32."""
    for k, wsc, xsc, terms, expect, expect_half, *_ in _rows("gemm_double_rounding.txt"):
        w, ws, x, xs = _terms_operands(int(k), wsc, xsc, terms)
        wd, xd = _decoded(w[:1], ws[:1])[0], _decoded(x[:1], xs[:1])[0]
        exact = sum(Fraction(float(a)) * Fraction(float(b)) for a, b in zip(wd, xd))
        assert _exact_bf16_rne(exact) == int(expect, 16)  # the fixture, from a library decode
        assert (oracle.gemm_bf16(w, ws, x, xs) == int(expect, 16)).all(), (k, terms)
        assert (oracle.gemm_bf16_scaled(w, ws, x, xs, 1.0) == int(expect, 16)).all(), (k, terms)
        assert (oracle.gemm_bf16_scaled(w, ws, x, xs, 0.5) == int(expect_half, 16)).all(), (k, terms)


@pytest.mark.parametrize("n,k,m", [(128, 32, 1), (128, 96, 3), (256, 256, 8), (128, 64, 5)])
def test_gemm_matches_exact_rational_sum(n, k, m):
    wl = synthetic.Workload("exact", n, k, m, exp_lo=-6, exp_hi=3, seed=31 + k + m)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    c = oracle.gemm_bf16(w, ws, x, xs)
    wv, xv = _decoded(w, ws), _decoded(x, xs)
    for t in range(m):
        for col in range(0, n, 7 if n > 128 else 1):
            exact = sum((Fraction(float(a)) * Fraction(float(b)) for a, b in zip(wv[col], xv[t])),
                        Fraction(0))
            assert int(c[t, col]) == _exact_bf16_rne(exact), (t, col)


def test_gemm_fp64_matches_library_matmul():
    wl = synthetic.Workload("lib", 384, 1024, 8, exp_lo=-4, exp_hi=2, seed=77)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    acc = oracle.gemm_fp64(w, ws, x, xs)
    ref = _decoded(x, xs) @ _decoded(w, ws).T
    np.testing.assert_allclose(acc, ref, rtol=1e-12, atol=1e-300)
    # and the transposed product is NOT what it computes (guards operand roles)
    assert acc.shape == (8, 384)


def test_gemm_integer_inputs_exact():
    w, ws, x, xs = synthetic.integer_operands(256, 2048, 8, seed=5)
    acc = oracle.gemm_fp64(w, ws, x, xs)
    wi = torch.from_numpy(w).view(torch.float8_e4m3fn).to(torch.float64).numpy().astype(np.int64)
    xi = torch.from_numpy(x).view(torch.float8_e4m3fn).to(torch.float64).numpy().astype(np.int64)
    wi = wi * np.repeat(1 << (ws.astype(np.int64) - 127), 32, axis=1)
    xi = xi * np.repeat(1 << (xs.astype(np.int64) - 127), 32, axis=1)
    exact = xi @ wi.T  # integer matmul: exact
    assert (acc == exact.astype(np.float64)).all()


def test_gemm_constant_closed_form():
    n, k, m = 128, 1024, 3
    for a_code, b_code, sw, sx in [(0x38, 0x40, 127, 129), (0x3c, 0xb0, 120, 131)]:
        w = np.full((n, k), a_code, np.uint8)
        ws = np.full((n, k // 32), sw, np.uint8)
        x = np.full((m, k), b_code, np.uint8)
        xs = np.full((m, k // 32), sx, np.uint8)
        acc = oracle.gemm_fp64(w, ws, x, xs)
        a = oracle.e4m3_value(a_code)
        b = oracle.e4m3_value(b_code)
        assert (acc == k * a * b * 2.0 ** (sw + sx - 254)).all()


def test_gemm_sign_pairs_and_duplicates():
    wl = synthetic.sweep_workload(6, 2048, 2048, 1)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    acc = oracle.gemm_fp64(w, ws, x, xs)
    for j in range(0, wl.m - 1, 2):
        assert (acc[j + 1] == -acc[j]).all()
    for base in range(0, wl.n - 1, 16):
        assert (acc[:, base + 1] == acc[:, base]).all()
    assert (acc[:, 3::64] == 0).all() and (acc[:, 5::64] == 0).all()


def test_gemm_sample_matches_full():
    wl = synthetic.Workload("sample", 512, 512, 5, exp_lo=-4, exp_hi=2, seed=9)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    c = oracle.gemm_bf16(w, ws, x, xs)
    rows = np.array([0, 4, 2, 3, 1], np.int32)
    cols = np.array([0, 511, 128, 7, 300], np.int32)
    assert (oracle.gemm_sample(w, ws, x, xs, rows, cols) == c[rows, cols]).all()


# --- the mailbox ----------------------------------------------------------

def _words_have_sentinel_or_negzero(words):
    lo = words & 0xFFFF
    hi = words >> 16
    return bool((words == oracle.SENTINEL).any() or (lo == 0x8000).any() or (hi == 0x8000).any())


def test_mailbox_init_is_all_sentinel():
    mb = oracle.Mailbox(8, 256)
    assert (mb.words == oracle.SENTINEL).all()
    assert list(mb.state) == [0, 0, 0, 0]


def test_publish_layout_and_sanitisation():
    mb = oracle.Mailbox(4, 16)
    c = np.arange(3 * 16, dtype=np.uint16).reshape(3, 16) + 0x3F00
    c[0, 0] = 0x8000  # negative zero, low half
    c[1, 5] = 0x8000  # negative zero, high half
    assert mb.publish(c) == oracle.OK
    g = 0
    assert list(mb.state) == [0, 0, 0, 0]  # state[1] := state[0] == 0
    for t in range(3):
        for wi in range(8):
            word = int(mb.words[g, t, wi])
            lo, hi = word & 0xFFFF, word >> 16
            assert lo == (0 if c[t, 2 * wi] == 0x8000 else c[t, 2 * wi])
            assert hi == (0 if c[t, 2 * wi + 1] == 0x8000 else c[t, 2 * wi + 1])
    assert not _words_have_sentinel_or_negzero(mb.words[g, :3])
    # rows >= m and other generations keep the sentinel
    assert (mb.words[g, 3:] == oracle.SENTINEL).all()
    assert (mb.words[1:] == oracle.SENTINEL).all()


def test_chain_state_sequence_and_reset():
    wl = synthetic.Workload("seq", 256, 128, 3, exp_lo=-3, exp_hi=3, seed=4)
    w, ws = synthetic.make_weights(wl)
    mb = oracle.Mailbox(8, 256)
    for i in range(7):
        x, xs = synthetic.make_activations(wl, m=1 + i % 3, salt=i)
        st, c, out = mb.chain(w, ws, x, xs)
        assert st == oracle.OK
        assert list(mb.state) == [(i + 1) % 3, i % 3, 0, 0]
        assert (mb.words == oracle.SENTINEL).all()
        assert (out == np.where(c == 0x8000, 0, c)).all()


def test_consume_without_publish_reports_sentinel():
    mb = oracle.Mailbox(8, 128)
    st, out = mb.consume(2)
    assert st == oracle.ERR_SENTINEL
    assert list(mb.state) == [1, 0, 0, 0]  # advances anyway, as the bounded poll does
    assert (mb.words == oracle.SENTINEL).all()


def test_bad_generation_is_rejected():
    mb = oracle.Mailbox(8, 128)
    mb.state[1] = 7
    st, _ = mb.consume(1)
    assert st == oracle.ERR_STATE
    mb.state[0] = 3
    assert mb.publish(np.zeros((1, 128), np.uint16)) == oracle.ERR_STATE


def test_scaled_gemm_closed_forms():
    # alpha = 1 is the unscaled product; a power of two scales exactly; any
    # alpha equals the rounding of alpha times the FP64 sum.
    wl = synthetic.Workload("scaled", 256, 512, 3, exp_lo=-4, exp_hi=2, seed=12)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    assert (oracle.gemm_bf16_scaled(w, ws, x, xs, 1.0) == oracle.gemm_bf16(w, ws, x, xs)).all()
    c = oracle.gemm_bf16(w, ws, x, xs)
    c4 = oracle.gemm_bf16_scaled(w, ws, x, xs, 0.25)
    v, v4 = oracle.bf16_bits_to_float(c), oracle.bf16_bits_to_float(c4)
    assert (v4 == v * 0.25).all()
    acc = oracle.gemm_fp64(w, ws, x, xs)
    a = float(np.float32(-1.7))
    want = np.array([[_exact_bf16_rne(Fraction(a) * Fraction(float(u))) for u in row] for row in acc],
                    dtype=np.uint16)
    assert (oracle.gemm_bf16_scaled(w, ws, x, xs, a) == want).all()
