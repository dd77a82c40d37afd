"""The oracle's pins catch plausible mistakes (CPU only).

Each case copies the oracle's C source to a temporary directory, plants one
mistake there (a dropped term, a wrong index or sign, a transposed operand, a
broken rounding or mailbox rule), builds it, and runs the pins of
``test_oracle`` against it: at least one pin must fail.  The committed oracle
is never modified.
"""
import subprocess
from pathlib import Path

import pytest

import oracle
import tests.test_oracle as pins
import tests.test_oracle_gather as gather_pins
import tests.test_oracle_tagged as tagged_pins

SOURCE = Path(oracle.__file__).resolve().parent / "mxfp8_oracle.c"

MUTANTS = {
    "drop the last K term": (
        "for (int kk = 0; kk < k; ++kk) sum += wv[kk] * xr[kk];",
        "for (int kk = 0; kk < k - 1; ++kk) sum += wv[kk] * xr[kk];"),
    "W scale block of 16": (
        "oracle_e8m0_value(w_scale[(size_t)col * blocks + kk / 32]);",
        "oracle_e8m0_value(w_scale[(size_t)col * blocks + kk / 16 % blocks]);"),
    "x scale of the wrong row": (
        "oracle_e8m0_value(x_scale[(size_t)t * blocks + kk / 32]);",
        "oracle_e8m0_value(x_scale[(size_t)0 * blocks + kk / 32]);"),
    "transposed activation index": (
        "xv[(size_t)t * k + kk] = oracle_e4m3_value(x[(size_t)t * k + kk]) *",
        "xv[(size_t)t * k + kk] = oracle_e4m3_value(x[(size_t)t * k + (k - 1 - kk)]) *"),
    "subtract instead of add": (
        "for (int kk = 0; kk < k; ++kk) sum += wv[kk] * xr[kk];",
        "for (int kk = 0; kk < k; ++kk) sum -= wv[kk] * xr[kk];"),
    "E4M3 bias 8": (
        "magnitude = ldexp(1.0 + (double)mantissa / 8.0, exponent - 7);",
        "magnitude = ldexp(1.0 + (double)mantissa / 8.0, exponent - 8);"),
    "E4M3 subnormal scale": (
        "magnitude = ldexp((double)mantissa / 8.0, -6);",
        "magnitude = ldexp((double)mantissa / 8.0, -7);"),
    "ties away from zero": (
        "rounded = (fmod(lower, 2.0) == 0.0) ? lower : lower + 1.0;",
        "rounded = lower + 1.0;"),
    "truncate instead of round": (
        "if (fraction > 0.5)\n    rounded = lower + 1.0;",
        "if (fraction > 2.0)\n    rounded = lower + 1.0;"),
    "keep negative zero": (
        "return half == 0x8000 ? (uint16_t)0x0000 : half;",
        "return half;"),
    "swapped halves": (
        "mailbox[((size_t)g * capacity + t) * half_n + w] = low | (high << 16);",
        "mailbox[((size_t)g * capacity + t) * half_n + w] = high | (low << 16);"),
    "no reset after consume": (
        "      mailbox[slot] = ORACLE_SENTINEL;\n",
        "\n"),
    "generation not advanced": (
        "state[0] = (g + 1) % ORACLE_GENERATIONS;",
        "state[0] = g;"),
    "active generation not handed over": (
        "  state[1] = g;\n  return ORACLE_OK;",
        "  return ORACLE_OK;"),
    "gather keeps the sentinel word": (
        "slot[i] = in[i] == ORACLE_SENTINEL ? 0u : in[i];",
        "slot[i] = in[i];"),
    "gather leaves its slot": (
        "    out[i] = slot[i];\n    slot[i] = ORACLE_SENTINEL;",
        "    out[i] = slot[i];"),
    "BF16 rounding through FP32 first": (
        "double magnitude = fabs(value);",
        "double magnitude = fabs((double)(float)value);"),
    "C rounded through FP32": (
        "for (size_t i = 0; i < (size_t)m * (size_t)n; ++i) c[i] = oracle_bf16_rne(acc[i]);",
        "for (size_t i = 0; i < (size_t)m * (size_t)n; ++i) c[i] = oracle_bf16_rne((double)(float)acc[i]);"),
    "global scale applied in FP32": (
        "c[i] = oracle_bf16_rne((double)alpha * acc[i]);",
        "c[i] = oracle_bf16_rne((double)(alpha * (float)acc[i]));"),
    "E8M0 bias 128": (
        "return ldexp(1.0, (int)code - 127);",
        "return ldexp(1.0, (int)code - 128);"),
    "E4M3 NaN code read as a number": (
        "if (exponent == 15 && mantissa == 7) return NAN;",
        "if (exponent == 16 && mantissa == 7) return NAN;"),
    "publish into the active generation": (
        "  int g = state[0];\n  if (g < 0 || g >= ORACLE_GENERATIONS) return ORACLE_ERR_STATE;\n"
        "  int half_n = n / 2;\n  for (int t = 0; t < m; ++t)\n    for (int w = 0; w < half_n; ++w) {\n"
        "      uint32_t low",
        "  int g = state[1];\n  if (g < 0 || g >= ORACLE_GENERATIONS) return ORACLE_ERR_STATE;\n"
        "  int half_n = n / 2;\n  for (int t = 0; t < m; ++t)\n    for (int w = 0; w < half_n; ++w) {\n"
        "      uint32_t low"),
    "consume swaps the halves it copies out": (
        "      out[(size_t)t * n + 2 * w] = (uint16_t)(word & 0xFFFF);\n"
        "      out[(size_t)t * n + 2 * w + 1] = (uint16_t)(word >> 16);",
        "      out[(size_t)t * n + 2 * w] = (uint16_t)(word >> 16);\n"
        "      out[(size_t)t * n + 2 * w + 1] = (uint16_t)(word & 0xFFFF);"),
    "sampled outputs read activation row 0": (
        "x + (size_t)t * k, x_scale + (size_t)t * blocks));",
        "x + (size_t)0 * k, x_scale + (size_t)0 * blocks));"),
    "global scale dropped": (
        "c[i] = oracle_bf16_rne((double)alpha * acc[i]);",
        "c[i] = oracle_bf16_rne(acc[i]);"),
    "tagged pair without its tag": (
        "      pairs[at + 1] = tag;\n",
        "      pairs[at + 1] = 1u;\n"),
    "tagged poll ignores stale tags": (
        "      if (pairs[at + 1] != tag) status = ORACLE_ERR_SENTINEL;\n",
        "\n"),
    "gather generation not advanced": (
        "  state[0] = (g + 1) % ORACLE_GENERATIONS;\n  state[1] = 0;\n  return status;",
        "  state[1] = 0;\n  return status;"),
}

PINS = [
    pins.test_e4m3_all_codes_match_torch,
    pins.test_format_code_points_golden,
    pins.test_bf16_rounding_golden,
    pins.test_clear_negative_zero,
    pins.test_gemm_worked_examples_golden,
    pins.test_gemm_rounds_the_exact_sum_once_golden,
    lambda: pins.test_gemm_matches_exact_rational_sum(128, 96, 3),
    pins.test_gemm_fp64_matches_library_matmul,
    pins.test_gemm_integer_inputs_exact,
    pins.test_gemm_constant_closed_form,
    pins.test_publish_layout_and_sanitisation,
    pins.test_chain_state_sequence_and_reset,
    pins.test_scaled_gemm_closed_forms,
    pins.test_gemm_sample_matches_full,
    gather_pins.test_gather_worked_examples_golden,
    gather_pins.test_gather_sequence_of_alternating_sizes,
    tagged_pins.test_pair_layout_and_unchanged_bits,
    tagged_pins.test_stale_tag_and_no_reset,
]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    old, new = MUTANTS[name]
    text = SOURCE.read_text()
    assert text.count(old) >= 1, f"mutation site missing: {name}"
    src = tmp_path / "mutant.c"
    src.write_text(text.replace(old, new, 1))
    lib = tmp_path / "libmutant.so"
    subprocess.run(["gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
                    str(src), "-o", str(lib), "-lm"], check=True)
    caught = []
    oracle.use_library(lib)
    try:
        for pin in PINS:
            try:
                pin()
            except (AssertionError, ValueError):
                caught.append(getattr(pin, "__name__", "pin"))
    finally:
        oracle.use_library(None)
    assert caught, f"no pin caught the mutant '{name}'"
