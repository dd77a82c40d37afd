"""Seeded synthetic inputs for the MXFP8 decode projection.

This module only draws operands.  It holds none of the method's arithmetic
(no product, no rounding to BF16, no mailbox rule) and imports neither the
oracle nor the CUDA package; both of those consume what it returns.

Every operand is a uint8 array: E4M3FN element codes ``W [N][K]`` and
``x [m][K]``, and E8M0FNU scale codes ``W scales [N][K/32]`` and
``x scales [m][K/32]``, one scale per 32-element K block.  The recipe follows
the workloads the source pages' decode projection runs (low batch, m <= 8):

* elements: N(0, 1) samples rounded to E4M3FN (round-to-nearest-even; |v|
  never comes near the 448 saturation point);
* scales: code 127 + e, e an integer drawn uniformly from ``[lo, hi]``;
* optional exact zeros in x: each element independently set to +0 (code
  0x00) with probability ``x_zero_fraction``;
* optional sign structure (the sweep): x rows in +/- pairs (row 2j + 1 is row
  2j with every sign bit flipped, same scales), duplicated W rows, and W rows
  that are all +0 or all -0, so some outputs are exactly +0 or -0.

Randomness is numpy's PCG64 (``numpy.random.default_rng(seed)``).  The
encoding to E4M3FN is torch's float32 -> float8_e4m3fn conversion on the CPU.
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np


@dataclass(frozen=True)
class Workload:
    """One synthetic problem: shapes, split-K cluster size and value recipe."""

    name: str
    n: int
    k: int
    m: int
    split_k: int = 1
    capacity: int = 8
    exp_lo: int = -3
    exp_hi: int = 3
    x_zero_fraction: float = 0.0
    signed_pairs: bool = False
    seed: int = 0
    extra: dict = field(default_factory=dict)

    @property
    def weight_bytes(self) -> int:
        """Algorithmic weight-stream bytes per call: E4M3 elements plus scales."""
        return self.n * self.k + self.n * (self.k // 32)

    @property
    def flops(self) -> int:
        return 2 * self.m * self.n * self.k


# The five workloads of the decode projection (sizes from the low-batch
# output projection: 7168 output columns, K up to 16384, m <= 8).
TINY = Workload("tiny N=256 K=256 m=1 S=1", 256, 256, 1, 1, exp_lo=-3, exp_hi=3, seed=1001)
CHAIN_4096 = Workload("N=4096 K=4096 m=4 S=1", 4096, 4096, 4, 1, exp_lo=-4, exp_hi=2, seed=1002)
GRAPH_8192 = Workload("N=7168 K=8192 m=8 S=2", 7168, 8192, 8, 2, exp_lo=-4, exp_hi=2,
                      x_zero_fraction=0.01, seed=1003)
HEADLINE = Workload("N=7168 K=16384 m=8 S=4", 7168, 16384, 8, 4, exp_lo=-4, exp_hi=2,
                    x_zero_fraction=0.01, seed=1004)
WORKLOADS = {w.name: w for w in (TINY, CHAIN_4096, GRAPH_8192, HEADLINE)}

SWEEP_M = tuple(range(1, 9))
SWEEP_N = (2048, 4096, 7168)
SWEEP_K = (2048, 4096, 8192, 16384)
SWEEP_S = (1, 2, 4)


def sweep_workload(m: int, n: int, k: int, s: int) -> Workload:
    """One case of the sweep: signed x row pairs, duplicated / zero W rows,
    scale exponents in [-6, 3]."""
    seed = 2000 + ((m * 7 + SWEEP_N.index(n)) * 5 + SWEEP_K.index(k)) * 3 + SWEEP_S.index(s)
    return Workload(f"sweep m={m} N={n} K={k} S={s}", n, k, m, s, exp_lo=-6, exp_hi=3,
                    signed_pairs=True, seed=seed)


def _e4m3_codes(values: np.ndarray) -> np.ndarray:
    import torch  # CPU only; the encoding is input generation, not the method

    t = torch.from_numpy(np.ascontiguousarray(values, dtype=np.float32))
    return t.to(torch.float8_e4m3fn).view(torch.uint8).numpy().copy()


def normal_e4m3(rng: np.random.Generator, shape) -> np.ndarray:
    """E4M3FN codes of N(0, 1) samples."""
    return _e4m3_codes(rng.standard_normal(size=shape, dtype=np.float32))


def scale_codes(rng: np.random.Generator, shape, lo: int, hi: int) -> np.ndarray:
    """E8M0FNU codes 127 + e with e uniform in [lo, hi]."""
    return (127 + rng.integers(lo, hi + 1, size=shape)).astype(np.uint8)


def make_weights(wl: Workload):
    """(W [N][K], W scales [N][K/32]) for a workload."""
    rng = np.random.default_rng([wl.seed, 1])
    w = normal_e4m3(rng, (wl.n, wl.k))
    ws = scale_codes(rng, (wl.n, wl.k // 32), wl.exp_lo, wl.exp_hi)
    if wl.signed_pairs:
        # Every 16th pair of rows duplicated; some rows all +0 and some all -0.
        for base in range(0, wl.n - 1, 16):
            w[base + 1] = w[base]
            ws[base + 1] = ws[base]
        w[3::64] = 0x00
        w[5::64] = 0x80
    return w, ws


def make_activations(wl: Workload, m: int | None = None, salt: int = 0):
    """(x [m][K], x scales [m][K/32]) for a workload; ``salt`` varies the draw
    between calls of one workload."""
    m = wl.m if m is None else m
    rng = np.random.default_rng([wl.seed, 2, salt])
    x = normal_e4m3(rng, (m, wl.k))
    xs = scale_codes(rng, (m, wl.k // 32), wl.exp_lo, wl.exp_hi)
    if wl.x_zero_fraction > 0:
        x[rng.random((m, wl.k)) < wl.x_zero_fraction] = 0x00
    if wl.signed_pairs:
        for row in range(1, m, 2):
            x[row] = x[row - 1] ^ 0x80
            xs[row] = xs[row - 1]
    return x, xs


def integer_operands(n: int, k: int, m: int, seed: int, max_abs: int = 8):
    """Integer-valued operands: elements in [-max_abs, max_abs] (all exactly
    representable in E4M3FN) with scale codes 127 or 128 (x1 or x2).  With
    K <= 16384 every partial sum is an integer below 2^24, so any summation
    order in FP32 or FP64 gives the exact result."""
    rng = np.random.default_rng([seed, 3])
    wv = rng.integers(-max_abs, max_abs + 1, size=(n, k)).astype(np.float32)
    xv = rng.integers(-max_abs, max_abs + 1, size=(m, k)).astype(np.float32)
    w = _e4m3_codes(wv)
    x = _e4m3_codes(xv)
    ws = (127 + rng.integers(0, 2, size=(n, k // 32))).astype(np.uint8)
    xs = (127 + rng.integers(0, 2, size=(m, k // 32))).astype(np.uint8)
    return w, ws, x, xs
