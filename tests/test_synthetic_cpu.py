"""The seeded input recipe on the CPU: the workloads' sizes, determinism per
seed, N(0, 1) elements rounded to E4M3FN (no NaN code, never saturated),
scale codes 127 + e with e uniform over the workload's range, the 1 % of
exact zeros in x of the N=7168 workloads, and the sweep's sign structure
(x rows in +/- pairs with equal scales, duplicated W rows, all +0 and all -0
W rows)."""
import numpy as np
import torch

import synthetic


def _decode(codes):
    return torch.from_numpy(codes.copy()).view(torch.float8_e4m3fn).to(torch.float64).numpy()


def test_workload_sizes_and_weight_bytes():
    got = {w.name: (w.n, w.k, w.m, w.split_k, w.exp_lo, w.exp_hi, w.x_zero_fraction)
           for w in (synthetic.TINY, synthetic.CHAIN_4096, synthetic.GRAPH_8192, synthetic.HEADLINE)}
    assert list(got.values()) == [(256, 256, 1, 1, -3, 3, 0.0), (4096, 4096, 4, 1, -4, 2, 0.0),
                                  (7168, 8192, 8, 2, -4, 2, 0.01), (7168, 16384, 8, 4, -4, 2, 0.01)]
    assert synthetic.HEADLINE.weight_bytes == 121_110_528  # N*K + N*K/32
    assert synthetic.GRAPH_8192.weight_bytes == 60_555_264
    assert synthetic.CHAIN_4096.weight_bytes == 17_301_504
    cases = {(m, n, k, s) for m in synthetic.SWEEP_M for n in synthetic.SWEEP_N
             for k in synthetic.SWEEP_K for s in synthetic.SWEEP_S}
    assert len(cases) == 288
    seeds = {synthetic.sweep_workload(*c).seed for c in cases}
    assert len(seeds) == 288  # every sweep case draws its own operands


def test_draws_are_deterministic_per_seed_and_salt():
    wl = synthetic.Workload("det", 256, 512, 4, exp_lo=-4, exp_hi=2, seed=77)
    a, b = synthetic.make_weights(wl), synthetic.make_weights(wl)
    assert all((p == q).all() for p, q in zip(a, b))
    x0, x0b, x1 = (synthetic.make_activations(wl), synthetic.make_activations(wl),
                   synthetic.make_activations(wl, salt=1))
    assert (x0[0] == x0b[0]).all() and (x0[1] == x0b[1]).all()
    assert (x0[0] != x1[0]).any()
    other = synthetic.make_weights(synthetic.Workload("det", 256, 512, 4, seed=78))
    assert (other[0] != a[0]).any()


def test_elements_are_normal_samples_in_e4m3():
    wl = synthetic.Workload("dist", 1024, 1024, 8, exp_lo=-4, exp_hi=2, seed=5)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    for codes in (w, x):
        assert codes.dtype == np.uint8
        assert not ((codes & 0x7F) == 0x7F).any()  # no NaN code
        v = _decode(codes)
        assert np.abs(v).max() < 8.0  # far from the 448 saturation point
    v = _decode(w)
    assert abs(v.mean()) < 0.01 and abs(v.std() - 1.0) < 0.02
    assert abs((v > 0).mean() - 0.5) < 0.01
    for codes, lo, hi in ((ws, -4, 2), (xs, -4, 2)):
        assert codes.min() == 127 + lo and codes.max() == 127 + hi
    counts = np.bincount(ws.ravel().astype(np.int64) - 123, minlength=7)
    assert (np.abs(counts / counts.sum() - 1 / 7) < 0.01).all()  # uniform exponents


def test_exact_zeros_in_x_of_the_large_workloads():
    wl = synthetic.GRAPH_8192
    x, _ = synthetic.make_activations(wl)
    zeros = (x == 0x00).mean()
    natural = (synthetic.make_activations(synthetic.Workload("nz", wl.n, wl.k, wl.m,
                                                             seed=wl.seed))[0] == 0x00).mean()
    assert natural < 0.002 and 0.009 < zeros - natural < 0.0115
    assert not (x == 0x80).any() or (x == 0x80).mean() < 0.002  # the planted zeros are +0


def test_sweep_sign_structure():
    wl = synthetic.sweep_workload(7, 2048, 2048, 2)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    assert wl.exp_lo == -6 and wl.exp_hi == 3 and wl.signed_pairs
    for row in range(1, 7, 2):
        assert (x[row] == x[row - 1] ^ 0x80).all() and (xs[row] == xs[row - 1]).all()
    assert (x[6] != x[5] ^ 0x80).any()  # m odd: the last row is unpaired
    for base in range(0, wl.n - 1, 16):
        assert (w[base + 1] == w[base]).all() and (ws[base + 1] == ws[base]).all()
    assert (w[3::64] == 0x00).all() and (w[5::64] == 0x80).all()


def test_integer_operands_are_small_integers_with_unit_or_double_scales():
    w, ws, x, xs = synthetic.integer_operands(128, 256, 3, seed=4)
    for codes in (w, x):
        v = _decode(codes)
        assert (v == np.round(v)).all() and np.abs(v).max() <= 8
    assert set(np.unique(ws)) <= {127, 128} and set(np.unique(xs)) <= {127, 128}
