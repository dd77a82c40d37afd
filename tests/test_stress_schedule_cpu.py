"""The stress tests' schedules and per-call checks, driven through the oracle
on the CPU.

The GPU stress tests replay thousands of calls and compare every call's
output with its own expected value on the device.  Here the same schedules
run through the oracle's mailbox and all-gather at small sizes, and a stale
word is planted on the host -- a word that a previous use of the same
generation left in the slot, read in place of the call's own -- to show that:

* with the stress schedules, every planted stale word is caught by the
  per-call check (the stale candidate differs from the expected value at
  almost every position);
* with the schedule the stress tests used before (three shapes over three
  generations, the same input every call), the same plant passes the check:
  such a test cannot see the race it stresses.

It also pins the device-side tolerance check against the host-side one.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from tests import stress_schedule as ss
from tests.gpu_util import bf16_mismatches

SMALL = synthetic.Workload("stress, small", 256, 256, 8, 1, exp_lo=-4, exp_hi=2,
                           x_zero_fraction=0.01, seed=7001)


def _expected_mailbox(wl, sizes, variants):
    """Sanitised oracle output of every (m, variant) of a schedule."""
    w, ws = synthetic.make_weights(wl)
    out = {}
    for v in range(variants):
        x, xs = synthetic.make_activations(wl, salt=v)
        c = oracle.gemm_bf16(w, ws, x, xs)
        clean = np.where(c == 0x8000, 0, c).astype(np.uint16)
        for m in sizes:
            out[(m, v)] = clean[:m]
    return w, ws, out


def _run_mailbox(wl, schedule, plant_at=None):
    """Drives the schedule through the oracle mailbox (publish, then consume).
    plant_at: {call: (row, column)}: after that call's publish, the word holding
    that column is overwritten with what the same generation's slot held there
    after the last publish that wrote that row (a stale word the consumer then
    reads).  Returns the outputs."""
    w, ws = synthetic.make_weights(wl)
    acts = {}
    mb = oracle.Mailbox(wl.capacity, wl.n)
    history = {}  # (generation, row) -> the row's words as last published
    outs = []
    for i, (m, v) in enumerate(schedule):
        if v not in acts:
            acts[v] = synthetic.make_activations(wl, salt=v)
        x, xs = acts[v]
        c = oracle.gemm_bf16(w, ws, x[:m], xs[:m])
        g = int(mb.state[0])
        assert mb.publish(c) == oracle.OK
        published = mb.words[g, :m].copy()
        if plant_at and i in plant_at:
            t, col = plant_at[i]
            mb.words[g, t, col // 2] = history[(g, t)][col // 2]
        for t in range(m):
            history[(g, t)] = published[t]
        st, out = mb.consume(m)
        assert st == oracle.OK
        outs.append(out)
    return outs


def _calls_flagged(outs, schedule, expected):
    return [bool(bf16_mismatches(out, expected[key]).any()) for out, key in zip(outs, schedule)]


def test_device_tolerance_matches_the_host_one():
    rng = np.random.default_rng(3)
    want = rng.integers(0, 2**16, size=200_000).astype(np.uint16)
    near = (want.astype(np.int64) + rng.integers(-4, 5, size=want.size)) & 0xFFFF
    far = rng.integers(0, 2**16, size=want.size)
    got = np.where(rng.random(want.size) < 0.5, near, far).astype(np.uint16)
    special = np.array([0x0000, 0x8000, 0x7F80, 0xFF80, 0x7FC0, 0x7FC1, 0x3C00, 0x3C10, 0x3C11,
                        0x3C80, 0x3C83, 0x0001, 0x8001], np.uint16)
    got = np.concatenate([got, np.repeat(special, special.size)])
    want = np.concatenate([want, np.tile(special, special.size)])
    host = bf16_mismatches(got, want)
    dev = ss.bf16_mismatch_mask(torch.from_numpy(got.view(np.int16)),
                                torch.from_numpy(want.view(np.int16))).numpy()
    assert (host == dev).all()
    assert 0 < host.sum() < host.size


@pytest.mark.parametrize("sizes,variants", [((1, 3, 8), 4), ((1, 3, 8, 5), 5)])
def test_stale_candidates_differ_from_the_expected_output(sizes, variants):
    # For every call after each generation's first use, the word a stale read
    # would return lies outside the tolerance at almost every position.
    calls = 3 * ss.period(len(sizes), variants)
    schedule = ss.mailbox_schedule(calls, sizes, variants)
    _, _, expected = _expected_mailbox(SMALL, sizes, variants)
    for i, ((stale, present), key) in enumerate(zip(ss.stale_rows(schedule, expected), schedule)):
        if not present.any():
            continue
        seen = bf16_mismatches(stale[present], expected[key][present])
        assert seen.mean() > 0.95, (i, key, seen.mean())


def test_old_schedule_cannot_see_a_stale_word():
    # Three shapes, three generations, one input: the stale candidate equals
    # the expected output everywhere.
    schedule = ss.mailbox_schedule(30, (1, 3, 8), 1)
    _, _, expected = _expected_mailbox(SMALL, (1, 3, 8), 1)
    for (stale, present), key in list(zip(ss.stale_rows(schedule, expected), schedule))[3:]:
        assert present.all() and (stale == expected[key]).all()


@pytest.mark.parametrize("sizes,variants", [((1, 3, 8), 4), ((1, 3, 8, 5), 5)])
def test_planted_stale_word_is_caught(sizes, variants):
    calls = 2 * ss.period(len(sizes), variants) + 3
    schedule = ss.mailbox_schedule(calls, sizes, variants)
    _, _, expected = _expected_mailbox(SMALL, sizes, variants)
    rng = np.random.default_rng(11)
    plant = {}
    for i, ((stale, present), (m, v)) in enumerate(zip(ss.stale_rows(schedule, expected),
                                                       schedule)):
        rows = np.flatnonzero(present)
        if i < 3 or rows.size == 0:
            continue
        t = int(rng.choice(rows))
        col = int(rng.integers(0, SMALL.n))
        plant[i] = (t, col)
    assert len(plant) >= calls - 6
    clean = _run_mailbox(SMALL, schedule)
    assert not any(_calls_flagged(clean, schedule, expected))
    planted = _run_mailbox(SMALL, schedule, plant)
    flagged = _calls_flagged(planted, schedule, expected)
    # A planted word whose two halves both happen to lie within tolerance of
    # the expected ones would pass: allow a handful.
    missed = [i for i in plant if not flagged[i]]
    assert len(missed) <= max(1, len(plant) // 20), missed
    assert not any(flagged[i] for i in range(calls) if i not in plant)


def test_planted_stale_word_passes_the_old_schedule():
    schedule = ss.mailbox_schedule(30, (1, 3, 8), 1)
    _, _, expected = _expected_mailbox(SMALL, (1, 3, 8), 1)
    plant = {i: (0, (7 * i) % SMALL.n) for i in range(3, 30)}
    planted = _run_mailbox(SMALL, schedule, plant)
    assert not any(_calls_flagged(planted, schedule, expected))


def _gather_inputs(sizes, variants):
    inputs, expected = {}, {}
    ref = oracle.Gather(max(sizes))
    for nbytes in sizes:
        for v in range(variants):
            rng = np.random.default_rng([nbytes, v])
            words = rng.integers(0, 2**32, size=nbytes // 4, dtype=np.uint64).astype(np.uint32)
            words[rng.random(words.size) < 0.05] = oracle.SENTINEL
            st, out = ref(words)
            assert st == oracle.OK
            inputs[(nbytes, v)], expected[(nbytes, v)] = words, out
    return inputs, expected


def test_gather_schedule_catches_a_stale_word_and_the_old_one_does_not():
    cap = 4096
    new_sizes, new_variants = (16, 1040, cap, 48), 5
    old_sizes = (16, 1040, cap)
    for sizes, variants, should_see in ((new_sizes, new_variants, True), (old_sizes, 1, False)):
        calls = 3 * ss.period(len(sizes), variants, 3)
        schedule = ss.gather_schedule(calls, sizes, variants)
        inputs, expected = _gather_inputs(sizes, variants)
        ref = oracle.Gather(cap)
        stale = ss.stale_words(schedule, expected)
        caught = total = 0
        for i, (key, (old, present)) in enumerate(zip(schedule, stale)):
            st, out = ref(inputs[key])
            assert st == oracle.OK and (out == expected[key]).all()
            where = np.flatnonzero(present)
            if where.size == 0:
                continue
            p = int(where[i % where.size])
            out[p] = old[p]  # the consumer read a word left in the slot
            total += 1
            caught += bool((out != expected[key]).any())
        assert total >= calls - 6
        if should_see:
            assert caught >= total - max(1, total // 50), (caught, total)
        else:
            assert caught == 0
