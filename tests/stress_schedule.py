"""Call schedules of the stress tests and the model of a stale word.

A Lamport slot is safe to read once no word of it is the sentinel.  A word
that a call left behind -- a reset that never happened, or a store that
landed after the slot was reset -- is not the sentinel either, so the next
call that uses the same generation can take it for its own payload (the
all-gather page, module description: a late word read by a later gather of
another size).  Such a read returns the word the slot held the last time that
generation was published: the *stale candidate* modelled here.

A per-call comparison can only see the stale read if the stale candidate
differs from what the call should return.  Cycling three shapes over three
generations with the same input every call gives every generation the same
shape and bytes on every use, so the candidate always equals the expected
value and the read is invisible.  The schedules here change the bytes (and,
for the gather and the shifting mailbox schedule, the shape) on every use of
a generation, so the candidate differs from the expected value almost
everywhere.

Nothing here computes the method's arithmetic: expected values come from the
oracle; this module only decides which input each call takes and where a
stale word would come from.
"""
from __future__ import annotations

from math import lcm

import numpy as np
import torch

GENERATIONS = 3


def period(*cycles: int) -> int:
    return lcm(*cycles)


def mailbox_schedule(calls: int, sizes, variants: int):
    """[(m, variant)] for each call: m cycles through ``sizes``, the
    activations through ``variants`` seeded inputs."""
    return [(sizes[i % len(sizes)], i % variants) for i in range(calls)]


def gather_schedule(calls: int, sizes, variants: int):
    """[(nbytes, variant)] for each call, as ``mailbox_schedule``."""
    return [(sizes[i % len(sizes)], i % variants) for i in range(calls)]


def stale_rows(schedule, expected):
    """The stale candidate of every call of a mailbox schedule.

    ``expected[(m, v)]`` is the sanitised BF16 output ``[m][N]`` of the call
    (uint16).  Returns, per call, ``(stale [m][N] uint16, present [m] bool)``:
    row t of the stale candidate is row t of the last earlier call on the same
    generation whose m covered t; ``present[t]`` is False when no earlier call
    wrote that row (the slot then only ever held the sentinel, which the poll
    would wait on)."""
    last = {}  # (generation, row) -> uint16 row
    out = []
    for i, (m, v) in enumerate(schedule):
        g = i % GENERATIONS
        want = expected[(m, v)]
        stale = np.zeros_like(want)
        present = np.zeros(m, dtype=bool)
        for t in range(m):
            if (g, t) in last:
                stale[t] = last[(g, t)]
                present[t] = True
        out.append((stale, present))
        for t in range(m):
            last[(g, t)] = want[t]
    return out


def stale_words(schedule, expected):
    """The stale candidate of every call of a gather schedule: per call
    ``(stale words uint32, present bool per word)``, word p taken from the
    last earlier call on the same generation whose payload covered p."""
    last = {}     # generation -> the slot's words as last published
    written = {}  # generation -> which of those words any call has published
    out = []
    for i, (nbytes, v) in enumerate(schedule):
        g = i % GENERATIONS
        words = nbytes // 4
        want = expected[(nbytes, v)]
        slot = last.setdefault(g, np.zeros(0, np.uint32))
        seen = written.setdefault(g, np.zeros(0, bool))
        stale = np.zeros(words, np.uint32)
        present = np.zeros(words, bool)
        k = min(words, slot.size)
        stale[:k], present[:k] = slot[:k], seen[:k]
        out.append((stale, present))
        if slot.size < words:
            slot = np.concatenate([slot, np.zeros(words - slot.size, np.uint32)])
            seen = np.concatenate([seen, np.zeros(words - seen.size, bool)])
        slot[:words], seen[:words] = want, True
        last[g], written[g] = slot, seen
    return out


# ------------------------------------------------- device-side tolerance
# The BF16 tolerance of the parity tests (within 2 ULPs in the ordered
# encoding with +0 and -0 equal, or within 1e-3 absolute where the expected
# magnitude is below 2^-6; NaN never), written in torch so a stress test can
# count mismatches on the device after every replay without copying every
# output back.
ULP_TOL = 2
ABS_TOL = 1e-3
SMALL = 2.0 ** -6


def _ordered(b16: torch.Tensor) -> torch.Tensor:
    b = b16.to(torch.int32) & 0xFFFF
    return torch.where((b & 0x8000) != 0, -(b & 0x7FFF), b)


def _is_nan(b16: torch.Tensor) -> torch.Tensor:
    b = b16.to(torch.int32) & 0xFFFF
    return ((b & 0x7F80) == 0x7F80) & ((b & 0x007F) != 0)


def _value(b16: torch.Tensor) -> torch.Tensor:
    return ((b16.to(torch.int32) & 0xFFFF) << 16).view(torch.float32).to(torch.float64)


def bf16_mismatch_mask(got: torch.Tensor, want: torch.Tensor) -> torch.Tensor:
    """Positions of ``got`` outside the tolerance around ``want`` (both BF16
    bits in int16 / bfloat16 storage, same shape, any device)."""
    g = got.view(torch.int16) if got.dtype == torch.bfloat16 else got
    w = want.view(torch.int16) if want.dtype == torch.bfloat16 else want
    ulp = (_ordered(g) - _ordered(w)).abs()
    gv, wv = _value(g), _value(w)
    small_ok = (wv.abs() < SMALL) & ((gv - wv).abs() <= ABS_TOL)
    ok = (ulp <= ULP_TOL) | small_ok
    return ~ok | _is_nan(g) | _is_nan(w)


def bf16_mismatch_count(got: torch.Tensor, want: torch.Tensor) -> torch.Tensor:
    return bf16_mismatch_mask(got, want).sum()
