"""Pins of the oracle's one-rank Lamport all-gather (CPU only): worked
examples from the all-gather page's sanitisation rule, the closed form
(output = input with the sentinel word cleared), the generation sequence,
the arrival count and the reset of every slot, over alternating sizes."""
from pathlib import Path

import numpy as np
import pytest

import oracle

GOLDEN = Path(__file__).resolve().parent / "golden"


def _pairs():
    lines = [l.split() for l in (GOLDEN / "all_gather_worked.txt").read_text().splitlines()
             if l.strip() and not l.startswith("#")]
    for a, b in zip(lines[0::2], lines[1::2]):
        assert a[0] == "in" and b[0] == "out"
        yield (np.array([int(w, 16) for w in a[1:]], np.uint32),
               np.array([int(w, 16) for w in b[1:]], np.uint32))


def test_gather_worked_examples_golden():
    for inp, want in _pairs():
        g = oracle.Gather(64)
        st, out = g(inp)
        assert st == oracle.OK and (out == want).all()


def test_gather_sequence_of_alternating_sizes():
    rng = np.random.default_rng(3)
    cap = 4096
    g = oracle.Gather(cap)
    sizes = [16, cap, 48, 1024, 16, cap - 16, 272]
    for i, nbytes in enumerate(sizes * 3):
        inp = rng.integers(0, 2**32, size=nbytes // 4, dtype=np.uint64).astype(np.uint32)
        inp[rng.random(inp.size) < 0.1] = oracle.SENTINEL
        st, out = g(inp)
        assert st == oracle.OK
        assert (out == np.where(inp == oracle.SENTINEL, 0, inp)).all()
        assert list(g.state) == [(i + 1) % 3, 0]
        assert (g.words == oracle.SENTINEL).all()
        assert not (out == oracle.SENTINEL).any()


@pytest.mark.parametrize("nbytes,cap", [(0, 64), (20, 64), (80, 64)])
def test_gather_rejects_bad_sizes(nbytes, cap):
    g = oracle.Gather(cap)
    st, _ = g(np.zeros(max(nbytes // 4, 0), np.uint32)) if nbytes else (
        oracle._load().oracle_all_gather(None, None, cap // 4, None, 0, None), None)
    assert st == oracle.ERR_ARGS


def test_gather_bad_generation():
    g = oracle.Gather(64)
    g.state[0] = 3
    st, _ = g(np.zeros(4, np.uint32))
    assert st == oracle.ERR_STATE
    with pytest.raises(ValueError):
        oracle.Gather(20)
