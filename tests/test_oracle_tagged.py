"""Pins of the oracle's tagged-pair mailbox (CPU only): the sync page's
Mailbox stores each 32-bit value beside the launch's tag, a consumer polls
until every tag matches, and nothing is reset.  Checked: the pair layout
(value word, tag) with column 2w in the low half, bits moved unchanged
(negative zero included), a stale tag detected, the armed state."""
import numpy as np

import oracle


def test_pair_layout_and_unchanged_bits():
    mb = oracle.TaggedMailbox(4, 16)
    assert (mb.pairs == 0).all()
    c = (np.arange(3 * 16, dtype=np.uint16).reshape(3, 16) * 1021 + 7).astype(np.uint16)
    c[0, 0] = 0x8000
    c[2, 15] = 0x8000
    assert mb.publish(c, 5) == oracle.OK
    for t in range(3):
        for w in range(8):
            assert mb.pairs[t, w, 0] == (int(c[t, 2 * w]) | (int(c[t, 2 * w + 1]) << 16))
            assert mb.pairs[t, w, 1] == 5
    assert (mb.pairs[3] == 0).all()  # rows >= m untouched
    st, out = mb.consume(3, 5)
    assert st == oracle.OK and (out == c).all()  # -0 arrives as -0


def test_stale_tag_and_no_reset():
    mb = oracle.TaggedMailbox(8, 128)
    rng = np.random.default_rng(1)
    c1 = rng.integers(0, 65536, size=(4, 128)).astype(np.uint16)
    c2 = rng.integers(0, 65536, size=(2, 128)).astype(np.uint16)
    mb.publish(c1, 1)
    assert mb.consume(4, 1)[0] == oracle.OK
    assert mb.consume(4, 1)[0] == oracle.OK  # nothing was reset: the same step reads again
    assert mb.consume(4, 2)[0] == oracle.ERR_SENTINEL  # next step before its publish: stale
    mb.publish(c2, 2)
    st, out = mb.consume(2, 2)
    assert st == oracle.OK and (out == c2).all()
    assert mb.consume(4, 2)[0] == oracle.ERR_SENTINEL  # rows 2..3 still carry tag 1


def test_tag_zero_and_bad_sizes_refused():
    mb = oracle.TaggedMailbox(2, 8)
    assert mb.publish(np.zeros((1, 8), np.uint16), 0) == oracle.ERR_ARGS
    assert mb.publish(np.zeros((3, 8), np.uint16), 1) == oracle.ERR_ARGS
    assert mb.consume(1, 0)[0] == oracle.ERR_ARGS
