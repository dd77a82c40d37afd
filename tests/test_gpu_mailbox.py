"""GPU parity of the mailbox kernels against the oracle: init, the standalone
publish, the consumer (poll, copy, reset, advance), its bounded poll and its
handling of a corrupted state word."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_gemm_mailbox_gb300 import ERR_STATE, ERR_TIMEOUT, OK, Mailbox, Mxfp8Error
from tests.gpu_util import bits, dev, mailbox_words, state_words

pytestmark = pytest.mark.gpu


def _random_c(m, n, seed):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 65536, size=(m, n)).astype(np.uint16)
    c[rng.random((m, n)) < 0.05] = 0x8000  # negative zeros to clear
    c[rng.random((m, n)) < 0.05] = 0x0000
    return c


@pytest.mark.parametrize("capacity,n", [(8, 256), (1, 8), (3, 7168), (8, 4096)])
def test_init_arms_every_slot(cuda, capacity, n):
    mb = Mailbox(capacity, n)
    mb.words.fill_(123)
    mb.state.fill_(9)
    mb.init()
    torch.cuda.synchronize()
    ref = oracle.Mailbox(capacity, n)
    assert (mailbox_words(mb) == ref.words).all()
    assert state_words(mb) == list(ref.state)


@pytest.mark.parametrize("capacity,n,ms", [(8, 256, [3, 1, 8, 2, 5]), (4, 1024, [4, 4, 1]),
                                           (8, 7168, [8, 3, 1, 8])])
def test_publish_and_consume_match_oracle(cuda, capacity, n, ms):
    mb = Mailbox(capacity, n)
    ref = oracle.Mailbox(capacity, n)
    for i, m in enumerate(ms):
        c = _random_c(m, n, seed=100 + i)
        mb.publish(dev(c.view(np.int16)))
        assert ref.publish(c) == oracle.OK
        torch.cuda.synchronize()
        # the mailbox between publish and consume: bit-exact
        assert (mailbox_words(mb) == ref.words).all()
        assert state_words(mb) == list(ref.state)
        out = mb.consume(m)
        st, want = ref.consume(m)
        assert st == oracle.OK
        torch.cuda.synchronize()
        assert (bits(out) == want).all()
        assert (mailbox_words(mb) == oracle.SENTINEL).all()
        assert state_words(mb) == list(ref.state) == [(i + 1) % 3, i % 3, 0, 0]
    assert mb.status()[0] == OK


def test_consume_of_an_oracle_made_mailbox(cuda):
    # The consumer alone, on a mailbox the oracle wrote (generation 2).
    capacity, n, m = 8, 512, 6
    ref = oracle.Mailbox(capacity, n)
    for _ in range(2):
        ref.state[0] = (ref.state[0] + 1) % 3
    c = _random_c(m, n, seed=7)
    ref.publish(c)
    mb = Mailbox(capacity, n)
    mb.words.copy_(torch.from_numpy(ref.words.reshape(-1).view(np.int32)))
    mb.state.copy_(torch.from_numpy(ref.state.copy()))
    out = mb.consume(m)
    st, want = ref.consume(m)
    torch.cuda.synchronize()
    assert (bits(out) == want).all()
    assert (mailbox_words(mb) == ref.words).all()
    assert state_words(mb) == list(ref.state) == [0, 2, 0, 0]


def test_consume_without_publish_times_out_and_drains(cuda):
    # Nothing published: every poll must give up after its limit (1 ms here),
    # flag the timeout, reset the slot, and the generation must still advance.
    mb = Mailbox(8, 1024)
    out = mb.consume(4, timeout_ns=1_000_000)
    torch.cuda.synchronize()
    status, words = mb.status()
    assert status == ERR_TIMEOUT
    assert words[:3] == [1, 0, 0] and words[3] & 0x1
    assert (mailbox_words(mb) == oracle.SENTINEL).all()
    assert (bits(out).view(np.uint32) == oracle.SENTINEL).all()  # copied what was there
    # the context stays usable: a normal publish + consume afterwards
    mb.init()
    c = _random_c(2, 1024, seed=3)
    mb.publish(dev(c.view(np.int16)))
    out = mb.consume(2)
    torch.cuda.synchronize()
    assert (bits(out) == np.where(c == 0x8000, 0, c)).all()
    assert mb.status()[0] == OK


def test_corrupted_generation_is_flagged_not_followed(cuda):
    mb = Mailbox(8, 256)
    before = mailbox_words(mb).copy()
    mb.state[1] = 7  # an active generation outside 0..2
    mb.consume(2)
    torch.cuda.synchronize()
    status, words = mb.status()
    assert status == ERR_STATE and words[3] & 0x4
    assert (mailbox_words(mb) == before).all()  # nothing addressed
    mb.init()
    mb.state[0] = 5
    mb.publish(dev(np.zeros((1, 256), np.int16)))
    torch.cuda.synchronize()
    assert mb.status()[0] == ERR_STATE
    assert (mailbox_words(mb) == before).all()


def test_host_side_errors_raise(cuda):
    mb = Mailbox(4, 256)
    with pytest.raises(Mxfp8Error, match="ERR_UNSUPPORTED"):
        mb.consume(5)
    with pytest.raises(ValueError):
        Mailbox(9, 256)
