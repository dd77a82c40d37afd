"""GPU parity of the tagged-pair mailbox against the oracle: the pairs in
memory, the consumer output (bits unchanged, negative zero kept), a stale
tag running into the bounded poll, and the protocol fed by the GEMM."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from mxfp8_gemm_mailbox_gb300 import PublishGemm, TaggedMailbox
from tests.gpu_util import bits, dev

pytestmark = pytest.mark.gpu


def _c(m, n, seed):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 65536, size=(m, n)).astype(np.uint16)
    c[rng.random((m, n)) < 0.05] = 0x8000
    return c


def _pairs(mb):
    return mb.pairs.cpu().numpy().view(np.uint32).reshape(mb.capacity, mb.n // 2, 2)


@pytest.mark.parametrize("capacity,n,ms", [(8, 256, [3, 8, 1, 5]), (8, 7168, [8, 1, 3]),
                                           (2, 8, [1, 2])])
def test_tagged_matches_oracle(cuda, capacity, n, ms):
    mb = TaggedMailbox(capacity, n)
    ref = oracle.TaggedMailbox(capacity, n)
    assert (_pairs(mb) == 0).all()
    for i, m in enumerate(ms):
        tag = 1000 + i
        c = _c(m, n, seed=i)
        mb.publish(dev(c.view(np.int16)), tag)
        assert ref.publish(c, tag) == oracle.OK
        torch.cuda.synchronize()
        assert (_pairs(mb) == ref.pairs).all()
        out = mb.consume(m, tag)
        st, want = ref.consume(m, tag)
        torch.cuda.synchronize()
        assert st == oracle.OK and (bits(out) == want).all() and (want == c).all()
    assert int(mb.flags.cpu()[0]) == 0


def test_stale_tag_runs_into_the_bounded_poll(cuda):
    mb = TaggedMailbox(4, 512)
    c1, c2 = _c(4, 512, 1), _c(4, 512, 2)
    mb.publish(dev(c1.view(np.int16)), 1)
    out = mb.consume(4, 2, timeout_ns=1_000_000)  # step 2 before its publish
    torch.cuda.synchronize()
    assert int(mb.flags.cpu()[0]) & 0x1
    assert (bits(out) == c1).all()  # what was there
    mb.flags.zero_()
    mb.publish(dev(c2.view(np.int16)), 2)
    out = mb.consume(4, 2)
    torch.cuda.synchronize()
    assert (bits(out) == c2).all() and int(mb.flags.cpu()[0]) == 0


def test_tagged_protocol_behind_the_gemm(cuda):
    wl = synthetic.Workload("tagged", 1024, 2048, 8, 2, exp_lo=-6, exp_hi=3, signed_pairs=True,
                            seed=77)
    w, ws = synthetic.make_weights(wl)
    g = PublishGemm(dev(w), dev(ws), __import__("mxfp8_gemm_mailbox_gb300").Mailbox(8, 1024),
                    split_k=2)
    mb = TaggedMailbox(8, 1024)
    for call in range(3):
        x, xs = synthetic.make_activations(wl, salt=call)
        c = torch.empty((8, 1024), dtype=torch.bfloat16, device="cuda")
        g.run_unfused(dev(x), dev(xs), c)
        mb.publish(c, call + 1)
        out = mb.consume(8, call + 1)
        torch.cuda.synchronize()
        assert (bits(out) == bits(c)).all()  # unchanged, -0 included
    assert int(mb.flags.cpu()[0]) == 0
