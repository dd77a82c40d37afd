"""Seeded random combinations of shape and tactic -- N, ragged K, m, split-K
S, ring depth, pipes, accumulation granularity, weight layout, TMEM read-out,
L2 prefetch (both groups of CTAs), fold, K per pipeline stage (cta_k),
mailbox capacity -- each run through GEMM and consumer on integer-valued
inputs and checked bit-exactly against the oracle: C, the published mailbox
words between the two kernels, the consumer's output, the state words and
the reset mailbox.  Combinations the library refuses (a ring
that does not fit, pipes that do not divide it, a fold with S = 8, one slot
per MMA or the 16x256b read-out, fold 8 with S > 1 or 4 pipes, cta_k 256
with fold 8, S = 8, one slot per MMA, the 16x256b read-out or an
accumulator ring that is not a multiple of 2 x pipes) must be refused on
the host with MXFP8_ERR_UNSUPPORTED."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from mxfp8_gemm_mailbox_gb300 import OK, Mailbox, Mxfp8Error, PublishGemm
from tests.gpu_util import bits, dev, mailbox_words, pack_words, sanitized, state_words

pytestmark = pytest.mark.gpu


def draw(rng):
    n = int(rng.choice([128, 256, 384, 640, 1024]))
    k = int(32 * rng.integers(1, 257))  # 32 .. 8192, ragged K tiles included
    m = int(rng.integers(1, 9))
    return dict(
        n=n, k=k, m=m,
        split_k=int(rng.choice([1, 2, 4, 8])),
        stages=int(rng.choice([0, 0, 2, 3, 4, 5, 6, 8, 12])),
        pipes=int(rng.choice([0, 0, 1, 2, 4])),
        acc_blocks=int(rng.choice([0, 1, 4])),
        w_layout=int(rng.choice([0, 1, 2])),
        tmem_load=int(rng.choice([0, 1, 2])),
        l2_prefetch=int(rng.choice([-1, 0, 3])),
        capacity=int(rng.integers(m, 9)),
        fold=int(rng.choice([0, 0, 1, 2, 4, 8])),
        l2_prefetch_early=int(rng.choice([-1, 0, 0, 2, 12])),
        cta_k=int(rng.choice([0, 0, 128, 256])),
    )


def test_random_shapes_and_tactics(cuda):
    rng = np.random.default_rng(20261202)
    ran = refused = 0
    for case in range(80):
        p = draw(rng)
        n, k, m, cap = p["n"], p["k"], p["m"], p["capacity"]
        w, ws, x, xs = synthetic.integer_operands(n, k, m, seed=case)
        mb = Mailbox(cap, n)
        try:
            g = PublishGemm(dev(w), dev(ws), mb, split_k=p["split_k"], stages=p["stages"],
                            acc_blocks=p["acc_blocks"], w_layout=p["w_layout"],
                            l2_prefetch=p["l2_prefetch"], pipes=p["pipes"],
                            tmem_load=p["tmem_load"], fold=p["fold"],
                            l2_prefetch_early=p["l2_prefetch_early"], cta_k=p["cta_k"])
        except Mxfp8Error as e:
            assert "ERR_UNSUPPORTED" in str(e), (p, str(e))
            refused += 1
            continue
        cfg = g.config()
        assert cfg["stages"] % cfg["pipes"] == 0, (p, cfg)
        want = oracle.gemm_bf16(w, ws, x, xs)
        c = torch.full((m, n), 0x7FFF, dtype=torch.int16, device="cuda")
        for call in range(2):
            g.run(dev(x), dev(xs), c)
            torch.cuda.synchronize()
            between = mailbox_words(mb).copy()
            out = mb.consume(m)
            torch.cuda.synchronize()
            assert (bits(c) == want).all(), (p, cfg, call)
            assert (bits(out) == sanitized(want)).all(), (p, cfg, call)
            expect = np.full((3, cap, n // 2), oracle.SENTINEL, np.uint32)
            expect[call % 3, :m] = pack_words(sanitized(want))
            assert (between == expect).all(), (p, cfg, call)
            assert state_words(mb) == [(call + 1) % 3, call % 3, 0, 0], (p, cfg, call)
            assert (mailbox_words(mb) == oracle.SENTINEL).all(), (p, cfg, call)
        assert mb.status()[0] == OK
        g.close()
        ran += 1
    assert ran >= 30 and ran + refused == 80, (ran, refused)
