"""GPU parity of the one-rank Lamport all-gather against the oracle: every
word bit-exact over alternating sizes, the generation sequence, the arrival
count and the reset of every slot; the stale-word stress of the all-gather
page (back-to-back gathers of alternating sizes replayed from CUDA graphs);
a corrupted generation flagged without any out-of-range access."""
import numpy as np
import pytest
import torch

import oracle
from mxfp8_gemm_mailbox_gb300 import ERR_STATE, OK, LamportGather
from tests import stress_schedule as ss
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

CAP = 256 * 1024  # "a few hundred kilobytes at most"


def _words(n, seed, sentinel_share=0.05):
    rng = np.random.default_rng(list(seed) if isinstance(seed, tuple) else seed)
    w = rng.integers(0, 2**32, size=n, dtype=np.uint64).astype(np.uint32)
    w[rng.random(n) < sentinel_share] = oracle.SENTINEL
    return w


def _mailbox(g):
    return g.words.cpu().numpy().view(np.uint32).reshape(3, -1)


def test_gather_matches_oracle_over_alternating_sizes(cuda):
    g = LamportGather(CAP)
    ref = oracle.Gather(CAP)
    sizes = [16, CAP, 48, 4112, 16, CAP - 16, 65536, 272]
    for i, nbytes in enumerate(sizes * 2):
        inp = _words(nbytes // 4, seed=i)
        out = g(dev(inp.view(np.int32)))
        st, want = ref(inp)
        assert st == oracle.OK
        torch.cuda.synchronize()
        got = out.cpu().numpy().view(np.uint32)
        assert (got == want).all(), f"call {i}, {nbytes} bytes"
        assert (_mailbox(g) == oracle.SENTINEL).all()
        assert [int(v) for v in g.state.cpu()] == [(i + 1) % 3, 0, 0, 0] == list(ref.state) + [0, 0]
    assert g.status()[0] == OK


def test_gather_stale_word_stress_in_graphs(cuda):
    # Back-to-back gathers of alternating sizes replayed from CUDA graphs (the
    # all-gather page's stress).  The sizes cycle with a period of 4 over the
    # 3 generations and each size has 5 inputs, so every use of a generation
    # gets another size and other bytes: a word that one call left in a slot
    # differs from what a later call reading it should return.  Every call
    # writes its own output, poisoned before each replay, and is compared on
    # the device with the oracle's answer for its input: 10,000 calls.
    g = LamportGather(CAP)
    ref = oracle.Gather(CAP)
    sizes, variants = (16, 4112, CAP, 48), 5
    per_graph = ss.period(len(sizes), variants, 3)  # 60 calls
    schedule = ss.gather_schedule(per_graph, sizes, variants)
    inputs, expect = {}, {}
    for nbytes in sizes:
        for v in range(variants):
            words = _words(nbytes // 4, seed=(nbytes, v))
            st, want = ref(words)
            assert st == oracle.OK
            inputs[(nbytes, v)] = dev(words.view(np.int32))
            expect[(nbytes, v)] = dev(want.view(np.int32))
    outs = [torch.empty(nbytes // 4, dtype=torch.int32, device="cuda") for nbytes, _ in schedule]
    stream = torch.cuda.Stream()
    with torch.cuda.stream(stream):
        for j, key in enumerate(schedule):  # eager warm-up
            g(inputs[key], outs[j])
        stream.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=stream):
            for j, key in enumerate(schedule):
                g(inputs[key], outs[j])
    torch.cuda.synchronize()
    calls = 10_020  # 167 replays of 60 calls
    mismatches = torch.zeros((), dtype=torch.int64, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(calls // per_graph):
            for o in outs:
                o.fill_(-(2**31))  # the sentinel word: never an output word
            graph.replay()
            for j, key in enumerate(schedule):
                mismatches += (outs[j] != expect[key]).sum()
    torch.cuda.synchronize()
    assert int(mismatches) == 0
    assert (_mailbox(g) == oracle.SENTINEL).all()
    total = per_graph + calls
    assert [int(v) for v in g.state.cpu()] == [total % 3, 0, 0, 0]
    assert g.status()[0] == OK


def test_gather_corrupted_generation_is_flagged(cuda):
    g = LamportGather(4096)
    before = _mailbox(g).copy()
    g.state[0] = 9
    out = torch.full((256,), 7, dtype=torch.int32, device="cuda")
    g(dev(_words(256, seed=1).view(np.int32)), out)
    torch.cuda.synchronize()
    assert g.status()[0] == ERR_STATE
    assert (_mailbox(g) == before).all()
    assert (out.cpu() == 7).all()
