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
from tests.gpu_util import dev

pytestmark = pytest.mark.gpu

CAP = 256 * 1024  # "a few hundred kilobytes at most"


def _words(n, seed, sentinel_share=0.05):
    rng = np.random.default_rng(seed)
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
    # Back-to-back gathers of alternating sizes replayed from CUDA graphs: a
    # word left behind by one call would show up in a later call of another
    # size.  Every output is compared on the device with its expected value.
    g = LamportGather(CAP)
    sizes = (16, 4112, CAP)
    inputs = {s: dev(_words(s // 4, seed=s).view(np.int32)) for s in sizes}
    expect = {s: torch.where(inputs[s] == -(2**31), torch.zeros_like(inputs[s]), inputs[s])
              for s in sizes}
    outs = {s: torch.empty_like(inputs[s]) for s in sizes}
    stream = torch.cuda.Stream()
    graphs = {}
    for s in sizes:
        graphs[s] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[s], stream=stream):
            g(inputs[s], outs[s])
    torch.cuda.synchronize()
    calls = 0
    mismatches = torch.zeros((), dtype=torch.int64, device="cuda")
    with torch.cuda.stream(stream):
        for _ in range(3000):
            for s in sizes:
                graphs[s].replay()
                calls += 1
                mismatches += (outs[s] != expect[s]).sum()
    torch.cuda.synchronize()
    assert int(mismatches) == 0
    assert (_mailbox(g) == oracle.SENTINEL).all()
    assert [int(v) for v in g.state.cpu()] == [calls % 3, 0, 0, 0]
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
