"""The four named workloads of the decode projection, end to end on the GPU:

* N=256, K=256, m=1, S=1: one call then one consume, every value checked;
* N=4096, K=4096, m=4, S=1: 100 back-to-back calls cycling the generations;
* N=7168, K=8192, m=8, S=2: GEMM and consumer captured in one CUDA graph;
* N=7168, K=16384, m=8, S=4: 10,000 graph replays with m alternating 1, 3, 8,
  in the launch configuration the benchmark times, checked against the full
  oracle; the mailbox must end with no stale or sentinel word left behind.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from mxfp8_gemm_mailbox_gb300 import OK, Mailbox, PublishGemm
from tests.gpu_util import (assert_bf16_close, bits, dev, mailbox_words, pack_words, sanitized,
                            state_words)

pytestmark = pytest.mark.gpu


def test_tiny_workload(cuda):
    wl = synthetic.TINY
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    ref = oracle.Mailbox(wl.capacity, wl.n)
    st, want_c, want_out = ref.chain(w, ws, x, xs)
    assert st == oracle.OK
    mb = Mailbox(wl.capacity, wl.n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=wl.split_k)
    c = torch.empty((wl.m, wl.n), dtype=torch.bfloat16, device="cuda")
    g.run(dev(x), dev(xs), c)
    torch.cuda.synchronize()
    between = mailbox_words(mb)
    expect = np.full_like(between, oracle.SENTINEL)
    expect[0, :wl.m] = pack_words(sanitized(bits(c)))
    assert (between == expect).all()
    out = mb.consume(wl.m)
    torch.cuda.synchronize()
    assert_bf16_close(bits(c), want_c, "C")
    assert_bf16_close(bits(out), want_out, "consumer output")
    assert (bits(out) == sanitized(bits(c))).all()
    assert (mailbox_words(mb) == ref.words).all()      # all sentinel again
    assert state_words(mb) == list(ref.state) == [1, 0, 0, 0]


def test_chain_4096_hundred_calls(cuda):
    wl = synthetic.CHAIN_4096
    w, ws = synthetic.make_weights(wl)
    xs_list = [synthetic.make_activations(wl, salt=s) for s in range(4)]
    wants = [oracle.gemm_bf16(w, ws, x, xs) for x, xs in xs_list]
    mb = Mailbox(wl.capacity, wl.n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=wl.split_k)
    dx = [(dev(x), dev(xs)) for x, xs in xs_list]
    outs = torch.empty((100, wl.m, wl.n), dtype=torch.bfloat16, device="cuda")
    cs = torch.empty((100, wl.m, wl.n), dtype=torch.bfloat16, device="cuda")
    states = torch.empty((100, 4), dtype=torch.int32, device="cuda")
    for i in range(100):
        X, XS = dx[i % 4]
        g.run(X, XS, cs[i])
        mb.consume(wl.m, outs[i])
        states[i].copy_(mb.state)
    torch.cuda.synchronize()
    st = states.cpu().numpy()
    for i in range(100):
        assert list(st[i]) == [(i + 1) % 3, i % 3, 0, 0], i
        assert_bf16_close(bits(cs[i]), wants[i % 4], f"call {i}")
        assert (bits(outs[i]) == sanitized(bits(cs[i]))).all(), i
    assert (mailbox_words(mb) == oracle.SENTINEL).all()
    assert mb.status()[0] == OK


def test_graph_8192_split2(cuda):
    wl = synthetic.GRAPH_8192
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    want = oracle.gemm_bf16(w, ws, x, xs)
    mb = Mailbox(wl.capacity, wl.n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=wl.split_k)
    X, XS = dev(x), dev(xs)
    c = torch.empty((wl.m, wl.n), dtype=torch.bfloat16, device="cuda")
    out = torch.empty((wl.m, wl.n), dtype=torch.bfloat16, device="cuda")
    g.precompile(wl.m)
    stream = torch.cuda.Stream()
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph, stream=stream):
        g.run(X, XS, c)
        mb.consume(wl.m, out)
    torch.cuda.synchronize()
    for replay in range(7):
        graph.replay()
        torch.cuda.synchronize()
        assert state_words(mb) == [(replay + 1) % 3, replay % 3, 0, 0]
        assert_bf16_close(bits(c), want, f"replay {replay}")
        assert (bits(out) == sanitized(bits(c))).all()
        assert (mailbox_words(mb) == oracle.SENTINEL).all()


def test_headline_graph_stress_ten_thousand_calls(cuda):
    wl = synthetic.HEADLINE
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    want = oracle.gemm_bf16(w, ws, x, xs)  # [8][7168]; m rows are its first m rows
    mb = Mailbox(wl.capacity, wl.n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=wl.split_k)  # the benchmark's tactic
    X, XS = dev(x), dev(xs)
    sizes = (1, 3, 8)
    outs = {m: torch.empty((m, wl.n), dtype=torch.bfloat16, device="cuda") for m in sizes}
    graphs = {}
    stream = torch.cuda.Stream()
    for m in sizes:
        g.precompile(m)
        graphs[m] = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graphs[m], stream=stream):
            g.run(X[:m], XS[:m])
            mb.consume(m, outs[m])
    torch.cuda.synchronize()
    # First cycle: every output against the full oracle.
    for m in sizes:
        graphs[m].replay()
    torch.cuda.synchronize()
    refs = {}
    for m in sizes:
        got = bits(outs[m])
        assert_bf16_close(got, sanitized(want[:m]), f"m={m}")
        assert not (got.view(np.uint32) == oracle.SENTINEL).any()
        refs[m] = outs[m].clone()
    assert state_words(mb) == [0, 2, 0, 0]
    # The rest: 9,999 more calls; every output compared on the device with the
    # first cycle's (the kernels are deterministic) and the state recorded
    # after every 3-call cycle.
    cycles = (10_000 - 3) // 3
    mismatches = torch.zeros((), dtype=torch.int64, device="cuda")
    history = torch.empty((cycles, 4), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for i in range(cycles):
            for m in sizes:
                graphs[m].replay()
                mismatches += (outs[m].view(torch.int16) != refs[m].view(torch.int16)).sum()
            history[i].copy_(mb.state)
        graphs[1].replay()  # the 10,000th call
        mismatches += (outs[1].view(torch.int16) != refs[1].view(torch.int16)).sum()
    torch.cuda.synchronize()
    assert int(mismatches) == 0
    h = history.cpu().numpy()
    assert (h == np.array([0, 2, 0, 0], np.int32)).all()
    total_calls = 3 + 3 * cycles + 1
    assert total_calls == 10_000
    assert state_words(mb) == [total_calls % 3, (total_calls - 1) % 3, 0, 0]
    assert (mailbox_words(mb) == oracle.SENTINEL).all()  # no stale word anywhere
    assert mb.status()[0] == OK
