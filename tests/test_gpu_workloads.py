"""The four named workloads of the decode projection, end to end on the GPU:

* N=256, K=256, m=1, S=1: one call then one consume, every value checked;
* N=4096, K=4096, m=4, S=1: 100 back-to-back calls cycling the generations;
* N=7168, K=8192, m=8, S=2: GEMM and consumer captured in one CUDA graph;
* N=7168, K=16384, m=8, S=4: 10,000 graph-replayed calls with m alternating
  1, 3, 8, in the launch configuration the benchmark times, with four inputs
  cycling beside the sizes so every use of a generation gets new bytes; every
  call checked against its own oracle answer; the mailbox must end with no
  stale or sentinel word left behind;
* the same stress on N=4096, K=4096 with sizes of period 4, so every
  generation sees every m.
"""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from mxfp8_gemm_mailbox_gb300 import OK, Mailbox, PublishGemm
from tests import stress_schedule as ss
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


def _stress(wl, sizes, variants, calls, graph_calls):
    """Replays ``calls`` chained calls (GEMM + consumer) from CUDA graphs of
    ``graph_calls`` calls, m cycling through ``sizes`` and the activations
    through ``variants`` seeded inputs, so that every use of a generation gets
    new bytes (a word left behind by an earlier call then differs from the
    expected one).  Every call has its own output buffer, poisoned with NaN
    before each replay; after each replay every call's output is checked on
    the device against its own oracle answer (the parity tolerance) and
    against the first replay's output for the same (m, input) (bit for bit),
    and the state words are recorded.  Returns the mailbox after the run."""
    w, ws = synthetic.make_weights(wl)
    acts = [synthetic.make_activations(wl, m=max(sizes), salt=v) for v in range(variants)]
    wants = [sanitized(oracle.gemm_bf16(w, ws, x, xs)) for x, xs in acts]  # [max m][N] each
    mb = Mailbox(wl.capacity, wl.n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=wl.split_k)  # the benchmark's tactic
    X = [(dev(x), dev(xs)) for x, xs in acts]
    schedule = ss.mailbox_schedule(graph_calls, sizes, variants)
    assert graph_calls % ss.period(len(sizes), variants, 3) == 0
    outs = torch.empty((graph_calls, 8, wl.n), dtype=torch.int16, device="cuda")
    want_dev = torch.zeros_like(outs)
    rows = torch.zeros((graph_calls, 8, 1), dtype=torch.bool, device="cuda")
    for j, (m, v) in enumerate(schedule):
        want_dev[j, :m] = torch.from_numpy(wants[v][:m].view(np.int16)).cuda()
        rows[j, :m] = True
    nan = torch.tensor(0x7FC1, dtype=torch.int16)  # never a result, never the sentinel half
    stream = torch.cuda.Stream()
    for m in sizes:
        g.precompile(m)

    def issue(js):
        for j in js:
            m, v = schedule[j]
            g.run(X[v][0][:m], X[v][1][:m])
            mb.consume(m, outs[j, :m].view(torch.bfloat16))

    # Eager warm-up calls (the handle's first run among them), then the
    # graphs: one of the whole period and, for the calls past its last whole
    # replay, one of the period's first `rest` calls.
    graph, tail = torch.cuda.CUDAGraph(), None
    with torch.cuda.stream(stream):
        issue(range(graph_calls))
        stream.synchronize()
        with torch.cuda.graph(graph, stream=stream):
            issue(range(graph_calls))
    eager = graph_calls
    replays, rest = divmod(calls, graph_calls)
    if rest:
        tail = torch.cuda.CUDAGraph()
        with torch.cuda.graph(tail, stream=stream):
            issue(range(rest))
    torch.cuda.synchronize()
    assert state_words(mb) == [eager % 3, (eager - 1) % 3, 0, 0]

    # First replay: every call against the full oracle on the host.
    outs.fill_(int(nan))
    with torch.cuda.stream(stream):
        graph.replay()
    torch.cuda.synchronize()
    first = outs.clone()
    host = outs.cpu().numpy().view(np.uint16)
    for j, (m, v) in enumerate(schedule):
        assert_bf16_close(host[j, :m], wants[v][:m], f"replayed call {j}: m={m}, input {v}")
        assert not (host[j, :m].view(np.uint32) == oracle.SENTINEL).any()
    done = graph_calls
    # The rest: counted on the device after every replay.
    bad_tol = torch.zeros((), dtype=torch.int64, device="cuda")
    bad_bits = torch.zeros((), dtype=torch.int64, device="cuda")
    history = torch.empty((replays - 1, 4), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(stream):
        for r in range(replays - 1):
            outs.fill_(int(nan))
            graph.replay()
            bad_tol += (ss.bf16_mismatch_mask(outs, want_dev) & rows).sum()
            bad_bits += ((outs != first) & rows).sum()
            history[r].copy_(mb.state)
        done += (replays - 1) * graph_calls
        if tail is not None:
            outs.fill_(int(nan))
            tail.replay()
            bad_tol += (ss.bf16_mismatch_mask(outs[:rest], want_dev[:rest]) & rows[:rest]).sum()
            bad_bits += ((outs[:rest] != first[:rest]) & rows[:rest]).sum()
            done += rest
    torch.cuda.synchronize()
    assert done == calls
    assert int(bad_tol) == 0, f"{int(bad_tol)} outputs outside the tolerance of their call"
    assert int(bad_bits) == 0, f"{int(bad_bits)} outputs differ from the same call's first run"
    h = history.cpu().numpy()
    assert (h == np.array([0, 2, 0, 0], np.int32)).all()  # graph_calls is a multiple of 3
    total = eager + calls
    assert state_words(mb) == [total % 3, (total - 1) % 3, 0, 0]
    assert (mailbox_words(mb) == oracle.SENTINEL).all()  # no stale word anywhere
    assert mb.status()[0] == OK
    g.close()
    return mb


def test_headline_graph_stress_ten_thousand_calls(cuda):
    # The spec stress: N=7168, K=16384, m=8, S=4 in the benchmark's
    # launch configuration, m alternating 1, 3, 8 each call, 10,000 calls
    # replayed from CUDA graphs.  Four activation inputs cycle beside the
    # three sizes, so generation g sees input (g + 3u) mod 4 on its u-th use:
    # new bytes every time.
    _stress(synthetic.HEADLINE, (1, 3, 8), 4, 10_000, 12)


def test_generation_shifting_stress(cuda):
    # Sizes cycling with a period of 4 over the 3 generations, so every
    # generation sees every m (a row that one use leaves unread is read by a
    # later one) and 5 inputs: 10,000 calls of the chain workload's shape.
    _stress(synthetic.CHAIN_4096, (1, 3, 8, 5), 5, 10_000, 60)
