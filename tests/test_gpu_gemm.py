"""GPU parity of the publishing GEMM against the oracle, element by element,
at sizes the oracle finishes in seconds: several tiles, ragged K, every m,
every split-K cluster size, integer-valued inputs (bit-exact), N(0, 1)
inputs (within 2 BF16 ULPs), the mailbox between GEMM and consume, the
negative-zero clearing, and the fused vs unfused equivalence."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from mxfp8_gemm_mailbox_gb300 import ERR_STATE, OK, Mailbox, Mxfp8Error, PublishGemm
from mxfp8_gemm_mailbox_gb300._lib import (TMEM_LOAD_16X256B, TMEM_LOAD_32X32B, W_IN_PLACE,
                                            W_TILED)
from tests.gpu_util import (assert_bf16_close, bits, dev, mailbox_words, pack_words, sanitized,
                            state_words)

pytestmark = pytest.mark.gpu


def run_chain(w, ws, x, xs, split_k, capacity=8, stages=0, mailbox=None, acc_blocks=0,
              w_layout=0, fold=0, **tactic):
    """GEMM (C requested) -> snapshot of mailbox + state -> consume.  Returns
    (C bits, mailbox words between the two kernels, state then, out bits,
    mailbox words after, state after, handle config)."""
    n = w.shape[0]
    m = x.shape[0]
    mb = mailbox or Mailbox(capacity, n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=split_k, stages=stages, acc_blocks=acc_blocks,
                    w_layout=w_layout, fold=fold, **tactic)
    c = torch.full((m, n), 0x7FFF, dtype=torch.int16, device="cuda")
    g.run(dev(x), dev(xs), c)
    torch.cuda.synchronize()
    between = mailbox_words(mb).copy()
    state_between = state_words(mb)
    out = mb.consume(m)
    torch.cuda.synchronize()
    cfg = g.config()
    g.close()
    return (bits(c), between, state_between, bits(out), mailbox_words(mb).copy(),
            state_words(mb), cfg)


def check_published(between, state_between, c_bits, capacity, n, generation=0):
    m = c_bits.shape[0]
    assert state_between[1] == generation
    expect = np.full((3, capacity, n // 2), oracle.SENTINEL, np.uint32)
    expect[generation, :m] = pack_words(sanitized(c_bits))
    assert (between == expect).all(), "mailbox between GEMM and consume"
    lo, hi = between & 0xFFFF, between >> 16
    pub = between[generation, :m]
    assert not (pub == oracle.SENTINEL).any()
    assert not ((pub & 0xFFFF) == 0x8000).any() and not ((pub >> 16) == 0x8000).any()
    del lo, hi


@pytest.mark.parametrize("fold", [1, 2, 4])
@pytest.mark.parametrize("w_layout", [W_IN_PLACE, W_TILED])
@pytest.mark.parametrize("split_k", [1, 2, 4])
@pytest.mark.parametrize("n,k,m", [(128, 128, 1), (384, 1024, 8), (256, 2048, 5), (512, 4096, 3),
                                   (128, 96, 2), (256, 160, 7), (128, 32, 8), (256, 1152, 4)])
def test_integer_inputs_bit_exact(cuda, n, k, m, split_k, w_layout, fold):
    """Every shape, split and W layout unfolded and folded (a CTA holding
    128/fold columns in fold K pieces; K padded to whole pieces, splits with
    no K tile contributing zeros)."""
    w, ws, x, xs = synthetic.integer_operands(n, k, m, seed=n + k + m)
    want = oracle.gemm_bf16(w, ws, x, xs)
    c, between, sb, out, after, state, cfg = run_chain(w, ws, x, xs, split_k, w_layout=w_layout,
                                                      fold=fold)
    assert cfg["split_k"] == split_k and cfg["fold"] == fold
    assert cfg["grid_ctas"] == n // (128 // fold) * split_k
    assert cfg["w_layout"] == {W_IN_PLACE: "in_place", W_TILED: "tiled"}[w_layout]
    assert (c == want).all(), f"{int((c != want).sum())} of {c.size} differ"
    check_published(between, sb, c, 8, n)
    assert (out == sanitized(c)).all()
    assert (after == oracle.SENTINEL).all()
    assert state == [1, 0, 0, 0]


@pytest.mark.parametrize("fold", [1, 2, 4])
@pytest.mark.parametrize("w_layout", [W_IN_PLACE, W_TILED])
@pytest.mark.parametrize("split_k", [1, 2, 4])
@pytest.mark.parametrize("n,k,m,lo,hi", [(256, 256, 1, -3, 3), (1024, 4096, 8, -4, 2),
                                         (640, 2048, 6, -6, 3), (384, 8192, 4, -4, 2),
                                         (256, 1056, 3, -4, 2)])
def test_normal_inputs_within_two_ulps(cuda, n, k, m, lo, hi, split_k, w_layout, fold):
    wl = synthetic.Workload("p", n, k, m, split_k, exp_lo=lo, exp_hi=hi, x_zero_fraction=0.01,
                            seed=7 * n + k + m)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    want = oracle.gemm_bf16(w, ws, x, xs)
    c, between, sb, out, after, state, cfg = run_chain(w, ws, x, xs, split_k, w_layout=w_layout,
                                                      fold=fold)
    assert cfg["fold"] == fold
    assert_bf16_close(c, want, f"N={n} K={k} m={m} S={split_k} fold={fold}")
    check_published(between, sb, c, 8, n)
    assert (out == sanitized(c)).all()
    assert (after == oracle.SENTINEL).all()


@pytest.mark.parametrize("w_layout", [W_IN_PLACE, W_TILED])
@pytest.mark.parametrize("pipes", [1, 2])
@pytest.mark.parametrize("n,k,m", [(128, 1024, 8), (256, 4096, 5), (512, 8192, 3), (128, 96, 2),
                                   (256, 1152, 4), (384, 2048, 1), (2048, 16384, 8)])
def test_fold_eight(cuda, n, k, m, pipes, w_layout):
    """Fold 8 (16-row tiles, 8 K pieces per stage, N = 64 MMAs, x-scale rows
    holding two columns, a 2-slot accumulator ring): bit-exact on integer
    inputs, within 2 ULP on N(0, 1) inputs, with the mailbox and consumer."""
    w, ws, x, xs = synthetic.integer_operands(n, k, m, seed=800 + n + k + m)
    want = oracle.gemm_bf16(w, ws, x, xs)
    mb = Mailbox(8, n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=1, fold=8, pipes=pipes, w_layout=w_layout)
    cfg = g.config()
    assert (cfg["fold"], cfg["pipes"], cfg["grid_ctas"]) == (8, pipes, n // 16), cfg
    c = torch.full((m, n), 0x7FFF, dtype=torch.int16, device="cuda")
    for call in range(2):
        g.run(dev(x), dev(xs), c)
        out = mb.consume(m)
        torch.cuda.synchronize()
        assert (bits(c) == want).all(), f"C, call {call}"
        assert (bits(out) == sanitized(want)).all(), f"consumer output, call {call}"
    assert mb.status()[0] == OK and (mailbox_words(mb) == oracle.SENTINEL).all()
    g.close()
    wl = synthetic.Workload("f8", n, k, m, 1, exp_lo=-4, exp_hi=2, x_zero_fraction=0.01,
                            seed=900 + n + k + m)
    wn, wsn = synthetic.make_weights(wl)
    xn, xsn = synthetic.make_activations(wl)
    c2, between, sb, out2, after, state, cfg2 = run_chain(wn, wsn, xn, xsn, 1, fold=8,
                                                          w_layout=w_layout)
    assert cfg2["fold"] == 8
    assert_bf16_close(c2, oracle.gemm_bf16(wn, wsn, xn, xsn), f"N={n} K={k} m={m} fold 8")
    check_published(between, sb, c2, 8, n)
    assert (out2 == sanitized(c2)).all()


def test_split_k_results_agree(cuda):
    """Every split and fold: within tolerance of the oracle on N(0, 1)
    inputs, identical bits on integer inputs."""
    wl = synthetic.Workload("s", 512, 4096, 8, exp_lo=-4, exp_hi=2, seed=3)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    want = oracle.gemm_bf16(w, ws, x, xs)
    tactics = [(s, f) for s in (1, 2, 4) for f in (1, 2, 4)]
    results = [run_chain(w, ws, x, xs, s, fold=f)[0] for s, f in tactics]
    for r in results:
        assert_bf16_close(r, want)
    wi, wsi, xi, xsi = synthetic.integer_operands(512, 4096, 8, seed=4)
    ints = [run_chain(wi, wsi, xi, xsi, s, fold=f)[0] for s, f in tactics]
    assert all((i == ints[0]).all() for i in ints)


@pytest.mark.parametrize("fold", [1, 4])
@pytest.mark.parametrize("stages", [2, 3, 7, 12])
def test_every_ring_depth(cuda, stages, fold):
    w, ws, x, xs = synthetic.integer_operands(256, 4096, 8, seed=stages)
    want = oracle.gemm_bf16(w, ws, x, xs)
    if stages * (16 + fold + 0.5) * 1024 > 227 * 1024:  # W, x and scale rings alone
        with pytest.raises(Mxfp8Error, match="ERR_UNSUPPORTED"):
            run_chain(w, ws, x, xs, 1, stages=stages, fold=fold)
        return
    c, *_, cfg = run_chain(w, ws, x, xs, 1, stages=stages, fold=fold)
    assert cfg["stages"] == stages and cfg["fold"] == fold
    assert (c == want).all()


@pytest.mark.parametrize("fold", [1, 4])
@pytest.mark.parametrize("stages", [2, 4, 5, 7, 10])
def test_short_rings_over_a_long_k_loop(cuda, stages, fold):
    """128 K tiles per CTA (32 folded stages) through a short ring, ten
    chained calls, with the default pipes for the ring (4, 2 or 1: each slot
    owned by one producer lane and one MMA issuer); every call bit-exact."""
    n, k = 1024, 16384
    w, ws, x, xs = synthetic.integer_operands(n, k, 8, seed=100 + stages)
    want = oracle.gemm_bf16(w, ws, x, xs)
    mb = Mailbox(8, n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=1, stages=stages, fold=fold)
    assert (g.config()["stages"], g.config()["fold"]) == (stages, fold)
    X, XS = dev(x), dev(xs)
    for call in range(10):
        c = torch.full((8, n), 0x7FFF, dtype=torch.int16, device="cuda")
        g.run(X, XS, c)
        out = mb.consume(8)
        torch.cuda.synchronize()
        assert (bits(c) == want).all(), f"C, call {call}"
        assert (bits(out) == sanitized(want)).all(), f"consumer output, call {call}"
    assert mb.status()[0] == OK and state_words(mb) == [10 % 3, 9 % 3, 0, 0]
    g.close()


def test_default_pipes_divide_the_ring(cuda):
    """Grids of at most one CTA per SM get 4 pipes on a ring that is a
    multiple of 4 (2 at fold 8, whose accumulator ring has 2 slots); the
    headline's two CTAs per SM get 2."""
    for n, k, split, pipes in [(2048, 16384, 1, 2), (4096, 4096, 1, 4), (7168, 8192, 2, 4),
                               (7168, 16384, 4, 2)]:
        w = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
        ws = torch.full((n, k // 32), 127, dtype=torch.uint8, device="cuda")
        g = PublishGemm(w, ws, Mailbox(8, n), split_k=split)
        cfg = g.config()
        assert cfg["pipes"] == pipes and cfg["stages"] % pipes == 0, cfg
        g.close()


def test_default_fold(cuda):
    """The largest fold that keeps the grid within one CTA per SM, pads K no
    further and leaves every split a stage (fold 8 only unsplit, from 8 stages
    per CTA, and not with 4 pipes asked for); 1 where the tactic asks for what
    folding does not take (one slot per MMA, the 16x256b read-out, S = 8)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    assert sms >= 128
    for n, k, split, extra, fold in [(4096, 4096, 1, {}, 4), (2048, 16384, 1, {}, 8),
                                     (2048, 4096, 1, {}, 4), (2048, 16384, 1, {"pipes": 4}, 4),
                                     (2048, 2048, 4, {}, 2), (7168, 8192, 2, {}, 1),
                                     (7168, 16384, 4, {}, 1), (4096, 4096, 1, {"acc_blocks": 1}, 1),
                                     (4096, 4096, 1, {"tmem_load": TMEM_LOAD_16X256B}, 1),
                                     (256, 2048, 8, {}, 1), (256, 96, 1, {}, 1), (256, 384, 1, {}, 1),
                                     (256, 512, 1, {}, 4), (256, 512, 2, {}, 2), (256, 256, 2, {}, 1),
                                     (256, 256, 4, {}, 1)]:
        w = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
        ws = torch.full((n, k // 32), 127, dtype=torch.uint8, device="cuda")
        g = PublishGemm(w, ws, Mailbox(8, n), split_k=split, **extra)
        cfg = g.config()
        assert cfg["fold"] == fold, (n, k, split, extra, cfg)
        assert cfg["grid_ctas"] == n // (128 // fold) * split, cfg
        assert cfg["tmem_columns"] <= 256, cfg
        g.close()


def test_plan_matches_create(cuda):
    """mxfp8_publish_gemm_plan, given this device's limits, resolves every
    tactic field, the shared memory, tensor-memory columns and grid exactly as
    creating the handle does."""
    from mxfp8_gemm_mailbox_gb300 import plan_gemm
    props = torch.cuda.get_device_properties(0)
    limits = (props.multi_processor_count,
              getattr(props, "shared_memory_per_multiprocessor", 233472),
              props.shared_memory_per_block_optin)
    for n, k, kw in [(7168, 16384, dict(split_k=4)), (7168, 8192, dict(split_k=2)),
                     (4096, 4096, dict(split_k=1)), (256, 256, dict(split_k=1)),
                     (2048, 2048, dict()), (1024, 4096, dict(split_k=2, stages=4)),
                     (512, 1152, dict(split_k=4, fold=2, l2_prefetch=3)),
                     (384, 8192, dict(acc_blocks=1, tmem_load=TMEM_LOAD_16X256B))]:
        w = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
        ws = torch.full((n, k // 32), 127, dtype=torch.uint8, device="cuda")
        g = PublishGemm(w, ws, Mailbox(8, n), **kw)
        assert plan_gemm(n, k, limits=limits, **kw) == g.config(), (n, k, kw)
        g.close()


def test_at_most_two_ctas_per_sm(cuda):
    """A clustered launch asks for more than a third of an SM's shared memory,
    short rings included, so at most two of its CTAs (each holding at most 256
    of the SM's 512 tensor-memory columns) share an SM and no allocation waits
    on a cluster peer; every launch holds at most 256 columns."""
    props = torch.cuda.get_device_properties(0)
    per_sm = getattr(props, "shared_memory_per_multiprocessor", 233472)
    for n, k, split, stages in [(128, 128, 4, 0), (256, 256, 1, 0), (128, 32, 8, 2),
                                (256, 512, 2, 2), (1024, 4096, 4, 2), (7168, 16384, 4, 0)]:
        w = torch.zeros((n, k), dtype=torch.uint8, device="cuda")
        ws = torch.full((n, k // 32), 127, dtype=torch.uint8, device="cuda")
        g = PublishGemm(w, ws, Mailbox(8, n), split_k=split, stages=stages)
        cfg = g.config()
        if split > 1:
            assert 3 * (cfg["smem_bytes"] + 1024) > per_sm, cfg  # 1 KB reserved per CTA
        assert cfg["tmem_columns"] <= 256, cfg
        g.close()


@pytest.mark.parametrize("fold", [1, 2, 4])
@pytest.mark.parametrize("stages,pipes", [(8, 4), (4, 4), (8, 2), (6, 2), (5, 1), (8, 1)])
def test_every_pipe_count_over_a_long_k_loop(cuda, stages, pipes, fold):
    """Each pipe count (producer lanes = MMA-issuing warps) on a ring it
    divides, 128 K tiles per CTA (128 / fold stages), five chained calls,
    bit-exact."""
    n, k = 1024, 16384
    w, ws, x, xs = synthetic.integer_operands(n, k, 8, seed=200 + stages * 8 + pipes)
    want = oracle.gemm_bf16(w, ws, x, xs)
    mb = Mailbox(8, n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=1, stages=stages, pipes=pipes, fold=fold)
    assert (g.config()["stages"], g.config()["pipes"], g.config()["fold"]) == (stages, pipes, fold)
    X, XS = dev(x), dev(xs)
    for call in range(5):
        c = torch.full((8, n), 0x7FFF, dtype=torch.int16, device="cuda")
        g.run(X, XS, c)
        out = mb.consume(8)
        torch.cuda.synchronize()
        assert (bits(c) == want).all(), f"C, call {call}"
        assert (bits(out) == sanitized(want)).all(), f"consumer output, call {call}"
    assert mb.status()[0] == OK
    g.close()


@pytest.mark.parametrize("fold", [1, 4])
@pytest.mark.parametrize("w_layout", [W_IN_PLACE, W_TILED])
@pytest.mark.parametrize("l2_prefetch,l2_prefetch_early", [(-1, 0), (0, 0), (3, 0), (40, 0),
                                                           (0, -1), (12, 2), (-1, 30)])
def test_l2_prefetch_leaves_results_unchanged(cuda, l2_prefetch, l2_prefetch_early, w_layout,
                                              fold):
    """Warming later W stages in L2 before the grid wait (the defaults: 16 for
    the later CTAs, 4 or none for the first 70 %; none; a few; more than the
    CTA has; different depths for the two groups) is bit-exact."""
    n, k = 512, 8192
    w, ws, x, xs = synthetic.integer_operands(n, k, 8, seed=300 + l2_prefetch)
    want = oracle.gemm_bf16(w, ws, x, xs)
    for split in (1, 4):
        mb = Mailbox(8, n)
        g = PublishGemm(dev(w), dev(ws), mb, split_k=split, w_layout=w_layout,
                        l2_prefetch=l2_prefetch, l2_prefetch_early=l2_prefetch_early, fold=fold)
        grid_ctas = n // (128 // fold) * split
        assert g.config()["grid_ctas"] == grid_ctas
        two_per_sm = grid_ctas > torch.cuda.get_device_properties(0).multi_processor_count
        assert g.config()["l2_prefetch"] == (16 if l2_prefetch == 0 else l2_prefetch)
        early = (l2_prefetch_early if l2_prefetch_early != 0 else
                 l2_prefetch if l2_prefetch != 0 else 4 if two_per_sm else -1)
        assert g.config()["l2_prefetch_early"] == early
        c = torch.full((8, n), 0x7FFF, dtype=torch.int16, device="cuda")
        g.run(dev(x), dev(xs), c)
        out = mb.consume(8)
        torch.cuda.synchronize()
        assert (bits(c) == want).all() and (bits(out) == sanitized(want)).all()
        assert mb.status()[0] == OK
        g.close()


@pytest.mark.parametrize("tmem_load", [1, 2])
@pytest.mark.parametrize("n,k,m", [(256, 2048, 8), (1024, 8192, 5), (384, 1152, 1), (128, 4096, 8)])
def test_split_eight_one_token_per_cta(cuda, n, k, m, tmem_load):
    """Split-K over a cluster of 8: each CTA owns one token and receives the
    other seven CTAs' (hi, lo) pairs for it in 8-byte stores; ragged K, every
    m (CTAs whose token is past m publish nothing), bit-exact on integer
    inputs and within 2 ULP on N(0, 1) ones, and the consumer's output."""
    wi, wsi, xi, xsi = synthetic.integer_operands(n, k, m, seed=n + k + m)
    c, between, sb, out, after, state, cfg = run_chain(wi, wsi, xi, xsi, 8)
    assert cfg["split_k"] == 8 and cfg["grid_ctas"] == (n // 128) * 8
    want = oracle.gemm_bf16(wi, wsi, xi, xsi)
    assert (c == want).all() and (out == sanitized(want)).all()
    check_published(between, sb, c, 8, n)
    wl = synthetic.Workload("s8", n, k, m, 8, exp_lo=-5, exp_hi=3, seed=n * 3 + m)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    mb = Mailbox(8, n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=8, tmem_load=tmem_load)
    cc = torch.full((m, n), 0x7FFF, dtype=torch.int16, device="cuda")
    g.run(dev(x), dev(xs), cc)
    o = mb.consume(m)
    torch.cuda.synchronize()
    assert_bf16_close(bits(cc), oracle.gemm_bf16(w, ws, x, xs))
    assert (bits(o) == sanitized(bits(cc))).all() and mb.status()[0] == OK
    g.close()


@pytest.mark.parametrize("acc_blocks", [1, 4])
@pytest.mark.parametrize("split_k", [1, 2, 4, 8])
def test_tmem_load_shapes_give_identical_bits(cuda, split_k, acc_blocks):
    """The 16x256b accumulator read-out (the gemm page's default shape) and
    the 32x32b one (its column_lanes = 1 case) fold each element's partial
    sums in the same order: C, the mailbox and the consumer output agree bit
    for bit, and both match the oracle (bit-exact on integer inputs, within
    2 ULP on N(0, 1) inputs)."""
    wl = synthetic.Workload("loads", 768, 6144, 7, split_k, exp_lo=-5, exp_hi=3, seed=41)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    wi, wsi, xi, xsi = synthetic.integer_operands(768, 6144, 8, seed=42)
    for (ww, wws, xx, xxs, exact) in ((w, ws, x, xs, False), (wi, wsi, xi, xsi, True)):
        got = {}
        for load in (TMEM_LOAD_32X32B, TMEM_LOAD_16X256B):
            mb = Mailbox(8, 768)
            g = PublishGemm(dev(ww), dev(wws), mb, split_k=split_k, acc_blocks=acc_blocks,
                            tmem_load=load, fold=1)
            assert g.config()["tmem_load"] == {1: "32x32b", 2: "16x256b"}[load]
            m = xx.shape[0]
            c = torch.full((m, 768), 0x7FFF, dtype=torch.int16, device="cuda")
            g.run(dev(xx), dev(xxs), c)
            torch.cuda.synchronize()
            words = mailbox_words(mb).copy()
            out = mb.consume(m)
            torch.cuda.synchronize()
            got[load] = (bits(c), words, bits(out))
            assert mb.status()[0] == OK
            g.close()
        a, b = got[TMEM_LOAD_32X32B], got[TMEM_LOAD_16X256B]
        assert (a[0] == b[0]).all() and (a[1] == b[1]).all() and (a[2] == b[2]).all()
        want = oracle.gemm_bf16(ww, wws, xx, xxs)
        if exact:
            assert (b[0] == want).all()
        else:
            assert_bf16_close(b[0], want)


def test_pipes_that_do_not_divide_the_ring_are_refused(cuda):
    w, ws, x, xs = synthetic.integer_operands(256, 4096, 8, seed=1)
    with pytest.raises(Mxfp8Error, match="ERR_UNSUPPORTED"):
        PublishGemm(dev(w), dev(ws), Mailbox(8, 256), split_k=1, stages=6, pipes=4)


@pytest.mark.parametrize("fold", [1, 4])
@pytest.mark.parametrize("split_k", [1, 2, 4])
def test_longest_k(cuda, split_k, fold):
    """K = 32768, the largest K taken: 256 K tiles per CTA at S = 1 (the most a
    split holds; 64 stages of 4 pieces folded), every output bit-exact
    (integer inputs keep every partial sum below 2^24)."""
    n, k, m = 256, 32768, 8
    w, ws, x, xs = synthetic.integer_operands(n, k, m, seed=77 + split_k)
    c, between, sb, out, after, state, cfg = run_chain(w, ws, x, xs, split_k, fold=fold)
    assert cfg["split_k"] == split_k and cfg["fold"] == fold
    want = oracle.gemm_bf16(w, ws, x, xs)
    assert (c == want).all() and (out == sanitized(want)).all()
    check_published(between, sb, c, 8, n)


def test_grid_of_two_waves(cuda):
    """N = 16384, K = 32768, S = 4: 512 CTAs, more than the GPU holds at once
    (two per SM), so the clusters run in waves; for m = 8 and m = 1, 2,048
    sampled outputs of C and of the consumer against the oracle, bit-exact on
    integer inputs, and a clean mailbox after every call."""
    n, k = 16384, 32768
    w, ws, x, xs = synthetic.integer_operands(n, k, 8, seed=91)
    mb = Mailbox(8, n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=4)
    assert g.config()["grid_ctas"] == 512
    rng = np.random.default_rng(5)
    for m in (8, 1):
        rows = rng.integers(0, m, 2048)
        cols = rng.integers(0, n, 2048)
        want = oracle.gemm_sample(w, ws, x[:m], xs[:m], rows, cols)
        c = torch.full((m, n), 0x7FFF, dtype=torch.int16, device="cuda")
        g.run(dev(x[:m]), dev(xs[:m]), c)
        out = mb.consume(m)
        torch.cuda.synchronize()
        assert (bits(c)[rows, cols] == want).all(), f"C, m={m}"
        assert (bits(out)[rows, cols] == sanitized(want)).all(), f"consumer, m={m}"
        assert mb.status()[0] == OK and (mailbox_words(mb) == oracle.SENTINEL).all()
    g.close()


@pytest.mark.parametrize("fold,split_k", [(1, 1), (2, 1), (4, 1), (8, 1), (1, 4), (2, 4), (4, 4)])
@pytest.mark.parametrize("shift", [100, -100, 60])
def test_scale_exponents_near_the_e8m0_limits(cuda, shift, split_k, fold):
    """W's scales moved up by `shift` powers of two and x's down by as many
    (E8M0 codes from 27 to 228): every product, hence every output, is
    unchanged, and exact; the scale plumbing must carry the extreme codes."""
    n, k, m = 384, 4096, 8
    w, ws, x, xs = synthetic.integer_operands(n, k, m, seed=500 + shift)
    want = oracle.gemm_bf16(w, ws, x, xs)
    ws_s = (ws.astype(np.int32) + shift).astype(np.uint8)
    xs_s = (xs.astype(np.int32) - shift).astype(np.uint8)
    assert (oracle.gemm_bf16(w, ws_s, x, xs_s) == want).all()
    c, between, sb, out, after, state, cfg = run_chain(w, ws_s, x, xs_s, split_k, fold=fold)
    assert cfg["fold"] == fold
    assert (c == want).all() and (out == sanitized(want)).all()


def test_ring_too_deep_for_shared_memory_is_refused(cuda):
    w, ws, x, xs = synthetic.integer_operands(256, 4096, 8, seed=1)
    with pytest.raises(Mxfp8Error, match="ERR_UNSUPPORTED"):
        PublishGemm(dev(w), dev(ws), Mailbox(8, 256), split_k=1, stages=16)


@pytest.mark.parametrize("acc_blocks", [1, 4])
@pytest.mark.parametrize("split_k", [1, 4])
def test_accumulation_granularity(cuda, acc_blocks, split_k):
    w, ws, x, xs = synthetic.integer_operands(512, 4096, 8, seed=17)
    want = oracle.gemm_bf16(w, ws, x, xs)
    c, between, sb, out, after, state, cfg = run_chain(w, ws, x, xs, split_k,
                                                      acc_blocks=acc_blocks, fold=1)
    assert cfg["acc_blocks"] == acc_blocks
    assert (c == want).all()
    check_published(between, sb, c, 8, 512)
    assert (out == sanitized(c)).all()


def test_negative_zero_is_cleared_in_the_mailbox_only(cuda):
    # Tiny negative sums round to -0 in BF16 (-2^-136 below half the smallest
    # subnormal); other rows are exactly +0 / -0 products.
    n, k, m = 256, 64, 4
    w = np.full((n, k), 0x38, np.uint8)
    ws = np.full((n, k // 32), 0x01, np.uint8)       # 2^-126
    x = np.full((m, k), 0xB8, np.uint8)              # -1
    xs = np.full((m, k // 32), 0x70, np.uint8)       # 2^-15
    w[128:] = 0x80                                   # -0 weights
    x[3] = 0x00
    want = oracle.gemm_bf16(w, ws, x, xs)
    c, between, sb, out, after, state, _ = run_chain(w, ws, x, xs, 1)
    assert_bf16_close(c, want)
    pub = between[0, :m]
    assert not ((pub & 0xFFFF) == 0x8000).any() and not ((pub >> 16) == 0x8000).any()
    assert (out == sanitized(c)).all()
    assert not (out == 0x8000).any()


@pytest.mark.parametrize("fold", [1, 2])
def test_capacity_and_row_limits(cuda, fold):
    w, ws, x, xs = synthetic.integer_operands(128, 256, 3, seed=1)
    mb = Mailbox(3, 128)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=1, fold=fold)
    g.precompile(3)
    with pytest.raises(Mxfp8Error, match="ERR_UNSUPPORTED"):
        g.precompile(4)
    x4 = dev(np.zeros((4, 256), np.uint8))
    with pytest.raises(Mxfp8Error, match="ERR_UNSUPPORTED"):
        g.run(x4, dev(np.full((4, 8), 127, np.uint8)))
    c = torch.empty((3, 128), dtype=torch.int16, device="cuda")
    g.run(dev(x), dev(xs), c)
    out = mb.consume(3)
    torch.cuda.synchronize()
    want = oracle.gemm_bf16(w, ws, x, xs)
    assert (bits(c) == want).all() and (bits(out) == sanitized(want)).all()
    assert mb.status()[0] == OK


@pytest.mark.parametrize("fold", [1, 0])
def test_fused_equals_unfused_bit_for_bit(cuda, fold):
    # The unfused path: the GEMM writes only C, the standalone publish kernel
    # reads it back; mailbox and consumer output must match the fused epilogue
    # (unfolded, and with the default fold, 4 here).
    wl = synthetic.Workload("u", 1024, 2048, 7, 2, exp_lo=-6, exp_hi=3, signed_pairs=True, seed=11)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    W, WS, X, XS = dev(w), dev(ws), dev(x), dev(xs)
    fused_mb, unfused_mb = Mailbox(8, 1024), Mailbox(8, 1024)
    gf = PublishGemm(W, WS, fused_mb, split_k=2, fold=fold)
    gu = PublishGemm(W, WS, unfused_mb, split_k=2, fold=fold)
    assert gf.config()["fold"] == gu.config()["fold"] == (fold or 4)
    for call in range(4):  # walk the generations
        cf = torch.empty((7, 1024), dtype=torch.int16, device="cuda")
        cu = torch.empty((7, 1024), dtype=torch.int16, device="cuda")
        gf.run(X, XS, cf)
        gu.run_unfused(X, XS, cu)
        unfused_mb.publish(cu)
        torch.cuda.synchronize()
        assert (bits(cf) == bits(cu)).all()
        assert (mailbox_words(fused_mb) == mailbox_words(unfused_mb)).all()
        assert state_words(fused_mb) == state_words(unfused_mb)
        of = fused_mb.consume(7)
        ou = unfused_mb.consume(7)
        torch.cuda.synchronize()
        assert (bits(of) == bits(ou)).all()
        assert state_words(fused_mb) == state_words(unfused_mb) == [(call + 1) % 3, call % 3, 0, 0]
    assert_bf16_close(bits(cf), oracle.gemm_bf16(w, ws, x, xs))


@pytest.mark.parametrize("fold", [1, 2])
def test_publish_without_c(cuda, fold):
    w, ws, x, xs = synthetic.integer_operands(256, 512, 8, seed=2)
    mb = Mailbox(8, 256)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=2, fold=fold)
    g.run(dev(x), dev(xs), None)
    out = mb.consume(8)
    torch.cuda.synchronize()
    assert (bits(out) == sanitized(oracle.gemm_bf16(w, ws, x, xs))).all()


@pytest.mark.parametrize("fold", [1, 2])
def test_bad_next_generation_is_flagged(cuda, fold):
    w, ws, x, xs = synthetic.integer_operands(128, 256, 2, seed=5)
    mb = Mailbox(8, 128)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=1, fold=fold)
    mb.state[0] = 4
    c = torch.empty((2, 128), dtype=torch.int16, device="cuda")
    g.run(dev(x), dev(xs), c)
    torch.cuda.synchronize()
    assert (mailbox_words(mb) == oracle.SENTINEL).all()  # no publish into a bad generation
    assert (bits(c) == oracle.gemm_bf16(w, ws, x, xs)).all()  # C is still written
    assert mb.status()[0] == ERR_STATE


@pytest.mark.parametrize("fold,alpha,split_k",
                         [(f, a, s) for f in (1, 0) for a, s in ((0.25, 1), (-1.7, 2), (3.0e-3, 4),
                                                                 (1.0, 4))] +
                         [(8, 0.25, 1), (8, -1.7, 1)])
def test_global_scale(cuda, alpha, split_k, fold):
    wl = synthetic.Workload("alpha", 768, 4096, 6, split_k, exp_lo=-4, exp_hi=2, seed=91)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    want = oracle.gemm_bf16_scaled(w, ws, x, xs, alpha)
    mb = Mailbox(8, 768)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=split_k, fold=fold)
    a = torch.tensor([alpha], dtype=torch.float32, device="cuda")
    c = torch.empty((6, 768), dtype=torch.bfloat16, device="cuda")
    g.run_scaled(dev(x), dev(xs), a, c)
    out = mb.consume(6)
    torch.cuda.synchronize()
    assert_bf16_close(bits(c), want, f"alpha={alpha}")
    assert (bits(out) == sanitized(bits(c))).all()
    # integer inputs with a power-of-two scale stay exact
    wi, wsi, xi, xsi = synthetic.integer_operands(768, 4096, 6, seed=3)
    g2 = PublishGemm(dev(wi), dev(wsi), Mailbox(8, 768), split_k=split_k, fold=fold)
    a2 = torch.tensor([0.5], dtype=torch.float32, device="cuda")
    g2.run_scaled(dev(xi), dev(xsi), a2, c)
    g2.mailbox.consume(6)
    torch.cuda.synchronize()
    assert (bits(c) == oracle.gemm_bf16_scaled(wi, wsi, xi, xsi, 0.5)).all()
    g.run_scaled(dev(x), dev(xs), None, c)  # NULL alpha is the plain run
    mb.consume(6)
    torch.cuda.synchronize()
    assert_bf16_close(bits(c), oracle.gemm_bf16(w, ws, x, xs))


@pytest.mark.parametrize("w_layout", [W_TILED, W_IN_PLACE])
def test_first_run_right_after_create_on_one_stream(cuda, w_layout):
    # Through the C ABI with no host synchronisation between create and the
    # first run: create's re-layout kernels write the scale chunks (and the
    # tiled weight) that the GEMM's producer reads before its grid wait, so
    # the handle's first launch takes a full stream dependency.  Several fresh
    # handles, each run once right away, must all match the oracle.
    import ctypes

    from mxfp8_gemm_mailbox_gb300 import _lib

    lib = _lib.load()
    stream = torch.cuda.Stream()
    sp = ctypes.c_void_p(stream.cuda_stream)
    n, k, m = 2048, 4096, 8
    for seed in range(4):
        wl = synthetic.Workload("first-run", n, k, m, 2, exp_lo=-4, exp_hi=2, seed=900 + seed)
        w, ws = synthetic.make_weights(wl)
        x, xs = synthetic.make_activations(wl)
        W, WS, X, XS = dev(w), dev(ws), dev(x), dev(xs)
        mb = Mailbox(8, n)
        desc = _lib.GemmDesc(n, k, 8, 2, 0, 0, 0, w_layout)
        ws_bytes = lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(desc))
        workspace = torch.empty(ws_bytes, dtype=torch.uint8, device="cuda")
        c = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        out = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        torch.cuda.synchronize()  # inputs and the armed mailbox are in place
        handle = ctypes.c_void_p()
        ptr = lambda t: ctypes.c_void_p(t.data_ptr())
        assert lib.mxfp8_publish_gemm_create(ctypes.byref(desc), ptr(W), ptr(WS), ptr(mb.words),
                                             ptr(mb.state), ptr(workspace), ws_bytes, sp,
                                             ctypes.byref(handle)) == OK
        assert lib.mxfp8_publish_gemm_run(handle, ptr(X), ptr(XS), m, ptr(c), sp) == OK
        assert lib.mailbox_consume(ptr(mb.words), ptr(mb.state), 8, n, m, ptr(out), 0, sp) == OK
        stream.synchronize()
        lib.mxfp8_publish_gemm_destroy(handle)
        want = oracle.gemm_bf16(w, ws, x, xs)
        assert_bf16_close(bits(c), want, f"seed {seed}")
        assert (bits(out) == sanitized(bits(c))).all()
        assert state_words(mb) == [1, 0, 0, 0]


# cta_k 256: two K tiles per pipeline stage.  Each tile's MMAs still fill one
# accumulator slot and the epilogue adds the slots in tile order, so every
# result is bit-identical to cta_k 128's.  Cases: a partial last stage (odd
# tile counts, ragged K), rings refilled many times, split-K 2 and 4, folds 2
# and 4 (whose 4-slot accumulator ring takes at most 2 pipes), 4 pipes at
# fold 2, both weight layouts.
K256_CASES = [
    # n, k, m, split_k, fold, w_layout, stages, pipes
    (256, 384, 3, 1, 1, W_TILED, 0, 0),
    (256, 352, 8, 1, 1, W_IN_PLACE, 0, 0),
    (512, 4096, 8, 1, 1, W_TILED, 2, 0),
    (512, 4096, 5, 2, 1, W_IN_PLACE, 4, 2),
    (768, 3072, 8, 4, 1, W_TILED, 0, 0),
    (1024, 4096, 4, 1, 4, W_TILED, 0, 0),
    (1024, 4096, 8, 2, 2, W_IN_PLACE, 0, 0),
    (256, 1536, 8, 1, 4, W_TILED, 0, 0),
    (256, 1664, 6, 2, 4, W_IN_PLACE, 2, 1),
    (2048, 16384, 8, 1, 2, W_TILED, 4, 4),
    (1024, 8192, 8, 4, 2, W_TILED, 3, 1),
]


@pytest.mark.parametrize("case", K256_CASES, ids=lambda c: "n%d-k%d-m%d-s%d-f%d-w%d-st%d-p%d" % c)
def test_cta_k_256_matches_cta_k_128(cuda, case):
    n, k, m, split_k, fold, w_layout, stages, pipes = case
    wl = synthetic.Workload("cta_k", n, k, m, split_k, exp_lo=-4, exp_hi=2, seed=n + k + m)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    ref = run_chain(w, ws, x, xs, split_k, w_layout=w_layout, fold=fold)
    got = run_chain(w, ws, x, xs, split_k, w_layout=w_layout, fold=fold, stages=stages,
                    pipes=pipes, cta_k=256)
    cfg = got[-1]
    assert cfg["cta_k"] == 256 and cfg["fold"] == fold and cfg["split_k"] == split_k
    if stages:
        assert cfg["stages"] == stages
    ring = 4 if fold == 4 else 8
    assert ring % (2 * cfg["pipes"]) == 0 and cfg["stages"] % cfg["pipes"] == 0
    for a, b, what in ((ref[0], got[0], "C"), (ref[1], got[1], "mailbox"),
                       (ref[3], got[3], "consumer output"), (ref[4], got[4], "mailbox after")):
        assert (a == b).all(), what
    assert ref[2] == got[2] and ref[5] == got[5]
    assert_bf16_close(got[0], oracle.gemm_bf16(w, ws, x, xs), "C vs oracle")


@pytest.mark.parametrize("case", K256_CASES[:6], ids=lambda c: "n%d-k%d-m%d-s%d-f%d-w%d-st%d-p%d" % c)
def test_cta_k_256_integer_inputs_bit_exact(cuda, case):
    n, k, m, split_k, fold, w_layout, stages, pipes = case
    w, ws, x, xs = synthetic.integer_operands(n, k, m, seed=k + 7)
    want = oracle.gemm_bf16(w, ws, x, xs)
    c, between, state_between, out, after, state_after, cfg = run_chain(
        w, ws, x, xs, split_k, w_layout=w_layout, fold=fold, stages=stages, pipes=pipes,
        cta_k=256)
    assert cfg["cta_k"] == 256
    assert (c == want).all()
    check_published(between, state_between, c, 8, n)
    assert (out == sanitized(want)).all()
    assert (after == oracle.SENTINEL).all() and state_after == [1, 0, 0, 0]


def test_cta_k_256_chained_calls(cuda):
    # Ten chained calls through one handle: the two-tile stages' barriers,
    # slots and ring refills hold across calls.
    n, k = 1024, 16384
    w, ws, x, xs = synthetic.integer_operands(n, k, 8, seed=256)
    want = oracle.gemm_bf16(w, ws, x, xs)
    mb = Mailbox(8, n)
    g = PublishGemm(dev(w), dev(ws), mb, split_k=1, cta_k=256, stages=3, fold=2)
    assert (g.config()["cta_k"], g.config()["stages"]) == (256, 3)
    X, XS = dev(x), dev(xs)
    for call in range(10):
        c = torch.full((8, n), 0x7FFF, dtype=torch.int16, device="cuda")
        g.run(X, XS, c)
        out = mb.consume(8)
        torch.cuda.synchronize()
        assert (bits(c) == want).all(), f"C, call {call}"
        assert (bits(out) == sanitized(want)).all(), f"consumer output, call {call}"
    assert mb.status()[0] == OK and state_words(mb) == [10 % 3, 9 % 3, 0, 0]
    g.close()
