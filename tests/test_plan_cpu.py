"""The tactic resolver on the CPU, through mxfp8_publish_gemm_plan: the plans
of the benchmarked workloads on GB300's limits, the invariants every plan
keeps over a grid of shapes and tactics (tensor memory within half an SM,
shared memory within a CTA's limit and covering every region the kernel
addresses, at most two CTAs of a clustered launch per SM, pipes dividing the
ring, folding only where it is taken and pads K no further), the refusals,
and how the fold follows the SM count."""
import itertools

import pytest

from mxfp8_gemm_mailbox_gb300 import Mxfp8Error, plan_gemm
from mxfp8_gemm_mailbox_gb300._lib import TMEM_LOAD_16X256B

SMS, SMEM_PER_SM, SMEM_OPTIN = 152, 233472, 232448


def test_plans_of_the_benchmarked_workloads():
    want = {
        (7168, 16384, 4): dict(fold=1, stages=6, pipes=2, l2_prefetch=16, l2_prefetch_early=4,
                               smem_bytes=113280, tmem_columns=128, grid_ctas=224),
        (7168, 8192, 2): dict(fold=1, stages=12, pipes=4, l2_prefetch=16, l2_prefetch_early=-1,
                              smem_bytes=224992, tmem_columns=256, grid_ctas=112),
        (4096, 4096, 1): dict(fold=4, stages=8, pipes=4, l2_prefetch=16, l2_prefetch_early=-1,
                              smem_bytes=173728, tmem_columns=256, grid_ctas=128),
        (256, 256, 1): dict(fold=2, stages=2, pipes=2, grid_ctas=4),
    }
    for (n, k, s), fields in want.items():
        plan = plan_gemm(n, k, split_k=s)
        got = {f: plan[f] for f in fields}
        assert got == fields, ((n, k, s), plan)
        assert plan["w_layout"] == "tiled" and plan["tmem_load"] == "32x32b"
        assert plan["acc_blocks"] == 4 and plan["cta_k"] == 128


def _k_tiles(k, fold):
    return -(-k // (128 * fold))


def _kernel_smem_need(plan, k):
    """Shared memory the kernel addresses for a plan, from its layout: the W,
    x and W-scale rings, the x-scale staging (a 16-byte row per MMA column,
    32 rows at most, per K tile of the split, plus the 384 bytes a 32-row
    copy of the last 128-byte chunk reads past it), 2 barriers per stage, 2
    per accumulator slot (8 at most) and 2 more, 16 bytes of words, and 1 KB
    to align the base to the 128-byte swizzle's 1024-byte period."""
    f, s, st = plan["fold"], plan["split_k"], plan["stages"]
    tps = -(-_k_tiles(k, f) // s)
    rings = st * (16384 + 1024 * f + 512)
    staging = tps * 16 * min(8 * f, 32) + 384
    return rings + staging + (2 * st + 2 * 8 + 2) * 8 + 16 + 1024


def _epilogue_fits_the_dead_ring(plan):
    """After the main loop the epilogue reuses the W ring: W stage 0 holds the
    BF16 tile (below 4 KB) and, folded, the parked pairs (8 KB from 4 KB);
    W stage 1 the split-K receive buffer."""
    f, s = plan["fold"], plan["split_k"]
    shard, rows = 8 // s, 128 // f
    run = min(8 // f, shard) if f > 1 else shard
    recv = (s - 1) * (128 if f > 1 else rows) * run * 8
    return (plan["stages"] >= 2 and shard * rows * 2 <= 4096 and 4096 + 128 * 8 * 8 <= 16384
            and recv <= 16384)


TACTICS = list(itertools.product([0, 1, 2, 4, 8], [0, 2, 3, 6, 12, 16], [0, 1, 4], [0, 1, 2, 4],
                                 [0, 1, 2, 4, 8], [0, TMEM_LOAD_16X256B]))


@pytest.mark.parametrize("n", [128, 256, 1024, 2048, 4096, 7168, 16384])
def test_every_plan_keeps_the_invariants(n):
    accepted = 0
    for k in (32, 96, 256, 1152, 4096, 16384, 32768):
        for split, stages, acc, pipes, fold, load in TACTICS:
            try:
                p = plan_gemm(n, k, split_k=split, stages=stages, acc_blocks=acc, pipes=pipes,
                              fold=fold, tmem_load=load)
            except Mxfp8Error as e:
                assert "ERR_UNSUPPORTED" in str(e), (n, k, split, stages, acc, pipes, fold, load)
                continue
            accepted += 1
            where = (n, k, split, stages, acc, pipes, fold, load, p)
            assert p["tmem_columns"] <= 256, where
            assert p["smem_bytes"] <= SMEM_OPTIN, where
            assert p["stages"] % p["pipes"] == 0, where
            assert p["grid_ctas"] == n // (128 // p["fold"]) * p["split_k"], where
            assert p["smem_bytes"] >= _kernel_smem_need(p, k), where
            assert _epilogue_fits_the_dead_ring(p), where
            # tensor memory: the accumulator ring (slots of 8 x fold columns, or
            # 32 with one slot per MMA; 2 slots at fold 8, 4 at fold 4 or one
            # per MMA, else 8) and a 4-column W-scale and x-scale slot per stage
            f = p["fold"]
            slot = 32 if p["acc_blocks"] == 1 else 8 * f
            ring = 2 if f == 8 else 4 if (f == 4 or p["acc_blocks"] == 1) else 8
            assert p["tmem_columns"] >= slot * ring + 8 * p["stages"], where
            assert p["tmem_columns"] in (32, 64, 128, 256), where
            # the epilogue stages at most 16 x-scale words per thread (128 threads)
            assert min(8 * p["fold"], 32) * -(-_k_tiles(k, p["fold"]) // p["split_k"]) <= 2048, where
            if p["split_k"] > 1:  # at most two CTAs of a clustered launch on an SM
                assert 3 * (p["smem_bytes"] + 1024) > SMEM_PER_SM, where
            for field, asked in (("split_k", split), ("stages", stages), ("acc_blocks", acc),
                                 ("pipes", pipes), ("fold", fold)):
                if asked:
                    assert p[field] == asked, where
            if p["fold"] == 8:  # its accumulator ring has 2 slots
                assert p["split_k"] == 1 and p["pipes"] <= 2, where
                if fold == 0:  # chosen only from 8 stages per CTA
                    assert _k_tiles(k, 8) >= 8, where
            if p["fold"] > 1:
                assert p["split_k"] <= 4 and p["acc_blocks"] == 4, where
                assert p["tmem_load"] == "32x32b", where
                if fold == 0:  # chosen: one CTA per SM at most, no more K padding
                    assert p["grid_ctas"] <= SMS, where
                    assert _k_tiles(k, p["fold"]) * p["fold"] == _k_tiles(k, 1), where
                    assert _k_tiles(k, p["fold"]) >= p["split_k"], where
            early = p["l2_prefetch_early"]
            assert p["l2_prefetch"] == 16 and early == (4 if p["grid_ctas"] > SMS else -1), where
    assert accepted > 0


def test_refusals_match_create():
    bad = [dict(fold=2, split_k=8), dict(fold=4, acc_blocks=1), dict(fold=2, tmem_load=2),
           dict(fold=3), dict(split_k=3), dict(stages=6, pipes=4), dict(l2_prefetch_early=65),
           dict(stages=1), dict(fold=8, split_k=2), dict(fold=8, pipes=4), dict(fold=8)]
    for kw in bad:
        with pytest.raises(Mxfp8Error, match="ERR_UNSUPPORTED"):
            plan_gemm(1024, 4096, **kw)
    with pytest.raises(Mxfp8Error, match="ERR_INVALID"):
        plan_gemm(200, 4096)
    with pytest.raises(Mxfp8Error, match="ERR_INVALID"):
        plan_gemm(1024, 4096, limits=(0, SMEM_PER_SM, SMEM_OPTIN))


def test_the_fold_follows_the_sm_count():
    # N=4096, K=4096, S=1: 32 tiles fold 4 ways on 152 SMs (128 CTAs); with 100
    # SMs four ways would not fit one CTA per SM, so two.
    assert plan_gemm(4096, 4096, split_k=1)["fold"] == 4
    assert plan_gemm(4096, 4096, split_k=1, limits=(100, SMEM_PER_SM, SMEM_OPTIN))["fold"] == 2
    assert plan_gemm(4096, 4096, split_k=1, limits=(40, SMEM_PER_SM, SMEM_OPTIN))["fold"] == 1


def test_split_choice_when_left_open():
    # S = 0: the largest of 2, 4 with at most two CTAs per SM and >= 2 K tiles
    # per split.
    assert plan_gemm(7168, 16384)["split_k"] == 4
    assert plan_gemm(16384, 16384)["split_k"] == 2
    assert plan_gemm(2048, 256)["split_k"] == 1
    assert plan_gemm(2048, 2048)["grid_ctas"] == 2048 // 64 * 4  # S = 4, fold 2


def test_gemm_wait_limit_field():
    # The GEMM's pipeline waits give up after wait_limit_ms: 0 asks for the
    # default of 2 s, an explicit value is kept, values outside 1..60000 are
    # refused before anything launches.
    assert plan_gemm(7168, 16384, split_k=4)["wait_limit_ms"] == 2000
    assert plan_gemm(7168, 16384, split_k=4, wait_limit_ms=1)["wait_limit_ms"] == 1
    assert plan_gemm(4096, 4096, wait_limit_ms=60000)["wait_limit_ms"] == 60000
    for bad in (-1, 60001):
        with pytest.raises(Mxfp8Error, match="ERR_UNSUPPORTED.*wait_limit_ms"):
            plan_gemm(4096, 4096, wait_limit_ms=bad)
    # the limit changes nothing else of the plan
    a, b = plan_gemm(7168, 8192, split_k=2), plan_gemm(7168, 8192, split_k=2, wait_limit_ms=5)
    assert {k: v for k, v in a.items() if k != "wait_limit_ms"} == \
        {k: v for k, v in b.items() if k != "wait_limit_ms"}


def test_split_k_receive_buffer_of_its_own_where_it_fits():
    # With split-K the peers' partials get a region of their own (so a CTA can
    # send as soon as its main loop is done) when it fits beside the resolved
    # ring within the ring's per-SM budget: N=7168, K=8192, S=2 (one CTA per
    # SM) takes (2-1) x 128 x 4 x 8 = 4096 more bytes than its ring layout; the
    # headline (two CTAs per SM, 6-stage ring) has no room for 6144 and keeps
    # the partials in its dead W ring.
    assert plan_gemm(7168, 8192, split_k=2)["smem_bytes"] == 220896 + 4096
    assert plan_gemm(7168, 16384, split_k=4)["smem_bytes"] == 113280
    # unsplit launches have no partials to exchange
    assert plan_gemm(4096, 4096, split_k=1)["smem_bytes"] == 173728



@pytest.mark.parametrize("n", [256, 2048, 4096, 7168])
def test_cta_k_256_plans_keep_the_invariants(n):
    # Two K tiles per stage: rings of 2 x stages tiles, a 4-column W-scale and
    # x-scale slot per tile, and every accumulator slot owned by one issuer
    # (the ring of 8 slots, 4 at fold 4, a multiple of 2 x pipes).
    accepted = 0
    for k in (256, 384, 1536, 4096, 16384):
        for split, stages, pipes, fold in itertools.product([0, 1, 2, 4], [0, 2, 3, 4, 6, 8],
                                                            [0, 1, 2, 4], [0, 1, 2, 4]):
            try:
                p = plan_gemm(n, k, split_k=split, stages=stages, pipes=pipes, fold=fold,
                              cta_k=256)
            except Mxfp8Error as e:
                assert "ERR_UNSUPPORTED" in str(e), (n, k, split, stages, pipes, fold)
                continue
            accepted += 1
            where = (n, k, split, stages, pipes, fold, p)
            f, st = p["fold"], p["stages"]
            assert p["cta_k"] == 256 and f in (1, 2, 4), where
            ring = 4 if f == 4 else 8
            assert ring % (2 * p["pipes"]) == 0 and st % p["pipes"] == 0, where
            assert p["tmem_columns"] <= 256, where
            assert p["tmem_columns"] >= 8 * f * ring + 2 * 4 * 2 * st, where
            tps = -(-_k_tiles(k, f) // p["split_k"])
            rings = 2 * st * (16384 + 1024 * f + 512)
            staging = tps * 16 * min(8 * f, 32) + 384
            assert p["smem_bytes"] >= rings + staging + (2 * st + 2 * 8 + 2) * 8 + 16 + 1024, where
            for field, asked in (("split_k", split), ("stages", stages), ("pipes", pipes),
                                 ("fold", fold)):
                if asked:
                    assert p[field] == asked, where
    assert accepted > 0


def test_cta_k_refusals():
    for kw in (dict(cta_k=384), dict(cta_k=64), dict(cta_k=256, fold=8),
               dict(cta_k=256, split_k=8), dict(cta_k=256, acc_blocks=1),
               dict(cta_k=256, tmem_load=TMEM_LOAD_16X256B),
               dict(cta_k=256, fold=4, stages=4, pipes=4)):  # 4 slots cannot serve 4 pipes x 2
        with pytest.raises(Mxfp8Error, match="ERR_UNSUPPORTED"):
            plan_gemm(1024, 4096, **kw)
    # the default stays 128, and 256 resolves with the pipes its ring allows
    assert plan_gemm(4096, 4096)["cta_k"] == 128
    p = plan_gemm(4096, 4096, split_k=1, cta_k=256)
    assert p["cta_k"] == 256 and p["fold"] == 4 and p["pipes"] <= 2
