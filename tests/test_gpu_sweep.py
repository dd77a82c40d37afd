"""The sweep: m in 1..8, N in {2048, 4096, 7168}, K in {2048, 4096, 8192,
16384}, S in {1, 2, 4} (288 cases), with x rows in +/- pairs and duplicated
and zero W rows, so some outputs are exactly +0 or -0 and the mailbox's
negative-zero clearing is exercised.  Every case against the oracle."""
import numpy as np
import pytest
import torch

import oracle
import synthetic
from mxfp8_gemm_mailbox_gb300 import OK, Mailbox, PublishGemm
from tests.gpu_util import bf16_mismatches, bits, dev, describe, mailbox_words, sanitized

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("n", synthetic.SWEEP_N)
@pytest.mark.parametrize("k", synthetic.SWEEP_K)
def test_sweep(cuda, n, k):
    # One weight and one 8-row activation per (N, K); m rows use the first m.
    wl = synthetic.sweep_workload(8, n, k, 1)
    w, ws = synthetic.make_weights(wl)
    x, xs = synthetic.make_activations(wl)
    want = oracle.gemm_bf16(w, ws, x, xs)
    exact_zero = oracle.gemm_fp64(w, ws, x, xs) == 0.0
    assert exact_zero.any()
    W, WS, X, XS = dev(w), dev(ws), dev(x), dev(xs)
    failures = []
    calls = 0
    for s in synthetic.SWEEP_S:
        mb = Mailbox(8, n)
        g = PublishGemm(W, WS, mb, split_k=s)
        for m in synthetic.SWEEP_M:
            c = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
            g.run(X[:m], XS[:m], c)
            out = mb.consume(m)
            torch.cuda.synchronize()
            got, o = bits(c), bits(out)
            bad = bf16_mismatches(got, want[:m])
            if bad.any():
                failures.append(f"m={m} S={s}: {describe(got, want[:m])}")
            if not (o == sanitized(got)).all():
                failures.append(f"m={m} S={s}: consumer output != sanitised C")
            if (o == 0x8000).any() or (o.view(np.uint32) == oracle.SENTINEL).any():
                failures.append(f"m={m} S={s}: -0 or sentinel in the consumer output")
            z = exact_zero[:m]
            if not ((got[z] & 0x7FFF) == 0).all() or not (o[z] == 0).all():
                failures.append(f"m={m} S={s}: exact zeros not +/-0 in C or not +0 in out")
            for j in range(0, m - 1, 2):  # sign pairs: C[2j+1] = -C[2j]
                nz = (got[j] & 0x7FFF) != 0
                if not ((got[j + 1][nz] ^ 0x8000) == got[j][nz]).all() or (
                        (got[j + 1][~nz] & 0x7FFF) != 0).any():
                    failures.append(f"m={m} S={s}: row {j + 1} is not -row {j}")
            if not (mailbox_words(mb) == oracle.SENTINEL).all():
                failures.append(f"m={m} S={s}: mailbox not reset")
            calls += 1
        st, words = mb.status()
        if st != OK or words[:3] != [len(synthetic.SWEEP_M) % 3, (len(synthetic.SWEEP_M) - 1) % 3, 0]:
            failures.append(f"S={s}: status {st} state {words}")
        g.close()
    assert calls == 24
    assert not failures, "\n".join(failures[:20])
