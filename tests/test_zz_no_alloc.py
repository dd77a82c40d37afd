"""The allocation-free publishing GEMM against the handle-based one.

Some callers cannot allocate device memory at the point they issue work
(inside a runtime that owns all device memory in a fixed pool, on an issue
path where an allocation could synchronise the device, from a C host with no
allocator), so
the library offers ``mxfp8_publish_gemm_run_noalloc``: no handle, no
workspace, W read in place and its scale chunks re-laid into the library's
own static scratch array on every call.  This file runs last in the suite;
it passes alone in a fresh process and after every other test.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import synthetic
from mxfp8_gemm_mailbox_gb300 import OK, Mailbox, PublishGemm, _lib
from tests.gpu_util import (assert_bf16_close, bits, dev, mailbox_words, pack_words, sanitized,
                            state_words)

pytestmark = pytest.mark.gpu


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(None)


@pytest.mark.parametrize("fold,cta_k", [(1, 0), (0, 0), (0, 256)])
def test_noalloc_matches_the_handle_path_on_two_calls(cuda, fold, cta_k):
    # Two calls in a row, each with its own weight scales: the second call's
    # re-layout overwrites the scratch the first call's GEMM read, and its
    # GEMM must see the new chunks.  Both paths run the same kernel with the
    # same tactic and summation order, so they agree bit for bit.
    lib = _lib.load()
    n, k, m, split = 1024, 4096, 5, 2
    desc = _lib.GemmDesc(n, k, 8, split, cta_k, 0, 0, 0, 0, 0, 0, fold)
    handle_mb, noalloc_mb = Mailbox(8, n), Mailbox(8, n)
    for call in range(2):
        wl = synthetic.Workload("noalloc", n, k, m, split, exp_lo=-4, exp_hi=2, seed=4242 + call)
        w, ws = synthetic.make_weights(wl)
        W, WS = dev(w), dev(ws)
        gemm = PublishGemm(W, WS, handle_mb, split_k=split, w_layout=_lib.W_IN_PLACE, fold=fold,
                           cta_k=cta_k)
        assert gemm.config()["fold"] == (fold or 4)  # 8 tiles x 2 splits fold 4 ways by default
        assert gemm.config()["cta_k"] == (cta_k or 128)
        x, xs = synthetic.make_activations(wl, salt=call)
        X, XS = dev(x), dev(xs)
        c_handle = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        c_noalloc = torch.empty((m, n), dtype=torch.bfloat16, device="cuda")
        gemm.run(X, XS, c_handle)
        out_handle = handle_mb.consume(m)
        status = lib.mxfp8_publish_gemm_run_noalloc(
            ctypes.byref(desc), _ptr(W), _ptr(WS), _ptr(X), _ptr(XS), m, _ptr(c_noalloc),
            _ptr(noalloc_mb.words), _ptr(noalloc_mb.state), _stream())
        assert status == OK, lib.mxfp8_last_error().decode()
        between = mailbox_words(noalloc_mb)
        out_noalloc = noalloc_mb.consume(m)
        torch.cuda.synchronize()
        assert (bits(c_noalloc) == bits(c_handle)).all(), f"C differs, call {call}"
        assert (bits(out_noalloc) == bits(out_handle)).all(), f"consumer output differs, call {call}"
        assert (between[call % 3, :m] == pack_words(sanitized(bits(c_handle)))).all(), call
        assert_bf16_close(bits(c_noalloc), oracle.gemm_bf16(w, ws, x, xs), f"vs oracle, call {call}")
        assert state_words(noalloc_mb) == state_words(handle_mb) == [(call + 1) % 3, call % 3, 0, 0]
        assert (mailbox_words(noalloc_mb) == oracle.SENTINEL).all()
        gemm.close()
    assert noalloc_mb.status()[0] == OK


def test_noalloc_refuses_what_does_not_fit(cuda):
    lib = _lib.load()
    mb = Mailbox(8, 128)
    dummy = torch.zeros(64, dtype=torch.uint8, device="cuda")
    big = _lib.GemmDesc(16384, 32768, 8, 4, 0, 0, 0, 0, 0)  # 16 MiB of scale chunks
    status = lib.mxfp8_publish_gemm_run_noalloc(
        ctypes.byref(big), _ptr(dummy), _ptr(dummy), _ptr(dummy), _ptr(dummy), 1, None,
        _ptr(mb.words), _ptr(mb.state), _stream())
    assert status == _lib.ERR_UNSUPPORTED
    assert "scratch" in lib.mxfp8_last_error().decode()
    tiled = _lib.GemmDesc(128, 256, 8, 1, 0, 0, 0, _lib.W_TILED, 0)
    status = lib.mxfp8_publish_gemm_run_noalloc(
        ctypes.byref(tiled), _ptr(dummy), _ptr(dummy), _ptr(dummy), _ptr(dummy), 1, None,
        _ptr(mb.words), _ptr(mb.state), _stream())
    assert status == _lib.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert (mailbox_words(mb) == oracle.SENTINEL).all() and mb.status()[0] == OK
