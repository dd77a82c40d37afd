"""MXFP8 low-batch decode projection with a Lamport-mailbox publishing
epilogue, for one GB300 (sm_103a).

The compute path is the CUDA library ``libmxfp8_mailbox.so`` (C ABI in
``include/mxfp8_mailbox.h``); this package only marshals arguments to it.
"""
from . import _lib
from ._lib import (ERR_CUDA, ERR_INVALID, ERR_STATE, ERR_TIMEOUT, ERR_UNSUPPORTED,
                   FLAG_BAD_STATE, FLAG_GEMM_TIMEOUT, FLAG_POLL_TIMEOUT, OK, Mxfp8Error)
from .api import LamportGather, Mailbox, PublishGemm, TaggedMailbox, plan_gemm

__all__ = ["LamportGather", "Mailbox", "TaggedMailbox", "PublishGemm", "plan_gemm", "Mxfp8Error",
           "OK", "ERR_INVALID", "ERR_UNSUPPORTED",
           "ERR_CUDA", "ERR_TIMEOUT", "ERR_STATE", "FLAG_POLL_TIMEOUT", "FLAG_GEMM_TIMEOUT",
           "FLAG_BAD_STATE"]
