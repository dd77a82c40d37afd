"""Thin Python binding over the C ABI: argument marshalling only.

PyTorch provides device memory and streams; every step of the path runs in the
library's CUDA kernels.  Names follow the C ABI (``include/mxfp8_mailbox.h``).
"""
from __future__ import annotations

import ctypes

import torch

from . import _lib
from ._lib import GemmDesc, check


def _ptr(t: torch.Tensor | None):
    return ctypes.c_void_p(t.data_ptr()) if t is not None else ctypes.c_void_p(None)


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    handle = stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)
    return ctypes.c_void_p(handle)


def _synchronize(stream, device) -> None:
    """Waits for the work issued so far on ``stream`` (as ``_stream`` reads it)."""
    if stream is None:
        torch.cuda.current_stream(device).synchronize()
    elif hasattr(stream, "synchronize"):
        stream.synchronize()
    elif int(stream) == 0:  # the legacy default stream waits for the whole device
        torch.cuda.synchronize(device)
    else:
        torch.cuda.ExternalStream(int(stream), device=device).synchronize()


def _on_device(t: torch.Tensor, name: str) -> None:
    if not t.is_cuda or not t.is_contiguous():
        raise ValueError(f"{name} must be a contiguous CUDA tensor")


def _codes(t: torch.Tensor, name: str, cols: int, min_rows: int = 0) -> int:
    """Checks a matrix of one-byte codes (E4M3 or E8M0) ``[rows][cols]`` with
    at least ``min_rows`` rows; returns rows.  The kernels read rows x cols
    bytes from its address, so a smaller tensor is refused here, where its
    size is still known."""
    if t.element_size() != 1:
        raise TypeError(f"{name} must hold one-byte codes (uint8 / float8), got {t.dtype}")
    if t.dim() != 2 or t.shape[1] != cols or t.shape[0] < min_rows:
        raise ValueError(f"{name} must be [rows >= {min_rows}][{cols}], got {tuple(t.shape)}")
    _on_device(t, name)
    return t.shape[0]


def _halves(t: torch.Tensor, name: str, min_rows: int, cols: int) -> int:
    """Checks a matrix of two-byte values (BF16 bits) ``[rows][cols]`` with at
    least ``min_rows`` rows, which the kernels write or read row by row;
    returns rows."""
    if t.element_size() != 2:
        raise TypeError(f"{name} must hold two-byte values (bfloat16 / int16), got {t.dtype}")
    if t.dim() != 2 or t.shape[1] != cols or t.shape[0] < min_rows:
        raise ValueError(f"{name} must be [rows >= {min_rows}][{cols}], got {tuple(t.shape)}")
    _on_device(t, name)
    return t.shape[0]


class Mailbox:
    """A 3-generation Lamport mailbox ``[3][capacity_m][n]`` BF16 and its four
    state words ``[next generation, active generation, arrivals, flags]``."""

    def __init__(self, capacity_m: int, n: int, device=None, stream=None):
        lib = _lib.load()
        nbytes = lib.mxfp8_mailbox_bytes(capacity_m, n)
        if nbytes == 0:
            raise ValueError(f"invalid mailbox shape capacity_m={capacity_m}, n={n}")
        device = torch.device(device or "cuda")
        self.capacity = capacity_m
        self.n = n
        self.words = torch.empty(nbytes // 4, dtype=torch.int32, device=device)
        self.state = torch.zeros(4, dtype=torch.int32, device=device)
        self.init(stream)

    def init(self, stream=None) -> None:
        check(_lib.load().mxfp8_mailbox_init(_ptr(self.words), _ptr(self.state), self.capacity,
                                             self.n, _stream(stream)), "mxfp8_mailbox_init")

    def publish(self, c: torch.Tensor, stream=None) -> None:
        """The unfused path's standalone publish of C [m][n] BF16."""
        m = _halves(c, "c", 0, self.n)
        check(_lib.load().mailbox_publish(_ptr(self.words), _ptr(self.state), self.capacity,
                                          self.n, m, _ptr(c), _stream(stream)),
              "mailbox_publish")

    def consume(self, m: int, out: torch.Tensor | None = None, timeout_ns: int = 0,
                stream=None) -> torch.Tensor:
        """The consumer: [m][n] BF16 copied out of the active generation."""
        if out is None:
            out = torch.empty((m, self.n), dtype=torch.bfloat16, device=self.words.device)
        _halves(out, "out", m, self.n)
        check(_lib.load().mailbox_consume(_ptr(self.words), _ptr(self.state), self.capacity,
                                          self.n, m, _ptr(out), timeout_ns, _stream(stream)),
              "mailbox_consume")
        return out

    def status(self, stream=None):
        """(status code, [4] state words); synchronises the stream."""
        words = (ctypes.c_int32 * 4)()
        st = _lib.load().mxfp8_mailbox_status(_ptr(self.state), words, _stream(stream))
        return st, list(words)


def _config_dict(d: GemmDesc, smem: int, tmem: int, grid: int) -> dict:
    return {"n": d.n, "k": d.k, "capacity_m": d.capacity_m, "split_k": d.split_k,
            "cta_k": d.cta_k, "stages": d.stages, "acc_blocks": d.acc_blocks,
            "w_layout": {1: "in_place", 2: "tiled"}.get(d.w_layout, d.w_layout),
            "l2_prefetch": d.l2_prefetch, "l2_prefetch_early": d.l2_prefetch_early,
            "pipes": d.pipes,
            "tmem_load": {1: "32x32b", 2: "16x256b"}.get(d.tmem_load, d.tmem_load),
            "fold": d.fold, "wait_limit_ms": d.wait_limit_ms, "smem_bytes": smem,
            "tmem_columns": tmem, "grid_ctas": grid}


# GB300: SMs, shared memory per SM, shared memory per CTA at most.
GB300_LIMITS = (152, 233472, 232448)


def plan_gemm(n: int, k: int, capacity_m: int = 8, split_k: int = 0, stages: int = 0,
              acc_blocks: int = 0, w_layout: int = 0, l2_prefetch: int = 0, pipes: int = 0,
              tmem_load: int = 0, fold: int = 0, l2_prefetch_early: int = 0,
              wait_limit_ms: int = 0, cta_k: int = 0, limits: tuple = GB300_LIMITS) -> dict:
    """The tactic PublishGemm would resolve for this shape on a device with
    `limits` = (SMs, shared memory per SM, shared memory per CTA), as
    PublishGemm.config() reports it; needs no GPU."""
    desc = GemmDesc(n, k, capacity_m, split_k, cta_k, stages, acc_blocks, w_layout, l2_prefetch,
                    pipes, tmem_load, fold, l2_prefetch_early, wait_limit_ms)
    out = GemmDesc()
    smem, tmem, grid = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
    check(_lib.load().mxfp8_publish_gemm_plan(ctypes.byref(desc), *limits, ctypes.byref(out),
                                              ctypes.byref(smem), ctypes.byref(tmem),
                                              ctypes.byref(grid)), "mxfp8_publish_gemm_plan")
    return _config_dict(out, smem.value, tmem.value, grid.value)


class PublishGemm:
    """One MXFP8 weight ``W [N][K]`` (E4M3 codes) with its scales ``[N][K/32]``
    (E8M0 codes), publishing into ``mailbox``.  The weight, mailbox and the
    workspace this object allocates stay borrowed by the native handle until
    :meth:`close`.

    The library's create launches the weight re-layout on ``stream`` (the
    current stream by default), and a run must come after it; this
    constructor waits for that stream, so runs may then be issued on any
    stream."""

    def __init__(self, w: torch.Tensor, w_scale: torch.Tensor, mailbox: Mailbox,
                 split_k: int = 0, stages: int = 0, acc_blocks: int = 0, w_layout: int = 0,
                 l2_prefetch: int = 0, pipes: int = 0, tmem_load: int = 0, fold: int = 0,
                 l2_prefetch_early: int = 0, wait_limit_ms: int = 0, cta_k: int = 0,
                 stream=None):
        lib = _lib.load()
        if w.dim() != 2:
            raise ValueError(f"w must be [N][K], got {tuple(w.shape)}")
        n, k = w.shape
        _codes(w, "w", k)
        if k % 32 == 0:  # other K are refused by the library below
            _codes(w_scale, "w_scale", k // 32, min_rows=n)
        self.desc = GemmDesc(n, k, mailbox.capacity, split_k, cta_k, stages, acc_blocks,
                             w_layout, l2_prefetch, pipes, tmem_load, fold, l2_prefetch_early,
                             wait_limit_ms)
        ws_bytes = lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(self.desc))
        if ws_bytes == 0:
            raise ValueError(f"invalid GEMM shape N={n}, K={k}")
        self.workspace = torch.empty(ws_bytes, dtype=torch.uint8, device=w.device)
        self.w = w
        self.mailbox = mailbox
        self.n, self.k = n, k
        handle = ctypes.c_void_p()
        check(lib.mxfp8_publish_gemm_create(ctypes.byref(self.desc), _ptr(w), _ptr(w_scale),
                                            _ptr(mailbox.words), _ptr(mailbox.state),
                                            _ptr(self.workspace), ws_bytes, _stream(stream),
                                            ctypes.byref(handle)), "mxfp8_publish_gemm_create")
        self._handle = handle
        # The re-layout kernels create launched must finish before a run on
        # another stream reads the workspace.
        _synchronize(stream, w.device)

    def config(self) -> dict:
        d = GemmDesc()
        smem, tmem, grid = ctypes.c_int32(), ctypes.c_int32(), ctypes.c_int32()
        check(_lib.load().mxfp8_publish_gemm_config(self._handle, ctypes.byref(d),
                                                    ctypes.byref(smem), ctypes.byref(tmem),
                                                    ctypes.byref(grid)), "mxfp8_publish_gemm_config")
        return _config_dict(d, smem.value, tmem.value, grid.value)

    def precompile(self, m: int) -> None:
        check(_lib.load().mxfp8_publish_gemm_precompile(self._handle, m),
              "mxfp8_publish_gemm_precompile")

    def run(self, x: torch.Tensor, x_scale: torch.Tensor, c: torch.Tensor | None = None,
            stream=None) -> torch.Tensor | None:
        """One publishing GEMM on x [m][K]; writes C [m][N] BF16 into ``c`` if
        given.  Must be followed by exactly one ``mailbox.consume``."""
        m = self._rows(x, x_scale, c)
        check(_lib.load().mxfp8_publish_gemm_run(self._handle, _ptr(x), _ptr(x_scale), m,
                                                 _ptr(c), _stream(stream)), "mxfp8_publish_gemm_run")
        return c

    def run_scaled(self, x: torch.Tensor, x_scale: torch.Tensor, alpha: torch.Tensor | None,
                   c: torch.Tensor | None = None, stream=None) -> torch.Tensor | None:
        """``run`` with C = alpha * (W x); alpha a one-element float32 CUDA tensor."""
        if alpha is not None and (alpha.dtype != torch.float32 or not alpha.is_cuda):
            raise TypeError("alpha must be a float32 CUDA tensor")
        m = self._rows(x, x_scale, c)
        check(_lib.load().mxfp8_publish_gemm_run_scaled(self._handle, _ptr(x), _ptr(x_scale),
                                                        m, _ptr(alpha), _ptr(c),
                                                        _stream(stream)),
              "mxfp8_publish_gemm_run_scaled")
        return c

    def run_unfused(self, x: torch.Tensor, x_scale: torch.Tensor, c: torch.Tensor,
                    stream=None) -> torch.Tensor:
        m = self._rows(x, x_scale, c)
        check(_lib.load().mxfp8_gemm_run_unfused(self._handle, _ptr(x), _ptr(x_scale), m,
                                                 _ptr(c), _stream(stream)), "mxfp8_gemm_run_unfused")
        return c

    def _rows(self, x: torch.Tensor, x_scale: torch.Tensor, c: torch.Tensor | None) -> int:
        """m, after checking x [m][K], x_scale [>= m][K/32] and C [>= m][N]."""
        m = _codes(x, "x", self.k)
        _codes(x_scale, "x_scale", self.k // 32, min_rows=m)
        if c is not None:
            _halves(c, "c", m, self.n)
        return m

    def close(self) -> None:
        if getattr(self, "_handle", None):
            _lib.load().mxfp8_publish_gemm_destroy(self._handle)
            self._handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


class LamportGather:
    """The one-rank Lamport all-gather on its own mailbox of ``capacity_bytes``
    (a multiple of 16): ``gather(x)`` returns x's words with 0x80000000 words
    cleared, through the publish / poll / reset protocol."""

    def __init__(self, capacity_bytes: int, device=None, stream=None):
        lib = _lib.load()
        nbytes = lib.lamport_gather_mailbox_bytes(capacity_bytes)
        if nbytes == 0:
            raise ValueError(f"invalid gather capacity {capacity_bytes}")
        device = torch.device(device or "cuda")
        self.capacity = capacity_bytes
        self.words = torch.empty(nbytes // 4, dtype=torch.int32, device=device)
        self.state = torch.zeros(4, dtype=torch.int32, device=device)
        check(lib.lamport_gather_init(_ptr(self.words), _ptr(self.state), capacity_bytes,
                                      _stream(stream)), "lamport_gather_init")

    def accepts(self, inp: torch.Tensor) -> bool:
        return 0 < inp.nbytes <= self.capacity and inp.nbytes % 16 == 0

    def __call__(self, inp: torch.Tensor, out: torch.Tensor | None = None, timeout_ns: int = 0,
                 stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty_like(inp)
        _on_device(inp, "inp")
        _on_device(out, "out")
        if out.nbytes < inp.nbytes:
            raise ValueError(f"out holds {out.nbytes} bytes, fewer than the input's {inp.nbytes}")
        check(_lib.load().lamport_all_gather(_ptr(self.words), _ptr(self.state), self.capacity,
                                             _ptr(inp), inp.nbytes, _ptr(out), timeout_ns,
                                             _stream(stream)), "lamport_all_gather")
        return out

    def status(self, stream=None):
        words = (ctypes.c_int32 * 4)()
        st = _lib.load().mxfp8_mailbox_status(_ptr(self.state), words, _stream(stream))
        return st, list(words)


class TaggedMailbox:
    """The tagged-pair mailbox ``[capacity_m][n/2]`` of (value word, tag):
    ``publish(c, tag)`` stores C with a nonzero tag; ``consume(m, tag)`` reads
    it back once every tag matches.  Nothing is reset; BF16 bits move
    unchanged."""

    def __init__(self, capacity_m: int, n: int, device=None, stream=None):
        lib = _lib.load()
        nbytes = lib.tagged_mailbox_bytes(capacity_m, n)
        if nbytes == 0:
            raise ValueError(f"invalid tagged mailbox shape capacity_m={capacity_m}, n={n}")
        device = torch.device(device or "cuda")
        self.capacity, self.n = capacity_m, n
        self.pairs = torch.empty(nbytes // 4, dtype=torch.int32, device=device)
        self.flags = torch.zeros(1, dtype=torch.int32, device=device)
        check(lib.tagged_mailbox_init(_ptr(self.pairs), capacity_m, n, _stream(stream)),
              "tagged_mailbox_init")

    def publish(self, c: torch.Tensor, tag: int, stream=None) -> None:
        m = _halves(c, "c", 0, self.n)
        check(_lib.load().tagged_publish(_ptr(self.pairs), self.capacity, self.n, m,
                                         _ptr(c), tag, _stream(stream)), "tagged_publish")

    def consume(self, m: int, tag: int, out: torch.Tensor | None = None, timeout_ns: int = 0,
                stream=None) -> torch.Tensor:
        if out is None:
            out = torch.empty((m, self.n), dtype=torch.bfloat16, device=self.pairs.device)
        _halves(out, "out", m, self.n)
        check(_lib.load().tagged_consume(_ptr(self.pairs), self.capacity, self.n, m, tag,
                                         _ptr(out), timeout_ns, _ptr(self.flags),
                                         _stream(stream)), "tagged_consume")
        return out
