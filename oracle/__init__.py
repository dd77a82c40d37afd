"""CPU oracle for the MXFP8 publishing GEMM and its Lamport mailbox.

TEST INFRASTRUCTURE ONLY.  Only the tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference legs may import this package.  The CUDA
library never links, loads or calls it, and this package imports nothing from
the CUDA side: the two share only the seeded input generator (``synthetic``),
which holds none of the method's arithmetic.

The arithmetic lives in plain C (``mxfp8_oracle.c``, compiled with gcc by
:func:`build`); this module only marshals numpy arrays through ctypes.  Each C
function cites the passage of the source pages it follows:

* page "vllm.models.deepseek_v41.nvidia.specialized_decode.boundary.
  publishing_gemm": the MXFP8 product, its BF16 rounding, the negative-zero
  clearing and the publish into ``mailbox[stage_state[0]]``;
* page "vllm.models.deepseek_v41.nvidia.ops.cute_dsl.all_gather": the sentinel,
  the three generations and the consume (poll, copy out, reset, advance).

Parity unpinned: nothing.  Every function here is pinned by ``-m "not gpu"``
tests against something other than itself (exact rational sums, closed forms,
a library float64 matmul, torch's float8 decoding, worked examples under
``tests/golden``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
from pathlib import Path

import numpy as np

_HERE = Path(__file__).resolve().parent
_SOURCE = _HERE / "mxfp8_oracle.c"
_LIBRARY = _HERE / "liboracle.so"

GENERATIONS = 3
SENTINEL = 0x80000000

OK = 0
ERR_ARGS = 1
ERR_SENTINEL = 4
ERR_STATE = 5


def build(force: bool = False) -> Path:
    """Compile ``mxfp8_oracle.c`` into ``liboracle.so`` (gcc, -O2, no fast-math,
    no FMA contraction, so every operation is the IEEE one written)."""
    if not force and _LIBRARY.exists() and _LIBRARY.stat().st_mtime >= _SOURCE.stat().st_mtime:
        return _LIBRARY
    tmp = _LIBRARY.with_suffix(f".{os.getpid()}.tmp")
    cmd = [
        "gcc", "-O2", "-std=c11", "-fPIC", "-shared", "-ffp-contract=off",
        "-fno-fast-math", str(_SOURCE), "-o", str(tmp), "-lm",
    ]
    subprocess.run(cmd, check=True)
    os.replace(tmp, _LIBRARY)
    return _LIBRARY


_lib = None


def use_library(path) -> None:
    """Load the oracle from another build of ``mxfp8_oracle.c`` (the tests use
    this to run the pins against deliberately broken copies); ``None`` goes
    back to the default library."""
    global _lib
    _lib = None
    if path is not None:
        _load(Path(path))


def _load(path: Path | None = None):
    global _lib
    if _lib is not None and path is None:
        return _lib
    if path is None:
        build()
        path = _LIBRARY
    lib = ctypes.CDLL(str(path))
    u8p = ctypes.POINTER(ctypes.c_uint8)
    u16p = ctypes.POINTER(ctypes.c_uint16)
    u32p = ctypes.POINTER(ctypes.c_uint32)
    i32p = ctypes.POINTER(ctypes.c_int32)
    f64p = ctypes.POINTER(ctypes.c_double)
    i = ctypes.c_int
    lib.oracle_e4m3_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e4m3_value.restype = ctypes.c_double
    lib.oracle_e8m0_value.argtypes = [ctypes.c_uint8]
    lib.oracle_e8m0_value.restype = ctypes.c_double
    lib.oracle_bf16_rne.argtypes = [ctypes.c_double]
    lib.oracle_bf16_rne.restype = ctypes.c_uint16
    lib.oracle_clear_negative_zero.argtypes = [ctypes.c_uint16]
    lib.oracle_clear_negative_zero.restype = ctypes.c_uint16
    lib.oracle_gemm_fp64.argtypes = [i, i, i, u8p, u8p, u8p, u8p, f64p]
    lib.oracle_gemm_bf16.argtypes = [i, i, i, u8p, u8p, u8p, u8p, u16p]
    lib.oracle_gemm_bf16_scaled.argtypes = [i, i, i, u8p, u8p, u8p, u8p, ctypes.c_float, u16p]
    lib.oracle_gemm_sample.argtypes = [i, i, i, u8p, u8p, u8p, u8p, i, i32p, i32p, u16p]
    lib.oracle_mailbox_init.argtypes = [u32p, i32p, i, i]
    lib.oracle_publish.argtypes = [u32p, i32p, i, i, i, u16p]
    lib.oracle_consume.argtypes = [u32p, i32p, i, i, i, u16p]
    lib.oracle_chain.argtypes = [i, i, i, u8p, u8p, u8p, u8p, u32p, i32p, i, u16p, u16p]
    lib.oracle_tagged_init.argtypes = [u32p, i, i]
    lib.oracle_tagged_publish.argtypes = [u32p, i, i, i, u16p, ctypes.c_uint32]
    lib.oracle_tagged_consume.argtypes = [u32p, i, i, i, ctypes.c_uint32, u16p]
    lib.oracle_gather_init.argtypes = [u32p, i32p, i]
    lib.oracle_all_gather.argtypes = [u32p, i32p, i, u32p, i, u32p]
    for name in ("oracle_gemm_fp64", "oracle_gemm_bf16", "oracle_gemm_bf16_scaled",
                 "oracle_gemm_sample",
                 "oracle_mailbox_init", "oracle_publish", "oracle_consume", "oracle_chain",
                 "oracle_gather_init", "oracle_all_gather", "oracle_tagged_init",
                 "oracle_tagged_publish", "oracle_tagged_consume"):
        getattr(lib, name).restype = ctypes.c_int
    _lib = lib
    return lib


def _ptr(array: np.ndarray, ctype):
    assert array.flags["C_CONTIGUOUS"]
    return array.ctypes.data_as(ctypes.POINTER(ctype))


def _u8(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint8:
        raise TypeError(f"expected uint8 bytes, got {a.dtype}")
    return a


def e4m3_value(code: int) -> float:
    """Exact value of one E4M3FN code."""
    return _load().oracle_e4m3_value(code)


def e8m0_value(code: int) -> float:
    """Exact value of one E8M0FNU scale code, 2^(code - 127)."""
    return _load().oracle_e8m0_value(code)


def bf16_rne(value: float) -> int:
    """BF16 bits of a double, rounded once to nearest, ties to even."""
    return _load().oracle_bf16_rne(float(value))


def clear_negative_zero(half: int) -> int:
    return _load().oracle_clear_negative_zero(half)


def _check_shapes(w, ws, x, xs):
    n, k = w.shape
    m = x.shape[0]
    if k % 32 or ws.shape != (n, k // 32) or x.shape != (m, k) or xs.shape != (m, k // 32):
        raise ValueError("shapes: W [N][K], W scales [N][K/32], x [m][K], x scales [m][K/32]")
    return n, k, m


def gemm_fp64(w, ws, x, xs) -> np.ndarray:
    """acc[t][n] = sum_k W[n, k] x[t, k] in FP64 (k ascending)."""
    w, ws, x, xs = map(_u8, (w, ws, x, xs))
    n, k, m = _check_shapes(w, ws, x, xs)
    acc = np.empty((m, n), dtype=np.float64)
    st = _load().oracle_gemm_fp64(n, k, m, _ptr(w, ctypes.c_uint8), _ptr(ws, ctypes.c_uint8),
                                  _ptr(x, ctypes.c_uint8), _ptr(xs, ctypes.c_uint8),
                                  _ptr(acc, ctypes.c_double))
    if st != OK:
        raise ValueError(f"oracle_gemm_fp64 status {st}")
    return acc


def gemm_bf16(w, ws, x, xs) -> np.ndarray:
    """C [m][N] as uint16 BF16 bits (rounded once from FP64, RNE)."""
    w, ws, x, xs = map(_u8, (w, ws, x, xs))
    n, k, m = _check_shapes(w, ws, x, xs)
    c = np.empty((m, n), dtype=np.uint16)
    st = _load().oracle_gemm_bf16(n, k, m, _ptr(w, ctypes.c_uint8), _ptr(ws, ctypes.c_uint8),
                                  _ptr(x, ctypes.c_uint8), _ptr(xs, ctypes.c_uint8),
                                  _ptr(c, ctypes.c_uint16))
    if st != OK:
        raise ValueError(f"oracle_gemm_bf16 status {st}")
    return c


def gemm_bf16_scaled(w, ws, x, xs, alpha: float) -> np.ndarray:
    """C = BF16(alpha * sum), alpha an FP32 value (rounded once from FP64)."""
    w, ws, x, xs = map(_u8, (w, ws, x, xs))
    n, k, m = _check_shapes(w, ws, x, xs)
    c = np.empty((m, n), dtype=np.uint16)
    st = _load().oracle_gemm_bf16_scaled(n, k, m, _ptr(w, ctypes.c_uint8),
                                         _ptr(ws, ctypes.c_uint8), _ptr(x, ctypes.c_uint8),
                                         _ptr(xs, ctypes.c_uint8), float(np.float32(alpha)),
                                         _ptr(c, ctypes.c_uint16))
    if st != OK:
        raise ValueError(f"oracle_gemm_bf16_scaled status {st}")
    return c


def gemm_sample(w, ws, x, xs, rows, cols) -> np.ndarray:
    """BF16 bits of C at the given (row, column) positions only."""
    w, ws, x, xs = map(_u8, (w, ws, x, xs))
    n, k, m = _check_shapes(w, ws, x, xs)
    rows = np.ascontiguousarray(rows, dtype=np.int32)
    cols = np.ascontiguousarray(cols, dtype=np.int32)
    out = np.empty(rows.shape[0], dtype=np.uint16)
    st = _load().oracle_gemm_sample(n, k, m, _ptr(w, ctypes.c_uint8), _ptr(ws, ctypes.c_uint8),
                                    _ptr(x, ctypes.c_uint8), _ptr(xs, ctypes.c_uint8),
                                    rows.shape[0], _ptr(rows, ctypes.c_int32),
                                    _ptr(cols, ctypes.c_int32), _ptr(out, ctypes.c_uint16))
    if st != OK:
        raise ValueError(f"oracle_gemm_sample status {st}")
    return out


class Mailbox:
    """The oracle's model of one mailbox and its four state words.

    ``words`` is ``[3][capacity][N/2]`` uint32 (column 2w in the low half of
    word w); ``state`` is ``[next generation, active generation, arrivals,
    error flags]``."""

    def __init__(self, capacity: int, n: int):
        self.capacity = capacity
        self.n = n
        self.words = np.empty((GENERATIONS, capacity, n // 2), dtype=np.uint32)
        self.state = np.empty(4, dtype=np.int32)
        st = _load().oracle_mailbox_init(_ptr(self.words, ctypes.c_uint32),
                                         _ptr(self.state, ctypes.c_int32), capacity, n)
        if st != OK:
            raise ValueError(f"oracle_mailbox_init status {st}")

    def publish(self, c: np.ndarray) -> int:
        c = np.ascontiguousarray(c, dtype=np.uint16)
        m = c.shape[0]
        return _load().oracle_publish(_ptr(self.words, ctypes.c_uint32),
                                      _ptr(self.state, ctypes.c_int32),
                                      self.capacity, self.n, m, _ptr(c, ctypes.c_uint16))

    def consume(self, m: int):
        """(status, out [m][N] uint16)."""
        out = np.empty((m, self.n), dtype=np.uint16)
        st = _load().oracle_consume(_ptr(self.words, ctypes.c_uint32),
                                    _ptr(self.state, ctypes.c_int32),
                                    self.capacity, self.n, m, _ptr(out, ctypes.c_uint16))
        return st, out

    def chain(self, w, ws, x, xs, want_c: bool = True):
        """One call of the whole path: (status, C, out)."""
        w, ws, x, xs = map(_u8, (w, ws, x, xs))
        n, k, m = _check_shapes(w, ws, x, xs)
        if n != self.n:
            raise ValueError("W has another column count than the mailbox")
        c = np.empty((m, n), dtype=np.uint16) if want_c else None
        out = np.empty((m, n), dtype=np.uint16)
        st = _load().oracle_chain(n, k, m, _ptr(w, ctypes.c_uint8), _ptr(ws, ctypes.c_uint8),
                                  _ptr(x, ctypes.c_uint8), _ptr(xs, ctypes.c_uint8),
                                  _ptr(self.words, ctypes.c_uint32),
                                  _ptr(self.state, ctypes.c_int32), self.capacity,
                                  _ptr(c, ctypes.c_uint16) if c is not None else None,
                                  _ptr(out, ctypes.c_uint16))
        return st, c, out


class TaggedMailbox:
    """The oracle's tagged-pair mailbox: ``pairs [capacity][N/2][2]`` uint32
    (value word, tag); tag 0 is the armed state."""

    def __init__(self, capacity: int, n: int):
        self.capacity, self.n = capacity, n
        self.pairs = np.empty((capacity, n // 2, 2), dtype=np.uint32)
        st = _load().oracle_tagged_init(_ptr(self.pairs, ctypes.c_uint32), capacity, n)
        if st != OK:
            raise ValueError(f"oracle_tagged_init status {st}")

    def publish(self, c: np.ndarray, tag: int) -> int:
        c = np.ascontiguousarray(c, dtype=np.uint16)
        return _load().oracle_tagged_publish(_ptr(self.pairs, ctypes.c_uint32), self.capacity,
                                             self.n, c.shape[0], _ptr(c, ctypes.c_uint16), tag)

    def consume(self, m: int, tag: int):
        out = np.empty((m, self.n), dtype=np.uint16)
        st = _load().oracle_tagged_consume(_ptr(self.pairs, ctypes.c_uint32), self.capacity,
                                           self.n, m, tag, _ptr(out, ctypes.c_uint16))
        return st, out


class Gather:
    """The oracle's one-rank Lamport all-gather: mailbox ``[3][capacity]``
    uint32 words and state ``[generation, arrivals]``."""

    def __init__(self, capacity_bytes: int):
        if capacity_bytes <= 0 or capacity_bytes % 16:
            raise ValueError("the capacity must be a positive multiple of 16 bytes")
        self.capacity_words = capacity_bytes // 4
        self.words = np.empty((GENERATIONS, self.capacity_words), dtype=np.uint32)
        self.state = np.empty(2, dtype=np.int32)
        st = _load().oracle_gather_init(_ptr(self.words, ctypes.c_uint32),
                                        _ptr(self.state, ctypes.c_int32), self.capacity_words)
        if st != OK:
            raise ValueError(f"oracle_gather_init status {st}")

    def __call__(self, inp: np.ndarray):
        """(status, output words) for input words (uint32)."""
        inp = np.ascontiguousarray(inp, dtype=np.uint32).reshape(-1)
        out = np.empty_like(inp)
        st = _load().oracle_all_gather(_ptr(self.words, ctypes.c_uint32),
                                       _ptr(self.state, ctypes.c_int32), self.capacity_words,
                                       _ptr(inp, ctypes.c_uint32), inp.size,
                                       _ptr(out, ctypes.c_uint32))
        return st, out


def bf16_bits_to_float(bits: np.ndarray) -> np.ndarray:
    """Widen BF16 bit patterns to float64 (exact)."""
    b = np.ascontiguousarray(bits, dtype=np.uint16).astype(np.uint32) << 16
    return b.view(np.float32).astype(np.float64)
