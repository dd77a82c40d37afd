"""ctypes declarations of the C ABI in ``include/mxfp8_mailbox.h``.

Loading fails loudly when ``libmxfp8_mailbox.so`` has not been built: there is
no other implementation to fall back to.
"""
from __future__ import annotations

import ctypes
from pathlib import Path

LIBRARY = Path(__file__).resolve().parent / "libmxfp8_mailbox.so"

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_TIMEOUT, ERR_STATE = range(6)
STATUS_NAMES = {OK: "OK", ERR_INVALID: "ERR_INVALID", ERR_UNSUPPORTED: "ERR_UNSUPPORTED",
                ERR_CUDA: "ERR_CUDA", ERR_TIMEOUT: "ERR_TIMEOUT", ERR_STATE: "ERR_STATE"}
W_IN_PLACE = 1
W_TILED = 2
TMEM_LOAD_32X32B = 1
TMEM_LOAD_16X256B = 2
FLAG_POLL_TIMEOUT = 0x1
FLAG_GEMM_TIMEOUT = 0x2
FLAG_BAD_STATE = 0x4
GENERATIONS = 3
SENTINEL = 0x80000000
MAX_ROWS = 8
NOALLOC_SCRATCH_BYTES = 4 << 20

# Every symbol the header declares, with (restype, argtypes).
_vp = ctypes.c_void_p
_i32 = ctypes.c_int32
_sz = ctypes.c_size_t
_u64 = ctypes.c_uint64


class GemmDesc(ctypes.Structure):
    _fields_ = [("n", _i32), ("k", _i32), ("capacity_m", _i32), ("split_k", _i32),
                ("cta_k", _i32), ("stages", _i32), ("acc_blocks", _i32), ("w_layout", _i32),
                ("l2_prefetch", _i32), ("pipes", _i32), ("tmem_load", _i32),
                ("fold", _i32), ("l2_prefetch_early", _i32), ("wait_limit_ms", _i32)]


SIGNATURES = {
    "mxfp8_mailbox_bytes": (_sz, [_i32, _i32]),
    "mxfp8_mailbox_init": (ctypes.c_int, [_vp, _vp, _i32, _i32, _vp]),
    "mxfp8_publish_gemm_workspace_bytes": (_sz, [ctypes.POINTER(GemmDesc)]),
    "mxfp8_publish_gemm_create": (ctypes.c_int, [ctypes.POINTER(GemmDesc), _vp, _vp, _vp, _vp, _vp,
                                                 _sz, _vp, ctypes.POINTER(_vp)]),
    "mxfp8_publish_gemm_config": (ctypes.c_int, [_vp, ctypes.POINTER(GemmDesc),
                                                 ctypes.POINTER(_i32), ctypes.POINTER(_i32),
                                                 ctypes.POINTER(_i32)]),
    "mxfp8_publish_gemm_plan": (ctypes.c_int, [ctypes.POINTER(GemmDesc), _i32, _i32, _i32,
                                               ctypes.POINTER(GemmDesc), ctypes.POINTER(_i32),
                                               ctypes.POINTER(_i32), ctypes.POINTER(_i32)]),
    "mxfp8_publish_gemm_precompile": (ctypes.c_int, [_vp, _i32]),
    "mxfp8_publish_gemm_run": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, _vp]),
    "mxfp8_gemm_run_unfused": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, _vp]),
    "mxfp8_publish_gemm_run_scaled": (ctypes.c_int, [_vp, _vp, _vp, _i32, _vp, _vp, _vp]),
    "mailbox_publish": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _vp, _vp]),
    "mailbox_consume": (ctypes.c_int, [_vp, _vp, _i32, _i32, _i32, _vp, _u64, _vp]),
    "mxfp8_mailbox_status": (ctypes.c_int, [_vp, ctypes.POINTER(_i32), _vp]),
    "lamport_gather_mailbox_bytes": (_sz, [_sz]),
    "tagged_mailbox_bytes": (_sz, [_i32, _i32]),
    "tagged_mailbox_init": (ctypes.c_int, [_vp, _i32, _i32, _vp]),
    "tagged_publish": (ctypes.c_int, [_vp, _i32, _i32, _i32, _vp, ctypes.c_uint32, _vp]),
    "tagged_consume": (ctypes.c_int, [_vp, _i32, _i32, _i32, ctypes.c_uint32, _vp, _u64, _vp,
                                      _vp]),
    "lamport_gather_init": (ctypes.c_int, [_vp, _vp, _sz, _vp]),
    "lamport_all_gather": (ctypes.c_int, [_vp, _vp, _sz, _vp, _sz, _vp, _u64, _vp]),
    "mxfp8_publish_gemm_destroy": (None, [_vp]),
    "mxfp8_publish_gemm_run_noalloc": (ctypes.c_int, [ctypes.POINTER(GemmDesc), _vp, _vp, _vp, _vp,
                                                      _i32, _vp, _vp, _vp, _vp]),
    "mxfp8_last_error": (ctypes.c_char_p, []),
}

_lib = None


def load() -> ctypes.CDLL:
    """The loaded library; raises if it has not been built."""
    global _lib
    if _lib is not None:
        return _lib
    if not LIBRARY.exists():
        raise RuntimeError(
            f"{LIBRARY.name} is not built: run `python -m mxfp8_gemm_mailbox_gb300.build` "
            "(nvcc, sm_103a). There is no fallback implementation.")
    lib = ctypes.CDLL(str(LIBRARY))
    for name, (restype, argtypes) in SIGNATURES.items():
        fn = getattr(lib, name)
        fn.restype = restype
        fn.argtypes = argtypes
    _lib = lib
    return lib


class Mxfp8Error(RuntimeError):
    def __init__(self, status: int, where: str, message: str):
        self.status = status
        super().__init__(f"{where}: {STATUS_NAMES.get(status, status)}: {message}")


def check(status: int, where: str) -> None:
    if status != OK:
        raise Mxfp8Error(status, where, load().mxfp8_last_error().decode())
