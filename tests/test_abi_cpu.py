"""The C-ABI library on the CPU: it builds, loads, exports every function the
header declares, and rejects bad arguments on the host before any launch."""
import ctypes
import re
from pathlib import Path

import pytest

from mxfp8_gemm_mailbox_gb300 import _lib
from mxfp8_gemm_mailbox_gb300 import build as build_mod

HEADER = Path(__file__).resolve().parents[1] / "include" / "mxfp8_mailbox.h"


@pytest.fixture(scope="module")
def lib():
    build_mod.build()
    return _lib.load()


def declared_functions():
    text = HEADER.read_text()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    names = re.findall(r"^[A-Za-z_][\w\s\*]*?\b((?:mxfp8|mailbox|lamport|tagged)_\w+)\s*\(", text, flags=re.M)
    return sorted(set(names))


def test_header_declares_the_boundary():
    names = declared_functions()
    for required in ("mxfp8_publish_gemm_create", "mxfp8_publish_gemm_precompile",
                     "mxfp8_publish_gemm_run", "mailbox_consume", "mxfp8_mailbox_init"):
        assert required in names


def test_library_exports_every_declared_symbol(lib):
    names = declared_functions()
    missing = [n for n in names if not hasattr(lib, n)]
    assert not missing, missing
    # and the binding declares a signature for each
    assert sorted(_lib.SIGNATURES) == names


def test_mailbox_bytes(lib):
    assert lib.mxfp8_mailbox_bytes(8, 7168) == 3 * 8 * 7168 * 2
    assert lib.mxfp8_mailbox_bytes(1, 8) == 48
    for cap, n in [(0, 128), (9, 128), (8, 0), (8, 12), (-1, 128)]:
        assert lib.mxfp8_mailbox_bytes(cap, n) == 0


def test_workspace_bytes(lib):
    in_place, tiled = _lib.W_IN_PLACE, _lib.W_TILED
    d = _lib.GemmDesc(7168, 16384, 8, 4, 0, 0, 0, in_place)
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 56 * 128 * 512
    d = _lib.GemmDesc(256, 96, 8, 1, 0, 0, 0, in_place)  # ragged K: one partial tile
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 2 * 1 * 512
    d = _lib.GemmDesc(7168, 16384, 8, 4, 0, 0, 0, tiled)  # + the tiled copy of W
    scales = 56 * 128 * 512
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == scales + 7168 * 16384
    d = _lib.GemmDesc(256, 96, 8, 1, 0, 0, 0, 0)  # 0 chooses the tiled copy
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 1024 + 2 * 16384
    d = _lib.GemmDesc(200, 256, 8, 1, 0, 0)
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 0


def test_workspace_bytes_folded(lib):
    # fold f: N / (128 / f) tiles x ceil(K / (128 f)) stages, 512 scale bytes and
    # 16 KB of W each; K pads to a multiple of 128 f.
    in_place, tiled = _lib.W_IN_PLACE, _lib.W_TILED
    d = _lib.GemmDesc(4096, 4096, 8, 1, 0, 0, 0, in_place, 0, 0, 0, 4)
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 128 * 8 * 512
    d = _lib.GemmDesc(4096, 4096, 8, 1, 0, 0, 0, tiled, 0, 0, 0, 4)
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 128 * 8 * 512 + 4096 * 4096
    d = _lib.GemmDesc(256, 96, 8, 1, 0, 0, 0, tiled, 0, 0, 0, 2)  # K pads to 256
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 4 * 512 + 4 * 16384
    d = _lib.GemmDesc(256, 640, 8, 1, 0, 0, 0, in_place, 0, 0, 0, 4)  # K pads to 1024
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 8 * 2 * 512
    d = _lib.GemmDesc(256, 1152, 8, 1, 0, 0, 0, tiled, 0, 0, 0, 8)  # 16 tiles, K pads to 2048
    assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 16 * 2 * 512 + 16 * 2 * 16384
    for fold in (3, 16, -1):
        d = _lib.GemmDesc(256, 256, 8, 1, 0, 0, 0, 0, 0, 0, 0, fold)
        assert lib.mxfp8_publish_gemm_workspace_bytes(ctypes.byref(d)) == 0


def _create(lib, desc, w=0x1000, ws=0x2000, mb=0x3000, st=0x4000, work=0x5000, nbytes=1 << 30):
    out = ctypes.c_void_p()
    status = lib.mxfp8_publish_gemm_create(ctypes.byref(desc), ctypes.c_void_p(w),
                                           ctypes.c_void_p(ws), ctypes.c_void_p(mb),
                                           ctypes.c_void_p(st), ctypes.c_void_p(work), nbytes,
                                           None, ctypes.byref(out))
    return status, out, lib.mxfp8_last_error().decode()


@pytest.mark.parametrize("desc,expect,needle", [
    ((100, 256, 8, 1, 0, 0), _lib.ERR_INVALID, "multiple of 128"),
    ((256, 250, 8, 1, 0, 0), _lib.ERR_INVALID, "multiple of 32"),
    ((256, 256, 0, 1, 0, 0), _lib.ERR_INVALID, "capacity_m"),
    ((256, 256, 9, 1, 0, 0), _lib.ERR_INVALID, "capacity_m"),
    ((256, 256, 8, 3, 0, 0), _lib.ERR_UNSUPPORTED, "split_k"),
    ((256, 256, 8, 16, 0, 0), _lib.ERR_UNSUPPORTED, "split_k"),
    ((256, 256, 8, 1, 64, 0), _lib.ERR_UNSUPPORTED, "cta_k"),
    ((256, 256, 8, 1, 0, 1), _lib.ERR_UNSUPPORTED, "stages"),
    ((256, 65536, 8, 1, 0, 0), _lib.ERR_UNSUPPORTED, "32768"),
    ((256, 256, 8, 1, 0, 0, 2), _lib.ERR_UNSUPPORTED, "acc_blocks"),
    ((256, 256, 8, 1, 0, 0, 0, 3), _lib.ERR_UNSUPPORTED, "w_layout"),
    ((256, 256, 8, 1, 0, 0, 0, 0, 65), _lib.ERR_UNSUPPORTED, "l2_prefetch"),
    ((256, 256, 8, 1, 0, 0, 0, 0, -2), _lib.ERR_UNSUPPORTED, "l2_prefetch"),
    ((256, 256, 8, 1, 0, 0, 0, 0, 0, 3), _lib.ERR_UNSUPPORTED, "pipes"),
    ((256, 256, 8, 1, 0, 0, 0, 0, 0, 0, 3), _lib.ERR_UNSUPPORTED, "tmem_load"),
    ((256, 256, 8, 1, 0, 0, 0, 0, 0, 0, 0, 3), _lib.ERR_UNSUPPORTED, "fold"),
    ((256, 256, 8, 1, 0, 0, 0, 0, 0, 0, 0, 0, 65), _lib.ERR_UNSUPPORTED, "l2_prefetch_early"),
    ((256, 256, 8, 1, 0, 0, 0, 0, 0, 0, 0, 0, -2), _lib.ERR_UNSUPPORTED, "l2_prefetch_early"),
    ((256, 256, 8, 1, 0, 0, 0, 0, 0, 0, 0, 16), _lib.ERR_UNSUPPORTED, "fold"),
    ((256, 2048, 8, 2, 0, 0, 0, 0, 0, 0, 0, 8), _lib.ERR_UNSUPPORTED, "fold 8 takes split_k 1"),
    ((256, 2048, 8, 1, 0, 0, 0, 0, 0, 4, 0, 8), _lib.ERR_UNSUPPORTED, "2 pipes"),
    ((256, 2048, 8, 8, 0, 0, 0, 0, 0, 0, 0, 2), _lib.ERR_UNSUPPORTED, "split_k 1, 2 or 4"),
    ((256, 256, 8, 1, 0, 0, 1, 0, 0, 0, 0, 2), _lib.ERR_UNSUPPORTED, "acc_blocks 4"),
    ((256, 256, 8, 1, 0, 0, 0, 0, 0, 0, 2, 4), _lib.ERR_UNSUPPORTED, "32x32b"),
])
def test_create_rejects_bad_descriptors(lib, desc, expect, needle):
    status, out, msg = _create(lib, _lib.GemmDesc(*desc))
    assert status == expect and not out.value
    assert needle in msg


def test_create_rejects_bad_pointers(lib):
    d = _lib.GemmDesc(256, 256, 8, 1, 0, 0)
    assert _create(lib, d, w=0x1001)[0] == _lib.ERR_INVALID          # W misaligned
    assert _create(lib, d, w=0)[0] == _lib.ERR_INVALID                # W NULL
    assert _create(lib, d, mb=0x3008)[0] == _lib.ERR_INVALID          # mailbox misaligned
    assert _create(lib, d, st=0x4004)[0] == _lib.ERR_INVALID          # state misaligned
    assert _create(lib, d, nbytes=10)[0] == _lib.ERR_INVALID          # workspace too small


def test_mailbox_calls_reject_bad_arguments(lib):
    mb, st, out = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    assert lib.mailbox_consume(None, st, 8, 128, 1, out, 0, None) == _lib.ERR_INVALID
    assert lib.mailbox_consume(mb, st, 8, 128, 0, out, 0, None) == _lib.ERR_UNSUPPORTED
    assert lib.mailbox_consume(mb, st, 4, 128, 5, out, 0, None) == _lib.ERR_UNSUPPORTED
    assert lib.mailbox_consume(mb, st, 8, 12, 1, out, 0, None) == _lib.ERR_INVALID
    assert lib.mailbox_consume(mb, st, 8, 128, 1, ctypes.c_void_p(0x3004), 0, None) == _lib.ERR_INVALID
    assert lib.mailbox_publish(mb, st, 8, 128, 9, out, None) == _lib.ERR_UNSUPPORTED
    assert lib.mxfp8_mailbox_init(ctypes.c_void_p(0x1004), st, 8, 128, None) == _lib.ERR_INVALID
    assert lib.mxfp8_mailbox_init(mb, st, 0, 128, None) == _lib.ERR_INVALID


def test_run_rejects_null_handle(lib):
    assert lib.mxfp8_publish_gemm_run(None, None, None, 1, None, None) == _lib.ERR_INVALID
    assert lib.mxfp8_publish_gemm_precompile(None, 1) == _lib.ERR_INVALID
    assert lib.mxfp8_publish_gemm_config(None, None, None, None, None) == _lib.ERR_INVALID
    lib.mxfp8_publish_gemm_destroy(None)  # a no-op


def test_binding_fails_loudly_without_the_library(monkeypatch, tmp_path):
    monkeypatch.setattr(_lib, "LIBRARY", tmp_path / "missing.so")
    monkeypatch.setattr(_lib, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        _lib.load()


def test_gather_calls_reject_bad_arguments(lib):
    mb, st, buf = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000), ctypes.c_void_p(0x3000)
    assert lib.lamport_gather_mailbox_bytes(4096) == 3 * 4096
    for cap in (0, 20, (64 << 20) + 16):
        assert lib.lamport_gather_mailbox_bytes(cap) == 0
        assert lib.lamport_gather_init(mb, st, cap, None) == _lib.ERR_INVALID
    assert lib.lamport_gather_init(ctypes.c_void_p(0x1008), st, 4096, None) == _lib.ERR_INVALID
    for nbytes in (0, 24, 4112):
        assert lib.lamport_all_gather(mb, st, 4096, buf, nbytes, buf, 0, None) == _lib.ERR_INVALID
    assert lib.lamport_all_gather(mb, st, 4096, ctypes.c_void_p(0x3004), 16, buf, 0,
                                  None) == _lib.ERR_INVALID
    assert "16-byte multiples" in (lib.lamport_all_gather(mb, st, 64, buf, 80, buf, 0, None)
                                   and lib.mxfp8_last_error().decode())


def test_tagged_calls_reject_bad_arguments(lib):
    pairs, buf = ctypes.c_void_p(0x1000), ctypes.c_void_p(0x2000)
    assert lib.tagged_mailbox_bytes(8, 7168) == 8 * 7168 * 4
    assert lib.tagged_mailbox_bytes(0, 128) == 0 and lib.tagged_mailbox_bytes(8, 12) == 0
    assert lib.tagged_publish(pairs, 8, 128, 1, buf, 0, None) == _lib.ERR_INVALID  # tag 0
    assert lib.tagged_publish(pairs, 8, 128, 9, buf, 1, None) == _lib.ERR_UNSUPPORTED
    assert lib.tagged_consume(pairs, 8, 128, 1, 0, buf, 0, None, None) == _lib.ERR_INVALID
    assert lib.tagged_consume(pairs, 8, 128, 1, 1, ctypes.c_void_p(0x2008), 0, None,
                              None) == _lib.ERR_INVALID
    assert lib.tagged_mailbox_init(ctypes.c_void_p(0x1004), 8, 128, None) == _lib.ERR_INVALID


C_CLIENT = r"""
#include <stdio.h>
#include <string.h>
#include "mxfp8_mailbox.h"

int main(void) {
  mxfp8_gemm_desc d;
  memset(&d, 0, sizeof d);
  d.n = 7168; d.k = 16384; d.capacity_m = 8; d.split_k = 4;
  /* host-only calls: sizes and argument checks, no device needed */
  if (mxfp8_mailbox_bytes(8, 7168) != 3u * 8u * 7168u * 2u) return 1;
  if (mxfp8_publish_gemm_workspace_bytes(&d) == 0) return 2;
  if (tagged_mailbox_bytes(8, 7168) == 0) return 3;
  if (lamport_gather_mailbox_bytes(1u << 20) != 3u * (1u << 20)) return 4;
  d.pipes = 3;
  mxfp8_publish_gemm* g = NULL;
  if (mxfp8_publish_gemm_create(&d, NULL, NULL, NULL, NULL, NULL, 0, NULL, &g) == MXFP8_OK) return 5;
  if (g != NULL || strlen(mxfp8_last_error()) == 0) return 6;
  printf("%s\n", mxfp8_last_error());
  return 0;
}
"""


def test_header_and_library_serve_a_c99_program(lib, tmp_path):
    """The boundary is plain C: a C99 program that includes only the header
    builds with warnings as errors, links against the library, and makes
    the host-only calls (sizes and an argument check)."""
    import shutil
    import subprocess

    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc not available")
    src = tmp_path / "client.c"
    src.write_text(C_CLIENT)
    exe = tmp_path / "client"
    libdir = Path(_lib.LIBRARY).parent
    cmd = [gcc, "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic", f"-I{HEADER.parent}",
           str(src), "-o", str(exe), f"-L{libdir}", f"-l:{Path(_lib.LIBRARY).name}",
           f"-Wl,-rpath,{libdir}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stderr
    run = subprocess.run([str(exe)], capture_output=True, text=True)
    assert run.returncode == 0, (run.returncode, run.stdout, run.stderr)
    assert "pipes" in run.stdout
