"""Build ``libmxfp8_mailbox.so`` in-tree with nvcc for sm_103a.

The translation units compile in parallel (one ``-gencode``), then link into
one shared library next to this file.  Run ``python -m
mxfp8_gemm_mailbox_gb300.build`` or call :func:`build`.
"""
from __future__ import annotations

import concurrent.futures
import os
import shutil
import subprocess
import sys
from pathlib import Path

PACKAGE = Path(__file__).resolve().parent
ROOT = PACKAGE.parent
CSRC = PACKAGE / "csrc"
INCLUDE = ROOT / "include"
BUILD_DIR = PACKAGE / "_build"
LIBRARY = PACKAGE / "libmxfp8_mailbox.so"
SOURCES = ("publish_gemm.cu", "publish_gemm_fold.cu", "publish_gemm_k256.cu", "mailbox.cu",
           "lamport_gather.cu", "tagged_mailbox.cu", "abi.cu")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def _nvcc() -> str:
    for cand in (os.environ.get("NVCC"), shutil.which("nvcc"), "/usr/local/cuda/bin/nvcc"):
        if cand and Path(cand).exists():
            return cand
    raise RuntimeError("nvcc not found: the CUDA toolkit is required to build the library")


def _stale() -> bool:
    if not LIBRARY.exists():
        return True
    newest = max(p.stat().st_mtime for p in list(CSRC.iterdir()) + list(INCLUDE.iterdir()))
    return LIBRARY.stat().st_mtime < newest


def build(force: bool = False, verbose: bool = False) -> Path:
    """Compile the CUDA library if a source is newer than it (or ``force``)."""
    if not force and not _stale():
        return LIBRARY
    nvcc = _nvcc()
    BUILD_DIR.mkdir(exist_ok=True)
    common = [nvcc, *ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC",
              f"-I{INCLUDE}", f"-I{CSRC}"]
    if verbose:
        common.append("-Xptxas=-v")

    def compile_one(name: str) -> Path:
        obj = BUILD_DIR / (name + ".o")
        cmd = [*common, "-c", str(CSRC / name), "-o", str(obj)]
        res = subprocess.run(cmd, capture_output=True, text=True)
        if res.returncode != 0:
            raise RuntimeError(f"nvcc failed on {name}:\n{res.stdout}\n{res.stderr}")
        if verbose and res.stderr:
            sys.stderr.write(res.stderr)
        return obj

    with concurrent.futures.ThreadPoolExecutor(max_workers=len(SOURCES)) as pool:
        objs = list(pool.map(compile_one, SOURCES))
    tmp = LIBRARY.with_suffix(f".{os.getpid()}.tmp")
    cmd = [nvcc, *ARCH, "-shared", "-Xcompiler", "-fPIC", *map(str, objs), "-o", str(tmp)]
    res = subprocess.run(cmd, capture_output=True, text=True)
    if res.returncode != 0:
        raise RuntimeError(f"linking failed:\n{res.stdout}\n{res.stderr}")
    os.replace(tmp, LIBRARY)
    return LIBRARY


if __name__ == "__main__":
    build(force="--force" in sys.argv, verbose="-v" in sys.argv)
    print(LIBRARY)
