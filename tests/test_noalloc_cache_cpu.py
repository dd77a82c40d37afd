"""The allocation-free call's set-up memo on the CPU: its header compiles on
its own with g++ and the check program shows that a repeated call (same
device, weight pointer and descriptor) reuses the plan -- the weight's tensor
map is encoded once -- while any difference builds a new one."""
import shutil
import subprocess
from pathlib import Path

import pytest

ROOT = Path(__file__).resolve().parents[1]


def test_repeated_calls_skip_the_encode(tmp_path):
    gxx = shutil.which("g++")
    if gxx is None:
        pytest.skip("g++ is not installed")
    exe = tmp_path / "noalloc_cache_check"
    subprocess.run([gxx, "-std=c++17", "-O1", "-Wall", "-Werror",
                    f"-I{ROOT / 'include'}", f"-I{ROOT / 'mxfp8_gemm_mailbox_gb300' / 'csrc'}",
                    str(ROOT / "tests" / "native" / "noalloc_cache_check.cpp"), "-o", str(exe)],
                   check=True)
    res = subprocess.run([str(exe)], capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    assert "FAIL" not in res.stdout and res.stdout.count("ok ") == 12, res.stdout
