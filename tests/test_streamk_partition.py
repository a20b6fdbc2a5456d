"""The stream-K work split of the tensor-core prefill GEMM, checked on the CPU
by brute force over every small (tiles, K steps, blocks) combination."""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))


@pytest.mark.skipif(shutil.which("g++") is None, reason="needs a host C++ compiler")
def test_streamk_partition(tmp_path):
    exe = tmp_path / "streamk_check"
    subprocess.run(["g++", "-O2", "-std=c++17", os.path.join(HERE, "streamk_check.cpp"), "-o", str(exe)],
                   check=True)
    r = subprocess.run([str(exe)], capture_output=True, text=True, timeout=300)
    assert r.returncode == 0 and r.stdout.startswith("ok"), r.stdout + r.stderr
