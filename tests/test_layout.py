"""The decode kernel's shared-memory carve-up, checked on the host.

A region that takes 16-byte (cp.async, float4) accesses at an offset that is
not a multiple of 16 faults the GPU with a misaligned address, so the
carve-up of every instantiated configuration is checked here, without a GPU:
tests/native/layout_check.cu includes the kernel header and runs the
layout function for every stage count and a range of batch sizes.
"""
import os
import shutil
import subprocess

import pytest

HERE = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(HERE)


def test_decode_layout_alignment(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc not found")
    exe = str(tmp_path / "layout_check")
    subprocess.run([nvcc, "-std=c++17", "-I", os.path.join(ROOT, "include"),
                    "-I", os.path.join(ROOT, "paged_kv_cache_273_gb300", "csrc"),
                    "-o", exe, os.path.join(HERE, "native", "layout_check.cu")],
                   check=True, capture_output=True, timeout=600)
    r = subprocess.run([exe], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0, r.stdout + r.stderr
    assert "layout check: 0 bad" in r.stdout
