"""The odd-start kernel's edge store sequences, checked on the host: for
every range of elements a row's edge lane can store and every vector width,
exactly the range's bytes are written, each from its own word
(tests/c/odd_edge_stores.cu, built with nvcc as host code; no GPU)."""
import os
import shutil
import subprocess

import pytest

from place_partial_rope_gb300 import build

HERE = os.path.dirname(os.path.abspath(__file__))


def test_edge_store_sequences(tmp_path):
    nvcc = shutil.which("nvcc") or "/usr/local/cuda/bin/nvcc"
    if not os.path.exists(nvcc):
        pytest.skip("nvcc is not installed")
    exe = str(tmp_path / "odd_edge_stores")
    subprocess.run([nvcc, "-std=c++17", "-O2", "-I", os.path.join(build.ROOT, "include"), "-I",
                    build.CSRC, os.path.join(HERE, "c", "odd_edge_stores.cu"), "-o", exe],
                   check=True, capture_output=True)
    out = subprocess.run([exe], capture_output=True, text=True)
    assert out.returncode == 0 and out.stdout.startswith("ok"), out.stdout + out.stderr
    # ranges per width: 16-bit 16-byte vectors 8, 8-byte 4; fp32 16-byte 4, 8-byte 2
    assert int(out.stdout.split()[1]) == 18, out.stdout
