"""The C ABI from plain C: include/rope_partial.h compiles as C99 on its
own, a C program that calls the library links against it (CPU), and on a
GPU that program's results match the oracle bit for bit; a second C program
splits a token grid across ranks (CPU: that call makes no CUDA call)."""
import os
import shutil
import subprocess

import numpy as np
import pytest

import oracle
from place_partial_rope_gb300 import binding

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
DEMO = os.path.join(ROOT, "tests", "c", "abi_demo.c")
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")


def _gcc():
    gcc = shutil.which("gcc")
    if gcc is None:
        pytest.skip("gcc is not installed")
    return gcc


def test_header_is_valid_c99(tmp_path):
    src = tmp_path / "h.c"
    src.write_text('#include "rope_partial.h"\nint main(void) { return ROPE_OK; }\n')
    r = subprocess.run([_gcc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-pedantic",
                        "-I", INCLUDE, "-c", str(src), "-o", str(tmp_path / "h.o")],
                       capture_output=True, text=True)
    assert r.returncode == 0, r.stderr


def build_demo(tmp_path) -> str:
    if not os.path.isdir(os.path.join(CUDA, "include")):
        pytest.skip("the CUDA toolkit headers are not installed")
    lib_dir = os.path.dirname(binding.library_path())
    if not os.path.exists(binding.library_path()):
        pytest.skip("librope_partial.so is not built")
    exe = str(tmp_path / "abi_demo")
    cmd = [_gcc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-O2", "-I", INCLUDE,
           "-I", os.path.join(CUDA, "include"), DEMO, "-o", exe,
           "-L", lib_dir, "-lrope_partial", f"-Wl,-rpath,{lib_dir}",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart", f"-Wl,-rpath,{os.path.join(CUDA, 'lib64')}",
           "-lm"]
    r = subprocess.run(cmd, capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    return exe


def test_c_program_links_against_the_library(tmp_path):
    assert os.path.exists(build_demo(tmp_path))


@pytest.mark.gpu
def test_c_program_results_match_the_oracle(tmp_path):
    exe = build_demo(tmp_path)
    out = tmp_path / "out.bin"
    r = subprocess.run([exe, str(out)], capture_output=True, text=True, timeout=120)
    assert r.returncode == 0 and "abi_demo ok" in r.stdout, r.stderr
    raw = out.read_bytes()
    B, S, N, D, st, en = np.frombuffer(raw[:48], dtype=np.int64)
    L, nx = en - st, B * S * N * D
    f = np.frombuffer(raw[48:], dtype=np.float32)
    x, f = f[:nx].reshape(B, S, N, D), f[nx:]
    r1, f = f[:S * L].reshape(1, S, 1, L), f[S * L:]
    r2, f = f[:S * L].reshape(1, S, 1, L), f[S * L:]
    g, f = f[:nx].reshape(B, S, N, D), f[nx:]
    y, dx = f[:nx].reshape(B, S, N, D), f[nx:2 * nx].reshape(B, S, N, D)
    assert np.array_equal(y.view(np.uint32), oracle.fwd(x, r1, r2, "fp32", st, en).view(np.uint32))
    assert np.array_equal(dx.view(np.uint32), oracle.bwd(g, r1, r2, "fp32", st, en).view(np.uint32))


@pytest.mark.parametrize("B,S,world", [(3, 5, 2), (2, 7, 3), (4, 8192, 8), (7, 1, 4)])
def test_c_program_splits_tokens(tmp_path, B, S, world):
    """rope_partial_token_shard from a plain C99 program (no GPU needed): the
    ranks' ranges tile [0, B*S) and each run is a contiguous block."""
    lib_dir = os.path.dirname(binding.library_path())
    exe = str(tmp_path / "shard_demo")
    r = subprocess.run([_gcc(), "-std=c99", "-Wall", "-Wextra", "-Werror", "-I", INCLUDE,
                        os.path.join(ROOT, "tests", "c", "shard_demo.c"), "-o", exe, "-L", lib_dir,
                        "-lrope_partial", "-Wl,-rpath," + lib_dir], capture_output=True, text=True)
    assert r.returncode == 0, r.stderr
    out = subprocess.run([exe, str(B), str(S), str(world)], capture_output=True, text=True,
                         timeout=60)
    assert out.returncode == 0 and out.stdout.rstrip().endswith("ok"), out.stdout + out.stderr
    prev = 0
    for line in out.stdout.splitlines()[:-1]:
        v = [int(t) for t in line.split()]
        rank, t0, t1, n, runs = v[0], v[1], v[2], v[3], v[4:]
        assert t0 == prev and len(runs) == 4 * n
        t = t0
        for k in range(n):
            b0, s0, nb, ns = runs[4 * k:4 * k + 4]
            assert b0 * S + s0 == t and (nb == 1 or (s0 == 0 and ns == S))
            t += nb * ns
        assert t == t1
        prev = t1
    assert prev == B * S
