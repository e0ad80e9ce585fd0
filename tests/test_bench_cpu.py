"""Host logic of the benchmark that needs no GPU: the stored-counter lookup
(an ncu summary's `traffic:` line applies only to the kernel sources it was
taken on, where comments and layout do not count) and the workload config."""
import os
import shutil

import pytest

import bench


def test_comment_stripping_keeps_code_and_literals():
    src = 'a = "x // y /* z */"; // tail\nb = 1; /* block\n comment */ c = \'/\';\n'
    assert bench.strip_c_comments(src) == 'a = "x // y /* z */"; b = 1; c = \'/\';'
    assert bench.strip_c_comments("x  =\n\n  y;") == "x = y;"
    assert bench.strip_c_comments('s = "a\\"//b";') == 's = "a\\"//b";'


def _hash_of(tmp_path, edit):
    d = tmp_path / "csrc"
    shutil.copytree(bench.CSRC, d)
    p = d / "rope_kernels.cuh"
    p.write_text(edit(p.read_text()))
    old = bench.CSRC
    bench.CSRC = str(d)
    try:
        return bench.kernel_source_hash()
    finally:
        bench.CSRC = old


def test_source_hash_ignores_comments_but_not_code(tmp_path):
    base = bench.kernel_source_hash()
    assert _hash_of(tmp_path / "a", lambda t: "// a new comment\n" + t.replace("\n", "\n\n", 3)) == base
    assert _hash_of(tmp_path / "b", lambda t: t.replace("kSign = sizeof(T) == 4", "kSign = sizeof(T) >= 4", 1)) != base


def test_traffic_lines_match_kernel_workload_and_sources(tmp_path, monkeypatch):
    sha = bench.kernel_source_hash()
    d = tmp_path / "profiles"
    d.mkdir()
    (d / "k.md").write_text(
        "text\n"
        f"traffic: kernel=K<float,8,false,4,0,false> workload=w1 source_sha={sha} dram_bytes_per_launch=123\n"
        f"traffic: kernel=K<float,8,false,4,1,false> workload=w1 source_sha={sha} dram_bytes_per_launch=456\n"
        "traffic: kernel=K<float,8,false,4,0,false> workload=w2 source_sha=0000000000000000 dram_bytes_per_launch=789\n")
    monkeypatch.setattr(bench, "PROFILES", str(d))
    assert bench.stored_traffic("K<float,8,false,4,0,false>", "w1") == 123
    assert bench.stored_traffic("K<float,8,false,4,1,false>", "w1") == 456
    assert bench.stored_traffic("K<float,8,false,4,0,false>", "w2") is None   # other sources
    assert bench.stored_traffic("K<float,8,false,2,0,false>", "w1") is None   # other kernel


def test_committed_profiles_hold_the_headline_kernels_traffic():
    """The committed summaries carry DRAM traffic for the headline workload's
    forward and backward kernels at the current sources (so a bench line
    reports `roofline.traffic`)."""
    from place_partial_rope_gb300 import synth
    w = synth.WORKLOADS["large_unaligned"]

    class P:  # the plan the headline runs (checked against the library in test_boundary)
        path, vec_bytes, heads_per_thread, r_per_head = 1, 8, 4, 0

    for d in (0, 1):
        t = bench.stored_traffic(bench.kernel_name(P, w.dtype, d), w.name)
        assert t is not None and t > w.algorithmic_bytes()


@pytest.mark.parametrize("name", ["gqa", "large_unaligned", "mla_decode_q"])
def test_workload_config_names_the_l2_regime(name):
    from place_partial_rope_gb300 import synth
    w = synth.WORKLOADS[name]
    c = bench.workload_config(w, 132 * 2**20)
    assert c["algorithmic_bytes_per_launch"] == w.algorithmic_bytes()
    big = w.algorithmic_bytes() > 1.5 * 132 * 2**20
    assert c["l2"].startswith("inputs larger than L2") == big
    assert c["l2"].startswith("NOT larger than L2") == (not big)


def test_dram_floor_of_the_named_workloads():
    """Aligned 128-byte slices need exactly their own bytes; the large fp32
    shape's 256-byte slice at byte 136 of 512-byte rows touches five 64-byte
    atoms (320 B) on the read and nine 32-byte sectors (288 B) on the write."""
    from place_partial_rope_gb300 import synth
    for name in ("tiny", "small_model", "gqa", "mla_decode_q"):
        w = synth.WORKLOADS[name]
        assert bench.dram_floor_bytes(w) == w.algorithmic_bytes(), name
    w = synth.WORKLOADS["large_unaligned"]
    rows = 4 * 8192 * 32
    assert bench.dram_floor_bytes(w) == rows * (320 + 288) + 2 * 4 * 8192 * 64 * 4


def test_dram_floor_with_rows_not_a_multiple_of_the_atom():
    """132-byte rows (fp16, D = 66) with the slice [1, 65): the row offsets
    cycle through every 4-byte phase of the 64-byte atom."""
    from place_partial_rope_gb300 import synth
    w = synth.Workload("t", "fp16", (1, 3, 5, 66), 1, 65, (1, 3, 1, 64), "arange", 0, 0, ("fwd",), "")
    pitch, off, length = 132, 2, 128

    def touched(lo, hi, g):
        return len({b // g for b in range(lo, hi)}) * g

    want = sum(touched(r * pitch + off, r * pitch + off + length, 64) +
               touched(r * pitch + off, r * pitch + off + length, 32) for r in range(15))
    assert bench.dram_floor_bytes(w) == want + 2 * 3 * 64 * 2


def test_reference_arm_under_torchrun_prints_one_line_from_rank_0():
    """`bench.py --impl reference` launched as two ranks (CPU only): rank 0
    times the oracle and prints the one JSON line, the other rank exits 0
    without work."""
    import json
    import socket
    import subprocess
    import sys

    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        port = s.getsockname()[1]
    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    cmd = [sys.executable, "-m", "torch.distributed.run", "--nnodes=1", "--nproc-per-node", "2",
           "--master-addr", "127.0.0.1", "--master-port", str(port), "bench.py", "--impl",
           "reference", "--gpus", "2", "--workload", "tiny", "--steps", "2", "--warmup", "1"]
    r = subprocess.run(cmd, cwd=root, capture_output=True, text=True, timeout=240)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.startswith("{")]
    assert len(lines) == 1, r.stdout
    out = json.loads(lines[0])
    assert out["impl"] == "reference" and out["n_gpus"] == 2 and out["value"] > 0
    assert out["cpu_baseline"]["kind"] == "oracle" and out["e2e"]["h2d_bytes_per_step"] == 0
