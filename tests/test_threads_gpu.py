"""Host threads calling the library at once: a fresh process (so the
library's device and occupancy caches start empty) runs 8 threads, each on
its own stream with its own kernel kind and dtype, released together by a
barrier; every result is then checked against the oracle."""
import os
import subprocess
import sys
import textwrap

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

SCRIPT = textwrap.dedent('''
    import sys, threading
    sys.path.insert(0, {root!r})
    sys.path.insert(0, {tests!r})
    import numpy as np
    import torch
    import oracle
    from gpu_util import assert_same, to_dev
    from place_partial_rope_gb300 import binding, synth

    jobs = []
    for i, (dtype, mode, shape, st, en) in enumerate([
            ("bf16", "interleave", (4, 64, 8, 64), 0, 64),
            ("fp16", "interleave", (4, 64, 8, 96), 3, 67),
            ("fp32", "interleave", (4, 64, 8, 128), 34, 98),
            ("fp16", "half", (4, 64, 8, 128), 0, 64),
            ("fp32", "half", (4, 64, 8, 128), 0, 96),
            ("bf16", "half", (4, 64, 8, 64), 1, 61)]):
        x, r1, r2, g = synth.case(shape, st, en, dtype, "BS1D", seed=1200 + i, layout=mode)
        jobs.append(("table", dtype, mode, x, r1, r2, g, st, en))
    barrier = threading.Barrier(8)
    out, errors = {{}}, []

    def table_job(k):
        kind, dtype, mode, x, r1, r2, g, st, en = jobs[k]
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            xd, gd = to_dev(x, dtype), to_dev(g, dtype)
            c, sn = to_dev(r1, dtype), to_dev(r2, dtype)
            s.synchronize()
            barrier.wait()
            for _ in range(3):
                binding.rope_partial_inplace_fwd_mode(xd, c, sn, st, en, mode)
                binding.rope_partial_inplace_bwd_mode(gd, c, sn, st, en, mode)
        s.synchronize()
        out[k] = (synth.from_torch(xd), synth.from_torch(gd))

    def qk_job():
        q, r1, r2, _ = synth.case((8, 4, 16, 96), 0, 64, "bf16", "BS1D", seed=1300)
        k = synth.normal((8, 4, 2, 64), "bf16", 1301)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            qd, kd = to_dev(q, "bf16"), to_dev(k, "bf16")
            c, sn = to_dev(r1, "bf16"), to_dev(r2, "bf16")
            s.synchronize()
            barrier.wait()
            binding.rope_partial_inplace_fwd_qk(qd, kd, c, sn, (0, 64), (0, 64))
        s.synchronize()
        out["qk"] = (q, k, r1, r2, synth.from_torch(qd), synth.from_torch(kd))

    def pos_job():
        x = synth.normal((4, 64, 8, 64), "fp32", 1400)
        pos = np.arange(4 * 64, dtype=np.int32).reshape(4, 64)
        s = torch.cuda.Stream()
        with torch.cuda.stream(s):
            xd, pd = to_dev(x, "fp32"), torch.from_numpy(pos).cuda()
            s.synchronize()
            barrier.wait()
            binding.rope_partial_inplace_fwd_pos(xd, pd, 0, 64, 10000.0, "half")
        s.synchronize()
        out["pos"] = (x, pos, synth.from_torch(xd))

    def guard(fn, *a):
        try:
            fn(*a)
        except BaseException as e:  # noqa: BLE001 - reported by the main thread
            errors.append(repr(e))
            barrier.abort()

    threads = [threading.Thread(target=guard, args=(table_job, k)) for k in range(len(jobs))]
    threads += [threading.Thread(target=guard, args=(qk_job,)), threading.Thread(target=guard, args=(pos_job,))]
    for t in threads:
        t.start()
    for t in threads:
        t.join()
    assert not errors, errors
    for k, (kind, dtype, mode, x, r1, r2, g, st, en) in enumerate(jobs):
        wx, wg = x, g
        for _ in range(3):
            wx = oracle.fwd(wx, r1, r2, dtype, st, en, oracle.GATHER_CHAIN, mode)
            wg = oracle.bwd(wg, r1, r2, dtype, st, en, oracle.GATHER_CHAIN, mode)
        assert_same(out[k][0], wx, dtype, f"job {{k}} fwd")
        assert_same(out[k][1], wg, dtype, f"job {{k}} bwd")
    q, k, r1, r2, gq, gk = out["qk"]
    wq, wk = oracle.rope_qk(oracle.FWD, q, k, r1, r2, "bf16", (0, 64), (0, 64))
    assert_same(gq, wq, "bf16", "qk query")
    assert_same(gk, wk, "bf16", "qk key")
    x, pos, got = out["pos"]
    want = oracle.rope_pos(oracle.FWD, x, pos, 10000.0, "fp32", 0, 64, "half").astype(np.float64)
    mag = np.concatenate([np.abs(x[..., :32]) + np.abs(x[..., 32:])] * 2, axis=-1).astype(np.float64)
    assert np.all(np.abs(got - want) <= 1e-6 * mag + 2 * np.spacing(np.abs(want).astype(np.float32)))
    print("threads ok")
''')


def test_eight_threads_at_once_in_a_fresh_process(tmp_path):
    script = tmp_path / "threads.py"
    script.write_text(SCRIPT.format(root=ROOT, tests=os.path.join(ROOT, "tests")))
    r = subprocess.run([sys.executable, str(script)], capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and "threads ok" in r.stdout, r.stdout[-2000:] + r.stderr[-4000:]
