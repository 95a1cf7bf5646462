"""Calls from several host threads at once, each thread with its own buffers
and stream.  The calls run in a fresh process, so the library's per-device
caches of launch properties (occupancy, cluster limits, shared-memory
attributes) are filled by first calls that race each other; every thread's
result must still equal the CPU oracle's, bit for bit, with a clean status.

Only call forms whose blocks never wait on other blocks beyond a hardware
cluster run here (fused dispatch and combine, the low-latency pair): the
shapes keep N within one cluster."""
from __future__ import annotations

import os
import subprocess
import sys
import textwrap

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))

CHILD = textwrap.dedent(r"""
    import sys, threading
    import numpy as np
    import torch
    sys.path.insert(0, sys.argv[1])
    from combine_expert_count_gb300 import moeroute as m, workloads as W
    from oracle import ref

    tiny = W.CONFIGS["tiny"]
    # shapes with different piece sizes, block sizes and expert counts, so the
    # racing first calls fill several cache entries of each launcher
    shapes = [tiny,
              tiny.replace(N=4, T=8, E=16, R=4, H=384, seed=tiny.seed + 101),
              tiny.replace(N=8, T=5, E=64, R=8, H=1280, seed=tiny.seed + 102),
              tiny.replace(N=16, T=3, E=32, R=3, H=128, seed=tiny.seed + 103)]
    data = [W.generate(w) for w in shapes]
    expect = []
    for w, d in zip(shapes, data):
        o = ref.layer(w.N, w.T, w.E, w.R, w.H, w.default_cap, d["x"], d["topk_idx"],
                      d["topk_w"], mode=0)
        q = ref.layer_ll(w.N, w.T, w.E, w.R, w.H, d["x"], d["topk_idx"], d["topk_w"], mode=0)
        expect.append((o["out"], q["out"]))

    threads_per_shape = 3
    jobs = [(k, j) for k in range(len(shapes)) for j in range(threads_per_shape)]
    dev = torch.device("cuda:0")
    torch.cuda.set_device(dev)
    # inputs and buffers first (torch allocation is not what is under test)
    prep = []
    for k, _ in jobs:
        w, d = shapes[k], data[k]
        x = torch.from_numpy(d["x"].view(np.int16)).to(dev)
        idx = torch.from_numpy(d["topk_idx"]).to(dev)
        wt = torch.from_numpy(d["topk_w"]).to(dev)
        buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, device=dev)
        ll = m.MoeLLBuffers(w.N, w.T, w.E, w.R, w.H, device=dev)
        prep.append((x, idx, wt, buf, ll, torch.cuda.Stream(device=dev)))
    torch.cuda.synchronize()

    start = threading.Barrier(len(jobs))
    errors = []

    def run(i):
        try:
            torch.cuda.set_device(dev)
            x, idx, wt, buf, ll, st = prep[i]
            start.wait()
            with torch.cuda.stream(st):
                for _ in range(2):
                    buf.dispatch(x, idx)
                    buf.expert(0)
                    buf.combine(idx, wt)
                    ll.dispatch(x, idx)
                    ll.expert(0)
                    ll.combine(wt)
            st.synchronize()
        except Exception as e:  # reported by the main thread
            errors.append(f"thread {i}: {e!r}")

    ts = [threading.Thread(target=run, args=(i,)) for i in range(len(jobs))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    torch.cuda.synchronize()
    assert not errors, errors
    for i, (k, _) in enumerate(jobs):
        x, idx, wt, buf, ll, st = prep[i]
        assert int(buf.status.item()) == 0 and int(ll.status.item()) == 0, f"status, job {i}"
        got = buf.out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, expect[k][0]), f"fused output, job {i}"
        got = ll.out.view(torch.int16).cpu().numpy().view(np.uint16)
        assert np.array_equal(got, expect[k][1]), f"low-latency output, job {i}"
    print(f"ok: {len(jobs)} threads")
""")


@pytest.mark.gpu
def test_concurrent_first_calls_from_host_threads():
    r = subprocess.run([sys.executable, "-c", CHILD, ROOT], capture_output=True, text=True,
                       timeout=600, cwd=ROOT)
    assert r.returncode == 0, r.stdout[-2000:] + r.stderr[-4000:]
    assert "ok: 12 threads" in r.stdout
