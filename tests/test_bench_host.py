"""Host-side logic of bench.py without a GPU: the reference arm (the CPU
oracle) prints a well-formed line, the byte model matches the documented
formulas, and the max-over-ranks reduction works across two gloo ranks."""
from __future__ import annotations

import json
import os
import socket
import subprocess
import sys

import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
from combine_expert_count_gb300 import workloads as W  # noqa: E402


def test_algorithmic_bytes_match_formulas():
    w = W.CONFIGS["dsv3_decode"]
    b = bench.algorithmic_bytes(w, w.A)
    assert round(b["s8d_dispatch"] / 1e6, 1) == 392.8
    assert round(b["s8d_combine"] / 1e6, 1) == 734.1
    per = b["separate"]
    assert per["combine_send"] == 4 * w.A * w.H
    assert per["dispatch_send"] > 2 * w.N * w.T * w.H
    # the fused calls skip exactly the two re-reads
    sep, fus = sum(b["separate"].values()), sum(b["fused"].values())
    row8 = w.H + 4 * (w.H // 128)
    assert abs((sep - fus) - (w.A * (row8 + 4) + w.A * 2 * w.H)) <= 24 * w.A


def test_reference_arm_prints_one_json_line():
    env = dict(os.environ, WORLD_SIZE="1", RANK="0")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "2", "--warmup", "1"],
                         capture_output=True, text=True, env=env, timeout=300, check=True).stdout
    lines = [ln for ln in out.splitlines() if ln.startswith("{")]
    assert len(lines) == 1
    d = json.loads(lines[0])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == bench.UNIT
    assert d["higher_is_better"] is False and d["value"] > 0
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["cores"] == 1
    # every timed step is one whole layer (no extrapolation from a sample)
    assert cb["layers"] == 2 and d["steps"] == 2
    assert abs(cb["dispatch_us"] + cb["combine_us"] - d["value"]) <= 0.01 * d["value"] + 0.2
    assert cb["all_cores"]["cores"] >= 1 and cb["all_cores"]["value"] > 0
    assert d["e2e"]["h2d_bytes_per_step"] == 0


def test_reference_arm_other_ranks_do_nothing():
    env = dict(os.environ, WORLD_SIZE="2", RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--config", "tiny", "--steps", "1", "--warmup", "1"],
                         capture_output=True, text=True, env=env, timeout=120, check=True).stdout
    assert out.strip() == ""


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, q):
    import torch.distributed as dist
    dist.init_process_group("gloo", init_method=f"tcp://127.0.0.1:{port}", rank=rank,
                            world_size=world)
    try:
        bench.barrier(world)
        v = bench.max_over_ranks(10.0 + rank, world)
        q.put((rank, v))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_two_ranks():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=10) for _ in range(2))
    assert got == [(0, 11.0), (1, 11.0)]


def test_per_kernel_table_ratios():
    """Each kernel row carries its algorithmic GB/s; rows with a committed
    DRAM record for the current source also carry DRAM GB/s and the
    DRAM / algorithmic ratio; the routing kernels are marked latency-bound."""
    w = W.CONFIGS["dsv3_decode"]
    nb = bench.algorithmic_bytes(w, w.A)
    favg = {"route": 0.010, "dispatch_fused": 0.050, "combine_fused": 0.085}
    savg = {"route": 0.010, "dispatch_send": 0.030, "dispatch_recv": 0.042,
            "combine_send": 0.083, "combine_recv": 0.039}
    rows = bench.per_kernel_table(nb, favg, savg, [[0.01], [0.006]], w.A, w, "dsv3_decode")
    by = {r["kernel"]: r for r in rows}
    assert {"route_count", "exchange", "route", "dispatch_send", "dispatch_recv",
            "combine_send", "combine_recv", "dispatch_fused", "combine_fused"} == set(by)
    for k in ("route_count", "exchange", "route"):
        assert by[k]["bound"] == "latency" and "algorithmic_gbs" not in by[k]
    c = by["combine_fused"]
    assert c["algorithmic_gbs"] == round(nb["fused"]["combine_fused"] / 85e-6 / 1e9, 1)
    dram = bench.dram_traffic("combine_fused", "dsv3_decode")
    if dram is None:
        assert "dram_mb" not in c
    else:
        assert c["dram_over_algorithmic"] == round(dram / nb["fused"]["combine_fused"], 3)
        assert 0.0 < c["dram_over_algorithmic"] <= 1.5


def test_traffic_record_follows_code_not_comments():
    src = bench.KERNEL_SOURCES["combine_fused"]
    csrc = os.path.join(ROOT, "combine_expert_count_gb300", "csrc")
    text = {f: open(os.path.join(csrc, f), encoding="utf-8").read() for f in src}
    base = bench.source_hash("combine_fused", read=lambda f: text[f])
    assert base == bench.source_hash("combine_fused")
    commented = dict(text)
    commented[src[0]] = "// a new comment\n/* and a block\n comment */" + \
        text[src[0]].replace("\n", "  \n", 3)
    assert bench.source_hash("combine_fused", read=lambda f: commented[f]) == base
    changed = dict(text)
    changed[src[0]] = text[src[0]] + "\nstatic int extra_code = 1;\n"
    assert bench.source_hash("combine_fused", read=lambda f: changed[f]) != base
    assert bench.code_only('x = "// kept"; // dropped\ny') == 'x = "// kept"; y'
