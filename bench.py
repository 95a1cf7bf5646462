#!/usr/bin/env python3
"""Dispatch + combine benchmark on one GB300.

One step = one MoE layer's hot path over one batch, through libmoeroute's C
ABI: moe_dispatch (route_count + exchange in one launch, then quantise +
pack + receive shuffle in one launch) and moe_combine (combine send +
receive in one launch).  Every output of the six separate calls of the
pages' steps is written each step; a second timing runs those separate
calls one by one.  The grouped-GEMM stand-in runs once before timing (its
output is the same every step) and is not timed.  Inputs are resident in HBM
when timing starts; L2 is flushed (512 MiB write) before every step, outside
the timed window.

Prints one JSON line: value = dispatch + combine microseconds per layer
(lower is better), achieved HBM GB/s over the bytes the timed calls must
move, the roofline of the dominant kernel, an end-to-end figure with host
buffers, the other configurations with their dispatch / combine split, and
the CPU oracle (whole layers of the same steps, one core and all cores) as
a baseline.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config NAME]
  python bench.py --impl reference ...   (the CPU oracle as the reference arm)
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import statistics
import subprocess
import sys
import tempfile
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "dispatch+combine µs/layer and achieved HBM GB/s (% of GB300 peak) at EP16 h7168"
UNIT = "us/layer"
NOMINAL_HBM_GBS = 8000.0
FALLBACK_HBM_GBS = 6800.0
L2_FLUSH_BYTES = 512 << 20
KERNELS = ("route", "dispatch_send", "dispatch_recv", "combine_send", "combine_recv")
FUSED = ("route", "dispatch_fused", "combine_fused")
KERNEL_SYMBOL = {"route": "k_route_cluster (route_count + exchange)",
                 "dispatch_send": "k_quant_pack_staged<kSend>",
                 "dispatch_recv": "k_row_copy<DispatchMap>",
                 "combine_send": "k_row_copy<CombineMap>", "combine_recv": "k_combine_reduce",
                 "dispatch_fused": "k_quant_pack_staged<kSendGrouped> (quantise + pack + receive "
                                   "shuffle)",
                 "combine_fused": "k_combine_fused (combine send + receive)"}


# ----------------------------------------------------------------- bytes


def algorithmic_bytes(w, A: int) -> dict:
    """Bytes per step, A = (token, expert) assignments routed, Row_fp8 =
    H + 4*H/128.  "s8d": every materialised buffer written once and read
    once (the separate calls move exactly this).  "fused": every buffer the
    fused calls read or write, once -- the same outputs without re-reading
    the send buffer and the combine send buffer."""
    N, T, H, R = w.N, w.T, w.H, w.R
    Sb = H // 128
    row8 = H + 4 * Sb
    x = 2 * N * T * H
    ids = 4 * N * T * R
    separate = {
        "route": 2 * ids,                                       # read ids, write slots
        "dispatch_send": x + A * (row8 + 4) + 4 * A,            # read x, slots; write rows+tok
        "dispatch_recv": A * (row8 + 4) + A * (row8 + 8),       # read rows+tok; write rows+src
        "combine_send": 2 * A * 2 * H,                          # read y rows; write csend rows
        "combine_recv": A * 2 * H + x + 12 * A,                 # read rows, idx/w/slot; write out
    }
    fused = {
        "route": 2 * ids,
        "dispatch_fused": x + 2 * A * row8 + 8 * A + 4 * A + 8 * A,  # x, ids+slots; rows, tok, src
        "combine_fused": 2 * A * 2 * H + x + 12 * A,            # y rows; csend rows, out; idx/w/slot
    }
    return {"separate": separate, "fused": fused,
            "s8d_dispatch": x + 3 * A * row8 + 8 * A,
            "s8d_combine": 3 * A * 2 * H + x + 8 * A}


def measured_peak():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


# Source files each kernel is built from: its DRAM-traffic record holds only
# while these are unchanged.
KERNEL_SOURCES = {
    "route": ("route.cu", "rank.cuh", "common.cuh"),
    "dispatch_fused": ("dispatch.cu", "rank.cuh", "shuffle.cuh", "common.cuh"),
    "combine_fused": ("combine.cu", "bf16.cuh", "common.cuh"),
    "dispatch_send": ("dispatch.cu", "rank.cuh", "shuffle.cuh", "common.cuh"),
    "dispatch_recv": ("shuffle.cu", "shuffle.cuh", "common.cuh"),
    "combine_send": ("shuffle.cu", "shuffle.cuh", "common.cuh"),
    "combine_recv": ("combine.cu", "bf16.cuh", "common.cuh"),
    "combine_partial": ("partial.cu", "bf16.cuh", "common.cuh"),
    "dispatch_signalled": ("dispatch.cu", "rank.cuh", "shuffle.cuh", "common.cuh"),
}


def code_only(src: str) -> str:
    """C/C++ source with comments removed and whitespace runs collapsed, so
    that a comment edit leaves the hash alone while any code edit changes it.
    String and character literals are kept whole."""
    out, i, n = [], 0, len(src)
    while i < n:
        c = src[i]
        if c in "\"'":
            j = i + 1
            while j < n and src[j] != c:
                j += 2 if src[j] == "\\" else 1
            out.append(src[i:j + 1])
            i = j + 1
        elif src.startswith("//", i):
            j = src.find("\n", i)
            i = n if j < 0 else j
        elif src.startswith("/*", i):
            j = src.find("*/", i + 2)
            out.append(" ")
            i = n if j < 0 else j + 2
        else:
            out.append(c)
            i += 1
    return " ".join("".join(out).split())


def source_hash(kernel: str, read=None) -> str:
    """Hash of the code (comments and whitespace aside) of a kernel's sources;
    ``read(name)`` returns a source's text (default: the working tree)."""
    csrc = os.path.join(ROOT, "combine_expert_count_gb300", "csrc")
    if read is None:
        def read(f):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                return fh.read()
    h = hashlib.sha256()
    for f in KERNEL_SOURCES[kernel]:
        h.update((f + "\n" + code_only(read(f))).encode())
    return h.hexdigest()[:16]


def dram_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from a committed ncu capture, or None when absent
    or taken on different kernel source."""
    p = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    try:
        lines = open(p).read().splitlines()
    except OSError:
        return None
    src = source_hash(kernel)
    for ln in lines:
        parts = ln.split()
        if len(parts) >= 4 and not ln.startswith("#") and parts[0] == kernel and \
                parts[1] == workload and parts[3] == src:
            return int(parts[2])
    return None


# ----------------------------------------------------------------- clocks


class ClockSampler:
    """nvidia-smi samples every 50 ms while the timed regions run."""

    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_id: str):
        self.idx = gpu_id
        self.proc = None
        self.file = None

    def __enter__(self):
        try:
            self.file = tempfile.NamedTemporaryFile("w+", suffix=".csv", delete=False)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.idx), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=self.file, stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.25)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()

    def summary(self):
        if self.proc is None or self.file is None:
            return None
        self.file.flush()
        rows = []
        with open(self.file.name) as f:
            for ln in f:
                p = [x.strip() for x in ln.split(",")]
                if len(p) >= 9:
                    rows.append(p)
        os.unlink(self.file.name)
        if not rows:
            return None
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None, "reasons": reasons,
                "samples": len(rows)}


def gpu_id(local: int) -> str:
    """nvidia-smi -i argument for this process's GPU (its UUID when torch
    exposes it, so CUDA_VISIBLE_DEVICES remapping does not matter)."""
    import torch
    try:
        u = str(torch.cuda.get_device_properties(local).uuid)
        return u if u.startswith("GPU-") else "GPU-" + u
    except (AttributeError, RuntimeError):
        vis = os.environ.get("CUDA_VISIBLE_DEVICES", "")
        ids = [v for v in vis.split(",") if v.strip()]
        return ids[local] if local < len(ids) else str(local)


# ----------------------------------------------------------------- dist


def dist_setup():
    import torch
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local))
    return world, rank, local


def max_over_ranks(v: float, world: int) -> float:
    if world <= 1:
        return v
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def barrier(world: int) -> None:
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


# ----------------------------------------------------------------- CPU oracle
#
# The CPU oracle as it stands, timed on the host cores over the same units
# the GPU value times: route_count + exchange + dispatch_send +
# dispatch_recv (dispatch) and combine_send + combine_recv (combine), on the
# full workload (every token of every rank), the expert stand-in run once
# outside the timer (oracle.ref.LayerTimer).


def oracle_layer_us(w, d, min_seconds: float, max_reps: int = 1000, warmup: int = 1):
    """Single-threaded oracle: mean microseconds per full layer (dispatch,
    combine, total) over whole layers until `min_seconds` of timed work (at
    least one layer), and the number of layers timed."""
    from oracle import ref
    lt = ref.LayerTimer(w.N, w.T, w.E, w.R, w.H, d["x"], d["topk_idx"], d["topk_w"],
                        1 if w.expert == "scale" else 0)
    for _ in range(warmup):
        lt.step()
    disp, comb = [], []
    spent = 0.0
    while len(disp) < max_reps and (not disp or spent < min_seconds):
        a, b = lt.step()
        disp.append(a)
        comb.append(b)
        spent += a + b
    return (statistics.mean(disp) * 1e6, statistics.mean(comb) * 1e6,
            statistics.mean(a + b for a, b in zip(disp, comb)) * 1e6, len(disp), spent)


def _all_cores_worker(path, shape, mode, steps, barrier, queue):
    """One process of the all-cores timing: its own copy of the layer."""
    try:
        from oracle import ref
        z = np.load(path)
        N, T, E, R, H = shape
        lt = ref.LayerTimer(N, T, E, R, H, z["x"], z["topk_idx"], z["topk_w"], mode)
        lt.step()                       # warm-up, untimed
    except Exception as e:              # noqa: BLE001 -- reported to the parent
        barrier.abort()
        queue.put(repr(e))
        return
    barrier.wait()
    t0 = time.perf_counter()
    for _ in range(steps):
        lt.step()
    queue.put((t0, time.perf_counter()))


def oracle_all_cores(w, d, steps: int = 2, procs: int = 0) -> dict:
    """The oracle on every host core at once: `procs` processes (default one
    per core), each timing `steps` full layers of the same workload after a
    common start; microseconds per layer = wall time / layers finished.  The
    oracle is plain single-threaded C, so the cores run independent layers
    (throughput, not the latency of one layer)."""
    import multiprocessing as mp
    n = procs or os.cpu_count() or 1
    ctx = mp.get_context("spawn")
    with tempfile.TemporaryDirectory() as tmp:
        path = os.path.join(tmp, "layer.npz")
        np.savez(path, x=d["x"], topk_idx=d["topk_idx"], topk_w=d["topk_w"])
        barrier, queue = ctx.Barrier(n), ctx.Queue()
        ps = [ctx.Process(target=_all_cores_worker,
                          args=(path, (w.N, w.T, w.E, w.R, w.H), 1 if w.expert == "scale" else 0,
                                steps, barrier, queue)) for _ in range(n)]
        for p in ps:
            p.start()
        spans = [queue.get(timeout=600) for _ in range(n)]
        for p in ps:
            p.join()
    errors = [x for x in spans if isinstance(x, str)]
    if errors:
        raise RuntimeError(f"oracle all-cores worker failed: {errors[0]}")
    wall = max(b for _, b in spans) - min(a for a, _ in spans)
    return {"cores": n, "value": round(wall / (n * steps) * 1e6, 1), "unit": UNIT,
            "layers": n * steps, "wall_s": round(wall, 2),
            "how": f"{n} processes, each {steps} full layers after a common start; "
                   "wall time / layers"}


def cpu_model() -> str:
    """The host CPU's model name as lscpu reports it (on Arm it decodes the
    part number), else the architecture."""
    import platform
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.startswith("Model name:"):
                return ln.split(":", 1)[1].strip()
    except (OSError, subprocess.SubprocessError):
        pass
    return platform.processor() or platform.machine()


def cpu_baseline_line(w, d, min_seconds: float, all_cores: bool, warmup: int = 1,
                      max_reps: int = 1000) -> dict:
    import platform
    dus, cus, tus, reps, spent = oracle_layer_us(w, d, min_seconds, max_reps, warmup)
    line = {"value": round(tus, 1), "unit": UNIT, "cores": 1, "kind": "oracle",
            "sample": f"the full layer ({w.N} ranks x {w.T} tokens, H={w.H}, E={w.E}, "
                      f"top-{w.R}), {reps} layers timed after {warmup} untimed, mean; "
                      "route_count + exchange + dispatch_send + dispatch_recv + "
                      "combine_send + combine_recv, stand-in outside the timer",
            "dispatch_us": round(dus, 1), "combine_us": round(cus, 1),
            "layers": reps, "cpu_seconds": round(spent, 2),
            "cpu": cpu_model(), "arch": platform.machine(), "nproc": os.cpu_count()}
    if all_cores:
        line["all_cores"] = oracle_all_cores(w, d)
    return line


# ----------------------------------------------------------------- arms


def run_reference(args) -> None:
    """The reference arm: the CPU oracle as it stands, one full layer per
    step on one host core (K timed layers after W untimed), plus the
    all-cores figure; rank 0 only under torchrun."""
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    from combine_expert_count_gb300 import workloads as W
    from oracle import ref
    ref.build()
    w = W.CONFIGS[args.config]
    d = W.generate(w)
    t0 = time.perf_counter()
    cb = cpu_baseline_line(w, d, float("inf"), all_cores=not args.no_all_cores,
                           warmup=args.warmup, max_reps=args.steps)
    wall = time.perf_counter() - t0
    value = cb["value"]
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(value / 1000, 4), "higher_is_better": False,
        "scaling": "weak", "vs_baseline": None, "dtype": "u8/f32 (plain C, fp32 accumulation)",
        "data": "synthetic (seeded)",
        "config": {"workload": f"{args.config}: N={w.N} ranks x T={w.T} tokens, H={w.H}, "
                               f"E={w.E}, top-{w.R}",
                   "N": w.N, "T": w.T, "H": w.H, "E": w.E, "R": w.R},
        "cpu_baseline": cb,
        "e2e": {"value": value, "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "wall_s": round(wall, 1),
    }
    print(json.dumps(line), flush=True)


def per_kernel_table(nbytes, favg, savg, rcx_k, A, w, workload) -> list:
    """Each kernel: event time (eager, L2 flushed), algorithmic bytes and GB/s,
    and where a committed ncu capture of the same source exists, its DRAM
    bytes per launch, GB/s and the ratio DRAM / algorithmic.  The routing
    kernels are latency-bound (a few KB): no roofline."""
    ids = 4 * w.N * w.T * w.R
    rows = []
    table = [("route_count", statistics.mean(rcx_k[0]), 2 * ids + 4 * w.N * w.E, None),
             ("exchange", statistics.mean(rcx_k[1]), 8 * w.N * w.E, None),
             ("route", favg["route"], nbytes["fused"]["route"], "route")]
    for k in ("dispatch_send", "dispatch_recv", "combine_send", "combine_recv"):
        table.append((k, savg[k], nbytes["separate"][k], k))
    for k in ("dispatch_fused", "combine_fused"):
        table.append((k, favg[k], nbytes["fused"][k], k))
    for name, ms, alg, key in table:
        r = {"kernel": name, "us": round(ms * 1000, 2), "algorithmic_mb": round(alg / 1e6, 2)}
        if name in ("route_count", "exchange", "route"):
            r["bound"] = "latency"
        else:
            r["algorithmic_gbs"] = round(alg / (ms * 1e-3) / 1e9, 1)
            dram = dram_traffic(key, workload) if key else None
            if dram is not None:
                r["dram_mb"] = round(dram / 1e6, 1)
                r["dram_gbs"] = round(dram / (ms * 1e-3) / 1e9, 1)
                r["dram_over_algorithmic"] = round(dram / alg, 3)
        rows.append(r)
    return rows


def fused_split(m, b, idx, wt, x, flush, K, peak, workload=None) -> dict:
    """Eager per-kernel times of the fused calls on one workload (L2 flushed
    before each step; an event after each launch): the route (latency-bound),
    the fused dispatch and the fused combine, each with its algorithmic
    bytes, GB/s and fraction of the measured copy peak."""
    import torch
    sh = b.shape
    tens = b.tensors(x=x, topk_idx=idx, topk_w=wt)
    calls = (lambda: m.moe_route(sh, idx, b.expert_count, b.send_off, b.expert_send_off,
                                 b.slot_row, b.grp_off, b.seg_off, b.csend_off, b.m_sizes,
                                 b.status),
             lambda: m.moe_dispatch_send_recv(sh, tens), lambda: m.moe_combine(sh, tens))
    st = torch.cuda.current_stream()
    for _ in range(3):
        flush.zero_()
        for c in calls:
            c()
    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(4)] for _ in range(K)]
    for k in range(K):
        flush.zero_()
        evs[k][0].record(st)
        for i, c in enumerate(calls):
            c()
            evs[k][i + 1].record(st)
    torch.cuda.synchronize()
    us = [statistics.mean(e[i].elapsed_time(e[i + 1]) for e in evs) * 1000 for i in range(3)]
    A = int(b.send_off[:, -1].sum().item())
    w = types_ns(N=b.N, T=b.T, H=b.H, R=b.R)
    nb = algorithmic_bytes(w, A)["fused"]
    out = {"route_us": round(us[0], 2)}
    for name, u in (("dispatch_fused", us[1]), ("combine_fused", us[2])):
        gbs = nb[name] / (u * 1e-6) / 1e9
        out[name] = {"us": round(u, 2), "algorithmic_mb": round(nb[name] / 1e6, 1),
                     "algorithmic_gbs": round(gbs, 1), "frac_of_peak": round(gbs / peak, 4)}
        dram = dram_traffic(name, workload) if workload else None
        if dram is not None:
            out[name]["dram_mb_ncu"] = round(dram / 1e6, 1)
    out["dispatch_us"] = round(us[0] + us[1], 2)
    out["combine_us"] = round(us[2], 2)
    return out


def types_ns(**kw):
    import types
    return types.SimpleNamespace(**kw)


def config_line(m, W, name, dev, capture, flush, K, W_, peak) -> dict:
    """Another configuration: fused and separate-call layer times (CUDA-graph
    replay), the dispatch / combine split with each fused kernel's roofline
    fraction (eager launches), and the 70%-of-nominal target of the
    separate-call byte model."""
    import torch
    w = W.CONFIGS[name]
    d = W.generate(w)
    b = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, device=dev)
    x = torch.from_numpy(d["x"].view(np.int16)).to(dev)
    idx = torch.from_numpy(d["topk_idx"]).to(dev)
    wt = torch.from_numpy(d["topk_w"]).to(dev)
    b.dispatch(x, idx)
    b.expert(1 if w.expert == "scale" else 0)
    b.combine(idx, wt)
    torch.cuda.synchronize()
    if int(b.status.item()) != 0:
        raise RuntimeError(f"{name}: device status {int(b.status.item())}")
    A = int(b.send_off[:, -1].sum().item())
    nb = algorithmic_bytes(w, A)
    st = torch.cuda.current_stream()
    res = {"workload": f"{name}: N={w.N} T={w.T} H={w.H} E={w.E} top-{w.R}, cap={b.cap}"}
    for key, calls in (("us", "fused"), ("separate_calls_us", "separate")):
        once = capture(lambda: (b.dispatch(x, idx, calls=calls), b.combine(idx, wt, calls=calls)))
        for _ in range(W_):
            flush.zero_()
            once()
        tt = []
        for _ in range(K):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            once()
            e1.record(st)
            tt.append((e0, e1))
        torch.cuda.synchronize()
        res[key] = round(statistics.mean(a.elapsed_time(c) for a, c in tt) * 1000, 2)
    moved = sum(nb["fused"].values())
    s8d = nb["s8d_dispatch"] + nb["s8d_combine"]
    res["bytes_moved_mb"] = round(moved / 1e6, 1)
    res["achieved_gbs"] = round(moved / (res["us"] * 1e-6) / 1e9, 1)
    res["frac_of_peak"] = round(moved / (res["us"] * 1e-6) / 1e9 / peak, 4)
    res.update(fused_split(m, b, idx, wt, x, flush, K, peak, name))
    res["separate_call_model_mb"] = round(s8d / 1e6, 1)
    res["target_us_70pct_nominal"] = round(s8d / (0.7 * NOMINAL_HBM_GBS * 1e9) * 1e6, 1)
    del b
    torch.cuda.empty_cache()
    return res


def oracle_table(args) -> None:
    """The CPU oracle, as it stands, per configuration and phase (dispatch =
    route_count + exchange + dispatch_send + dispatch_recv; combine =
    combine_send + combine_recv), single-threaded on full layers, and the
    DSv3 layer on all host cores; one JSON line."""
    import platform
    from combine_expert_count_gb300 import workloads as W
    from oracle import ref
    ref.build()
    out = {"cpu": cpu_model(), "arch": platform.machine(), "nproc": os.cpu_count(),
           "configs": []}
    for name in ("tiny", "dsv3_decode", "kimi_k2_decode", "qwen3_skew", "qwen3_worst", "prefill"):
        w = W.CONFIGS[name]
        d = W.generate(w)
        dus, cus, tus, reps, _ = oracle_layer_us(w, d, 0.0 if name == "prefill" else 3.0,
                                                 max_reps=1 if name == "prefill" else 1000)
        out["configs"].append({"workload": name, "layers": reps, "dispatch_us": round(dus, 1),
                               "combine_us": round(cus, 1), "layer_us": round(tus, 1)})
        del d
    w = W.CONFIGS["dsv3_decode"]
    out["all_cores_dsv3_decode"] = oracle_all_cores(w, W.generate(w))
    print(json.dumps(out), flush=True)


def pairs_of(w, idx) -> int:
    """(token, expert rank) pairs: the rows the send-side reduction sends."""
    ranks = np.asarray(idx).reshape(w.N * w.T, w.R) // w.Er
    return int(sum(len(set(r.tolist())) for r in ranks))


def partial_combine_line(m, buf, w, d, x, idx, wt, tens, capture, time_steps, time_kernels,
                         flush, K, W_, world):
    """moe_combine_partial timed beside moe_combine on the same step."""
    import torch
    buf.combine(idx, wt, calls="partial")
    torch.cuda.synchronize()
    once = capture(lambda: (m.moe_dispatch(buf.shape, tens), buf.combine(idx, wt,
                                                                          calls="partial")))
    for _ in range(W_):
        flush.zero_()
        once()
    step_ms = time_steps(once, K)
    kern = time_kernels((lambda: buf.combine(idx, wt, calls="partial"),), K)[0]
    A = int(buf.send_off[:, -1].sum().item())
    pairs = pairs_of(w, d["topk_idx"])
    nbytes = A * 2 * w.H + pairs * 2 * w.H + 2 * w.N * w.T * w.H + 12 * A
    k_us = statistics.mean(kern) * 1000
    return {"us": round(max_over_ranks(statistics.mean(step_ms), world) * 1000, 2),
            "combine_kernel_us": round(k_us, 2),
            "rows_sent": pairs, "rows_sent_receive_side": A,
            "bytes_moved_mb": round(nbytes / 1e6, 1),
            "achieved_gbs": round(nbytes / (k_us * 1e-6) / 1e9, 1),
            "how": "moe_dispatch + moe_combine_partial (per token, one bf16 partial row per "
                   "expert rank summed on the sending side, then added on the receiving side), "
                   "CUDA-graph replay; combine_kernel_us alone"}


def skew_line(m, W, name, dev, capture, flush, K, W_, peak) -> dict:
    """One layer (moe_dispatch + moe_combine, and with moe_combine_partial) on
    a skewed-routing workload."""
    import torch
    w = W.CONFIGS[name]
    d = W.generate(w)
    b = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, device=dev)
    x = torch.from_numpy(d["x"].view(np.int16)).to(dev)
    idx = torch.from_numpy(d["topk_idx"]).to(dev)
    wt = torch.from_numpy(d["topk_w"]).to(dev)
    b.dispatch(x, idx)
    b.expert(1 if w.expert == "scale" else 0)
    b.combine(idx, wt)
    torch.cuda.synchronize()
    if int(b.status.item()) != 0:
        raise RuntimeError(f"{name}: device status {int(b.status.item())}")
    res = {"workload": name, "max_recv_rows": int(b.grp_off[:, -1].max().item()),
           "mean_recv_rows": round(float(b.grp_off[:, -1].float().mean().item()), 1)}
    st = torch.cuda.current_stream()
    for key, calls in (("us", "fused"), ("us_send_side_reduction", "partial")):
        once = capture(lambda: (b.dispatch(x, idx), b.combine(idx, wt, calls=calls)))
        for _ in range(W_):
            flush.zero_()
            once()
        tt = []
        for _ in range(K):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(st)
            once()
            e1.record(st)
            tt.append((e0, e1))
        torch.cuda.synchronize()
        res[key] = round(statistics.mean(a.elapsed_time(c) for a, c in tt) * 1000, 2)
    res["rows_sent_send_side"] = pairs_of(w, d["topk_idx"])
    res["rows_sent_receive_side"] = int(b.send_off[:, -1].sum().item())
    res.update(fused_split(m, b, idx, wt, x, flush, K, peak, name))
    del b
    torch.cuda.empty_cache()
    return res


def run_ours(args) -> None:
    import torch

    from combine_expert_count_gb300 import moeroute as m
    from combine_expert_count_gb300 import workloads as W

    world, rank, local = dist_setup()
    dev = torch.device("cuda", local)
    torch.cuda.set_device(dev)
    m.lib()  # raises if the library is not built

    w = W.CONFIGS[args.config]
    d = W.generate(w)
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, cap=args.cap, device=dev)
    x = torch.from_numpy(d["x"].view(np.int16)).to(dev)
    idx = torch.from_numpy(d["topk_idx"]).to(dev)
    wt = torch.from_numpy(d["topk_w"]).to(dev)
    sh = buf.shape
    mode = 1 if w.expert == "scale" else 0

    # one untimed pass, and the expert stand-in whose output every step reuses
    buf.dispatch(x, idx)
    buf.expert(mode)
    buf.combine(idx, wt)
    torch.cuda.synchronize()
    status = int(buf.status.item())
    if status != 0:
        raise RuntimeError(f"device status {status}: {m.strerror(status)}")
    A = int(buf.send_off[:, -1].sum().item())
    nbytes = algorithmic_bytes(w, A)

    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    tens = buf.tensors(x=x, topk_idx=idx, topk_w=wt)
    route = lambda: m.moe_route(sh, idx, buf.expert_count, buf.send_off,  # noqa: E731
                                buf.expert_send_off, buf.slot_row, buf.grp_off, buf.seg_off,
                                buf.csend_off, buf.m_sizes, buf.status)
    fused_calls = (route, lambda: m.moe_dispatch_send_recv(sh, tens),
                   lambda: m.moe_combine(sh, tens))
    # a1 and a2 as their own calls (the separate-call form of the route)
    route_split = (
        lambda: m.moe_route_count(sh, idx, buf.expert_count, buf.send_off, buf.expert_send_off,
                                  buf.slot_row, buf.status),
        lambda: m.moe_exchange(sh, buf.expert_count, buf.send_off, buf.grp_off, buf.seg_off,
                               buf.csend_off, buf.m_sizes, buf.status))
    separate_calls = (
        route,
        lambda: m.moe_dispatch_send(sh, x, buf.slot_row, buf.send_q, buf.send_s, buf.send_tok,
                                    buf.status),
        lambda: m.moe_dispatch_recv(sh, buf.send_q, buf.send_s, buf.send_tok, buf.expert_count,
                                    buf.expert_send_off, buf.seg_off, buf.grp_q, buf.grp_s,
                                    buf.grp_src, buf.status),
        lambda: m.moe_combine_send(sh, buf.y, buf.expert_count, buf.expert_send_off,
                                   buf.send_off, buf.seg_off, buf.csend_off, buf.csend,
                                   buf.status),
        lambda: m.moe_combine_recv(sh, buf.csend, idx, wt, buf.slot_row, buf.send_off,
                                   buf.csend_off, buf.out, buf.status),
    )

    def run_calls(calls, ev=None):
        for i, c in enumerate(calls):
            c()
            if ev is not None:
                ev[i + 1].record(stream)

    def step_fused():
        """The headline step through the public API: moe_dispatch + moe_combine."""
        m.moe_dispatch(sh, tens)
        m.moe_combine(sh, tens)

    K = args.steps
    W_ = max(args.warmup, 3)

    # Each step form captured once as a CUDA graph (the library never waits on
    # the host, so the sequences capture); replays run exactly those kernels.
    def capture(fn):
        if args.eager:
            return fn
        cs = torch.cuda.Stream(device=dev)
        cs.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            fn()
        torch.cuda.synchronize()
        return g.replay

    fused_once = capture(step_fused)
    separate_once = capture(lambda: run_calls(separate_calls))
    for _ in range(W_):
        for f in (fused_once, separate_once):
            flush.zero_()
            f()
    torch.cuda.synchronize()

    xh = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
    xh.copy_(x)
    ih = torch.empty(idx.shape, dtype=idx.dtype, pin_memory=True)
    ih.copy_(idx)
    wh = torch.empty(wt.shape, dtype=wt.dtype, pin_memory=True)
    wh.copy_(wt)
    oh = torch.empty(buf.out.shape, dtype=buf.out.dtype, pin_memory=True)
    x2, i2, w2 = torch.empty_like(x), torch.empty_like(idx), torch.empty_like(wt)

    def ev_pair():
        return torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)

    def time_steps(fn, n):
        evs = [ev_pair() for _ in range(n)]
        for k in range(n):
            flush.zero_()
            evs[k][0].record(stream)
            fn()
            evs[k][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    def time_kernels(calls, n):
        # untimed passes of the same eager sequence first: the first eager
        # launches after the graph replays measured several µs slow
        for _ in range(W_):
            flush.zero_()
            run_calls(calls)
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(len(calls) + 1)]
               for _ in range(n)]
        for k in range(n):
            flush.zero_()
            evs[k][0].record(stream)
            run_calls(calls, evs[k])
        torch.cuda.synchronize()
        return [[ev[i].elapsed_time(ev[i + 1]) for ev in evs] for i in range(len(calls))]

    def time_in_graph(n):
        """The headline step captured again with an event node before, between
        and after its two calls, replayed as the timed steps are (L2 flushed
        before each): how long moe_dispatch (route + fused dispatch) and
        moe_combine (the fused combine kernel alone) take inside a graph
        replay.  None where this torch records no events as graph nodes."""
        try:
            ev = [torch.cuda.Event(enable_timing=True, external=True) for _ in range(3)]
            cs = torch.cuda.Stream(device=dev)
            cs.wait_stream(stream)
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=cs):
                ev[0].record(cs)
                m.moe_dispatch(sh, tens)
                ev[1].record(cs)
                m.moe_combine(sh, tens)
                ev[2].record(cs)
            torch.cuda.synchronize()
            out = ([], [])
            for k in range(n + W_):
                flush.zero_()
                g.replay()
                torch.cuda.synchronize()
                if k >= W_:
                    out[0].append(ev[0].elapsed_time(ev[1]))
                    out[1].append(ev[1].elapsed_time(ev[2]))
            return out
        except (TypeError, RuntimeError):
            return None

    barrier(world)
    torch.cuda.synchronize()
    with ClockSampler(gpu_id(local)) as clk:
        # (1) headline: whole steps, L2 flushed before each (outside the window)
        t_wall = time.perf_counter()
        step_ms = time_steps(fused_once, K)
        t_wall = time.perf_counter() - t_wall
        barrier(world)
        # (2) the same outputs through the separate calls of the pages' steps
        sep_ms = time_steps(separate_once, K)
        # (3) per-kernel breakdowns: eager launches, an event after each call
        fused_k = time_kernels(fused_calls, K)
        sep_k = time_kernels(separate_calls, K)
        rcx_k = time_kernels(route_split, K)
        in_graph = None if args.eager else time_in_graph(K)
        # (4) end to end through the public API with host buffers in pinned
        # memory, all transfers inside the window: the router's ids and
        # weights are copied host -> device, the kernels read x from host
        # memory and write the combined output to host memory directly over
        # the CPU-GPU link
        e2e_ms = []
        for k in range(K + W_):
            flush.zero_()
            e0, e1 = ev_pair()
            e0.record(stream)
            i2.copy_(ih, non_blocking=True)
            w2.copy_(wh, non_blocking=True)
            buf.dispatch(xh, i2)
            buf.combine(i2, w2, out=oh)
            e1.record(stream)
            torch.cuda.synchronize()
            if k >= W_:
                e2e_ms.append(e0.elapsed_time(e1))
        if not torch.equal(oh.view(torch.int16), buf.out.cpu().view(torch.int16)):
            buf.combine(idx, wt)
            torch.cuda.synchronize()
            if not torch.equal(oh.view(torch.int16), buf.out.cpu().view(torch.int16)):
                raise RuntimeError("end-to-end output differs from the device-buffer output")
        # the same with explicit copies (pinned host -> device, device -> host)
        e2e_copy_ms = []
        for k in range(K + W_):
            flush.zero_()
            e0, e1 = ev_pair()
            e0.record(stream)
            x2.copy_(xh, non_blocking=True)
            i2.copy_(ih, non_blocking=True)
            w2.copy_(wh, non_blocking=True)
            buf.dispatch(x2, i2)
            buf.combine(i2, w2)
            oh.copy_(buf.out, non_blocking=True)
            e1.record(stream)
            torch.cuda.synchronize()
            if k >= W_:
                e2e_copy_ms.append(e0.elapsed_time(e1))

    # the low-latency calls on the same workload, when T fits
    ll = None
    if w.T <= 1024:
        llb = m.MoeLLBuffers(w.N, w.T, w.E, w.R, w.H, device=dev)
        llb.dispatch(x, idx)
        llb.expert(mode)
        llb.combine(wt)
        torch.cuda.synchronize()
        if int(llb.status.item()) != 0 or not torch.equal(llb.out, buf.out):
            raise RuntimeError("low-latency output differs from the main path")
        ll_once = capture(lambda: (llb.dispatch(x, idx), llb.combine(wt)))
        for _ in range(W_):
            flush.zero_()
            ll_once()
        ll_ms = time_steps(ll_once, K)
        ll_k = time_kernels((lambda: llb.dispatch(x, idx), lambda: llb.combine(wt)), K)
        row8 = w.H + 4 * (w.H // 128)
        ll_bytes = {"dispatch_ll": 2 * w.N * w.T * w.H + A * (row8 + 4) + 8 * A + 4 * A,
                    "combine_ll": A * 2 * w.H + 2 * w.N * w.T * w.H + 8 * A}
        ll_us = max_over_ranks(statistics.mean(ll_ms), world) * 1000
        ll = {"us": round(ll_us, 2),
              "kernel_us": {"dispatch_ll": round(statistics.mean(ll_k[0]) * 1000, 2),
                            "combine_ll": round(statistics.mean(ll_k[1]) * 1000, 2)},
              "bytes_moved_mb": {k: round(v / 1e6, 1) for k, v in ll_bytes.items()},
              "achieved_gbs": round(sum(ll_bytes.values()) / (ll_us * 1e-6) / 1e9, 1),
              "how": "moe_dispatch_ll + moe_combine_ll (fixed T-row regions per (expert, "
                     "sender); no send or combine send buffers), CUDA-graph replay"}
        del llb

    # the signalled dispatch: route, then send and receive shuffle in one
    # kernel handing rows over by per-(sender, receiver) flags; same outputs
    # as moe_dispatch, moving the bytes of the separate send + receive
    buf.dispatch(x, idx, calls="signalled")
    torch.cuda.synchronize()
    if int(buf.status.item()) != 0:
        raise RuntimeError("signalled dispatch raised a status")
    sig_once = capture(lambda: (buf.dispatch(x, idx, calls="signalled"), buf.combine(idx, wt)))
    for _ in range(W_):
        flush.zero_()
        sig_once()
    sig_ms = time_steps(sig_once, K)
    sig_k = time_kernels((route, lambda: buf.dispatch(x, idx, calls="signalled")), K)
    sig_disp_us = (statistics.mean(sig_k[1]) - statistics.mean(sig_k[0])) * 1000
    sig_bytes = nbytes["separate"]["dispatch_send"] + nbytes["separate"]["dispatch_recv"]
    signalled = {
        "us": round(max_over_ranks(statistics.mean(sig_ms), world) * 1000, 2),
        "dispatch_call_us": round(statistics.mean(sig_k[1]) * 1000, 2),
        "kernel_us": round(sig_disp_us, 2),
        "bytes_moved_mb": round(sig_bytes / 1e6, 1),
        "achieved_gbs": round(sig_bytes / (sig_disp_us * 1e-6) / 1e9, 1) if sig_disp_us > 0
        else None,
        "how": "moe_dispatch_signalled (route + one co-resident kernel: every CTA packs its "
               "tokens, publishing (sender, receiver) groups, then pulls its send rows as their "
               "groups are published) + moe_combine, CUDA-graph replay; kernel_us = call minus "
               "the route kernel"}

    # the combine with send-side reduction on the same expert outputs
    partial = partial_combine_line(m, buf, w, d, x, idx, wt, tens, capture, time_steps,
                                   time_kernels, flush, K, W_, world)
    others = None
    if rank == 0 and not args.no_skew:
        others = [config_line(m, W, name, dev, capture, flush, min(K, 20), W_, measured_peak()[0])
                  for name in ("kimi_k2_decode", "prefill")]
    if rank == 0 and not args.no_skew:
        skew = [skew_line(m, W, name, dev, capture, flush, K, W_, measured_peak()[0])
                for name in ("qwen3_zipf0", "qwen3_zipf0.5", "qwen3_zipf1", "qwen3_zipf1.5",
                             "qwen3_skew")]
    else:
        skew = None

    mean_step_ms = max_over_ranks(statistics.mean(step_ms), world)
    sep_step_ms = max_over_ranks(statistics.mean(sep_ms), world)
    e2e_us = max_over_ranks(statistics.mean(e2e_ms), world) * 1000
    h2d = xh.numel() * xh.element_size() + ih.numel() * 4 + wh.numel() * 4
    d2h = oh.numel() * oh.element_size()
    status = int(buf.status.item())
    if status != 0:
        raise RuntimeError(f"device status {status}: {m.strerror(status)}")
    if rank != 0:
        return

    peak, peak_kind = measured_peak()
    us = mean_step_ms * 1000
    moved = sum(nbytes["fused"].values())
    achieved = moved / (us * 1e-6) / 1e9
    favg = {n: statistics.mean(v) for n, v in zip(FUSED, fused_k)}
    savg = {n: statistics.mean(v) for n, v in zip(KERNELS, sep_k)}
    dom = max(("dispatch_fused", "combine_fused"), key=favg.get)
    # the dominant kernel's duration: inside the graph replays where events
    # can be graph nodes (moe_combine is the fused combine kernel alone),
    # else its eager launch
    dom_ms, dom_how = favg[dom], "eager launch, an event on each side, L2 flushed before the step"
    if in_graph is not None and dom == "combine_fused":
        dom_ms = statistics.mean(in_graph[1])
        dom_how = ("inside CUDA-graph replays of the headline step (event nodes around "
                   "moe_combine, L2 flushed before each step)")
    dom_gbs = nbytes["fused"][dom] / (dom_ms * 1e-3) / 1e9
    line = {
        "metric": METRIC, "value": round(us, 2), "unit": UNIT, "n_gpus": world, "steps": K,
        "warmup": W_, "ms_per_step": round(mean_step_ms, 5),
        "higher_is_better": False, "scaling": "weak", "vs_baseline": None,
        "dtype": "fp8-e4m3 dispatch (fp32 scales), bf16 combine with f32 accumulation",
        "data": "synthetic (seeded N(0,1) activations, softmax top-k routing)",
        "config": {"workload": f"{args.config}: N={w.N} ranks x T={w.T} tokens, H={w.H}, "
                               f"E={w.E}, top-{w.R}, cap={buf.cap}, expert stand-in "
                               f"{'per-expert scale' if mode else 'identity'}",
                   "N": w.N, "T": w.T, "H": w.H, "E": w.E, "R": w.R, "cap": buf.cap,
                   "l2": "flushed before every step (512 MiB write, outside the timed window)",
                   "path": "moe_dispatch + moe_combine (fused calls; all outputs of the six "
                           "separate calls written every step)",
                   "parallelism": "ranks simulated as slices of one GPU; replicas across GPUs"},
        "timing": "CUDA-graph replay" if not args.eager else "eager launches",
        "separate_calls_us": round(sep_step_ms * 1000, 2),
        "low_latency": ll,
        "signalled": signalled,
        "send_side_reduction": partial,
        "routing_skew": skew,
        "other_configs": others,
        "per_kernel": per_kernel_table(nbytes, favg, savg, rcx_k, A, w, args.config),
        "dispatch_us": round((favg["route"] + favg["dispatch_fused"]) * 1000, 2),
        "combine_us": round(favg["combine_fused"] * 1000, 2),
        "achieved_gbs": round(achieved, 1),
        "frac_of_peak": round(achieved / peak, 4), "peak_gbs": peak, "peak_kind": peak_kind,
        "frac_of_nominal_8tbs": round(achieved / NOMINAL_HBM_GBS, 4),
        "bytes_moved_mb": {k: round(v / 1e6, 1) for k, v in nbytes["fused"].items()},
        "separate_call_model_mb": {"dispatch": round(nbytes["s8d_dispatch"] / 1e6, 1),
                                   "combine": round(nbytes["s8d_combine"] / 1e6, 1),
                                   "note": "bytes if every buffer of the six separate calls is "
                                           "written once and read once; the fused calls skip "
                                           "two of those reads, so no bandwidth is quoted on "
                                           "this model"},
        "kernel_us": {n: round(v * 1000, 2) for n, v in favg.items()},
        "separate_kernel_us": {n: round(v * 1000, 2) for n, v in savg.items()},
        "kernel_us_in_graph": None if in_graph is None else {
            "dispatch_call": round(statistics.mean(in_graph[0]) * 1000, 2),
            "combine_fused": round(statistics.mean(in_graph[1]) * 1000, 2)},
        "roofline": {"bound": "hbm", "kernel": KERNEL_SYMBOL[dom],
                     "achieved": round(dom_gbs, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(dom_gbs / peak, 4),
                     "traffic": dram_traffic(dom, args.config),
                     "algorithmic_bytes": nbytes["fused"][dom],
                     "kernel_us": round(dom_ms * 1000, 2), "how": dom_how},
        "e2e": {"value": round(e2e_us, 2), "unit": UNIT, "h2d_bytes_per_step": int(h2d),
                "d2h_bytes_per_step": int(d2h),
                "how": "pinned host x read and out written by the kernels (zero copy); ids "
                       "and weights copied host -> device",
                "with_explicit_copies_us": round(statistics.mean(e2e_copy_ms) * 1000, 2)},
        "gpu_launches": len(FUSED) * K,  # our kernels in the headline timed region
        "clocks": clk.summary(),
        "status": status,
        "wall_s_timed": round(t_wall, 3),
    }
    if world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline_line(w, d, args.cpu_seconds,
                                                 all_cores=not args.no_all_cores)
    print(json.dumps(line), flush=True)


def profile_pass(args) -> None:
    """A fixed launch sequence for a profiler, nothing timed: every kernel of
    the main path, the separate calls, the signalled dispatch and the
    send-side-reduction combine, twice (the first pass warms up).  The
    low-latency layout is left out (its fixed regions hold several GB)."""
    import torch

    from combine_expert_count_gb300 import moeroute as m
    from combine_expert_count_gb300 import workloads as W

    w = W.CONFIGS[args.config]
    d = W.generate(w)
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, cap=args.cap)
    x = torch.from_numpy(d["x"].view(np.int16)).cuda()
    idx = torch.from_numpy(d["topk_idx"]).cuda()
    wt = torch.from_numpy(d["topk_w"]).cuda()
    mode = 1 if w.expert == "scale" else 0
    buf.dispatch(x, idx)
    buf.expert(mode)
    torch.cuda.synchronize()
    for _ in range(2):
        buf.dispatch(x, idx)                          # k_route_cluster, dispatch fused
        buf.combine(idx, wt)                          # k_combine_fused
        buf.dispatch(x, idx, calls="fused_route")     # route, quant + pack, receive shuffle
        buf.combine(idx, wt, calls="separate")        # combine pack, combine reduce
        buf.dispatch(x, idx, calls="signalled")       # route, signalled dispatch
        buf.combine(idx, wt, calls="partial")         # send-side reduction, one pass
        buf.combine(idx, wt, calls="partial_separate")
        torch.cuda.synchronize()
    if int(buf.status.item()) != 0:
        raise RuntimeError(f"device status {int(buf.status.item())}")
    print("profile pass done: 13 library launches per pass", flush=True)


def profile_headline(args) -> None:
    """The headline step only (moe_dispatch + moe_combine) eight times, L2
    flushed before each, nothing timed: a launch list of exactly the kernels
    the headline number times."""
    import torch

    from combine_expert_count_gb300 import moeroute as m
    from combine_expert_count_gb300 import workloads as W

    w = W.CONFIGS[args.config]
    d = W.generate(w)
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, cap=args.cap)
    x = torch.from_numpy(d["x"].view(np.int16)).cuda()
    idx = torch.from_numpy(d["topk_idx"]).cuda()
    wt = torch.from_numpy(d["topk_w"]).cuda()
    buf.dispatch(x, idx)
    buf.expert(1 if w.expert == "scale" else 0)
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device="cuda")
    xin, out = x, None
    if args.host_io:
        # the end-to-end form: x read from and out written to pinned host memory
        xin = torch.empty(x.shape, dtype=x.dtype, pin_memory=True)
        xin.copy_(x)
        out = torch.empty(buf.out.shape, dtype=buf.out.dtype, pin_memory=True)
    for _ in range(8):
        flush.zero_()
        buf.dispatch(xin, idx)
        buf.combine(idx, wt, out=out)
    torch.cuda.synchronize()
    if int(buf.status.item()) != 0:
        raise RuntimeError(f"device status {int(buf.status.item())}")
    print("headline profile pass done: 8 steps of 3 library launches"
          + (" (pinned host x and out)" if args.host_io else ""), flush=True)


PROFILE_CALLS = ("route", "dispatch", "combine", "dispatch_send", "dispatch_recv",
                 "combine_send", "combine_recv", "dispatch_ll", "combine_ll", "signalled",
                 "partial")


def profile_kernel(args) -> None:
    """One call form launched a few times for a single-kernel ncu capture,
    nothing timed: one untimed pass of the whole layer (which launches every
    kernel of the path once), then `--profile-reps` launches of the named call,
    L2 flushed before each.  With --cap (grouped rows per rank) or --tokens
    the case stays small enough for a full-set capture."""
    import torch

    from combine_expert_count_gb300 import moeroute as m
    from combine_expert_count_gb300 import workloads as W

    w = W.CONFIGS[args.config]
    if args.tokens:
        w = w.replace(T=args.tokens)
    d = W.generate(w)
    dev = torch.device("cuda", 0)
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, cap=args.cap, device=dev)
    x = torch.from_numpy(d["x"].view(np.int16)).to(dev)
    idx = torch.from_numpy(d["topk_idx"]).to(dev)
    wt = torch.from_numpy(d["topk_w"]).to(dev)
    mode = 1 if w.expert == "scale" else 0
    sh = buf.shape
    tens = buf.tensors(x=x, topk_idx=idx, topk_w=wt)
    buf.dispatch(x, idx)
    buf.expert(mode)
    buf.combine(idx, wt)
    ll = None
    if args.profile_kernel in ("dispatch_ll", "combine_ll"):
        ll = m.MoeLLBuffers(w.N, w.T, w.E, w.R, w.H, device=dev)
        ll.dispatch(x, idx)
        ll.expert(mode)
        ll.combine(wt)
    calls = {
        "route": lambda: buf.route(idx),
        "dispatch": lambda: m.moe_dispatch_send_recv(sh, tens),
        "combine": lambda: m.moe_combine(sh, tens),
        "dispatch_send": lambda: m.moe_dispatch_send(sh, x, buf.slot_row, buf.send_q, buf.send_s,
                                                     buf.send_tok, buf.status),
        "dispatch_recv": lambda: m.moe_dispatch_recv(sh, buf.send_q, buf.send_s, buf.send_tok,
                                                     buf.expert_count, buf.expert_send_off,
                                                     buf.seg_off, buf.grp_q, buf.grp_s,
                                                     buf.grp_src, buf.status),
        "combine_send": lambda: m.moe_combine_send(sh, buf.y, buf.expert_count,
                                                   buf.expert_send_off, buf.send_off, buf.seg_off,
                                                   buf.csend_off, buf.csend, buf.status),
        "combine_recv": lambda: m.moe_combine_recv(sh, buf.csend, idx, wt, buf.slot_row,
                                                   buf.send_off, buf.csend_off, buf.out,
                                                   buf.status),
        "dispatch_ll": lambda: ll.dispatch(x, idx),
        "combine_ll": lambda: ll.combine(wt),
        "signalled": lambda: buf.dispatch(x, idx, calls="signalled"),
        "partial": lambda: buf.combine(idx, wt, calls="partial"),
    }
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    for _ in range(args.profile_reps):
        flush.zero_()
        calls[args.profile_kernel]()
    torch.cuda.synchronize()
    st = int(buf.status.item())
    if st != 0:
        raise RuntimeError(f"device status {st}")
    print(f"profile-kernel {args.profile_kernel}: {args.config} N={w.N} T={w.T} H={w.H} E={w.E} "
          f"top-{w.R} cap={buf.cap}, {args.profile_reps} launches after one layer pass, "
          f"{buf.device_bytes() / 1e9:.2f} GB of buffers", flush=True)


def token_sweep(args) -> None:
    """Layer time against tokens per rank on one configuration's shape: the
    fused calls (moe_dispatch + moe_combine) and the low-latency calls, each a
    CUDA-graph replay with L2 flushed before every step; one JSON line.  The
    low-latency layout holds N*E*T rows, so it runs up to --sweep-ll-max."""
    import torch

    from combine_expert_count_gb300 import moeroute as m
    from combine_expert_count_gb300 import workloads as W

    base = W.CONFIGS[args.config]
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    m.lib()
    flush = torch.empty(L2_FLUSH_BYTES, dtype=torch.uint8, device=dev)
    stream = torch.cuda.current_stream()
    K, W_ = args.steps, max(args.warmup, 3)
    mode = 1 if base.expert == "scale" else 0

    def capture(fn):
        cs = torch.cuda.Stream(device=dev)
        cs.wait_stream(stream)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=cs):
            fn()
        torch.cuda.synchronize()
        return g.replay

    def mean_us(once):
        for _ in range(W_):
            flush.zero_()
            once()
        evs = []
        for _ in range(K):
            flush.zero_()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            once()
            e1.record(stream)
            evs.append((e0, e1))
        torch.cuda.synchronize()
        return round(statistics.mean(a.elapsed_time(b) for a, b in evs) * 1000, 2)

    rows = []
    with ClockSampler(gpu_id(0)) as clk:
        for T in args.sweep_tokens:
            w = base.replace(T=T, seed=base.seed + 1000 + T)
            d = W.generate(w)
            b = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, device=dev)
            x = torch.from_numpy(d["x"].view(np.int16)).to(dev)
            idx = torch.from_numpy(d["topk_idx"]).to(dev)
            wt = torch.from_numpy(d["topk_w"]).to(dev)
            b.dispatch(x, idx)
            b.expert(mode)
            b.combine(idx, wt)
            torch.cuda.synchronize()
            if int(b.status.item()) != 0:
                raise RuntimeError(f"T={T}: device status {int(b.status.item())}")
            row = {"T": T, "tokens": w.N * T,
                   "fused_us": mean_us(capture(lambda: (b.dispatch(x, idx),
                                                        b.combine(idx, wt))))}
            if T <= args.sweep_ll_max:
                llb = m.MoeLLBuffers(w.N, w.T, w.E, w.R, w.H, device=dev)
                llb.dispatch(x, idx)
                llb.expert(mode)
                llb.combine(wt)
                torch.cuda.synchronize()
                if int(llb.status.item()) != 0 or not torch.equal(llb.out, b.out):
                    raise RuntimeError(f"T={T}: low-latency output differs from the main path")
                row["low_latency_us"] = mean_us(capture(lambda: (llb.dispatch(x, idx),
                                                                 llb.combine(wt))))
                del llb
            rows.append(row)
            del b
            torch.cuda.empty_cache()
    print(json.dumps({"sweep": "tokens per rank", "workload": args.config,
                      "shape": {"N": base.N, "H": base.H, "E": base.E, "R": base.R},
                      "steps": K, "warmup": W_, "timing": "CUDA-graph replay, L2 flushed "
                      "before every step", "clocks": clk.summary(), "rows": rows}), flush=True)


def main() -> None:
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--config", default="dsv3_decode")
    ap.add_argument("--cap", type=int, default=0,
                    help="grouped rows per rank (0: N*T*min(R,E/N), the library default)")
    ap.add_argument("--eager", action="store_true",
                    help="time eager launches instead of CUDA-graph replays")
    ap.add_argument("--impl", choices=("ours", "reference"), default="ours")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="minimum CPU time spent on the single-threaded oracle baseline")
    ap.add_argument("--no-all-cores", action="store_true",
                    help="skip the oracle timing on every host core")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-skew", action="store_true",
                    help="skip the skewed-routing (Zipf) layer lines")
    ap.add_argument("--profile-pass", action="store_true",
                    help="run every kernel twice without timing (for ncu) and exit")
    ap.add_argument("--oracle-table", action="store_true",
                    help="time the CPU oracle per configuration and phase, then exit")
    ap.add_argument("--profile-headline", action="store_true",
                    help="run only the headline step eight times without timing (for ncu)")
    ap.add_argument("--host-io", action="store_true",
                    help="with --profile-headline: x and out in pinned host memory (the "
                         "end-to-end form)")
    ap.add_argument("--profile-kernel", choices=PROFILE_CALLS,
                    help="launch one call a few times without timing (for a single-kernel "
                         "ncu capture), then exit")
    ap.add_argument("--profile-reps", type=int, default=3)
    ap.add_argument("--tokens", type=int, default=0,
                    help="tokens per rank for --profile-kernel (0: the config's)")
    ap.add_argument("--token-sweep", action="store_true",
                    help="time the layer against tokens per rank (fused and low-latency), "
                         "then exit")
    ap.add_argument("--sweep-tokens", type=int, nargs="+",
                    default=[1, 4, 16, 32, 64, 128, 256, 512])
    ap.add_argument("--sweep-ll-max", type=int, default=256,
                    help="largest T of the sweep that also runs the low-latency calls")
    args = ap.parse_args()
    if args.profile_kernel:
        profile_kernel(args)
    elif args.token_sweep:
        token_sweep(args)
    elif args.profile_headline:
        profile_headline(args)
    elif args.profile_pass:
        profile_pass(args)
    elif args.oracle_table:
        oracle_table(args)
    elif args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
