"""GPU parity of the combine with send-side reduction (moe_combine_partial,
and moe_combine_partial_send + moe_combine_partial_recv) against the CPU
oracle: the partial rows and the combined output bit for bit, rows of an
(expert rank, sender, token) without an expert of that rank untouched."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from combine_expert_count_gb300 import moeroute as m
from combine_expert_count_gb300 import workloads as W
from oracle import ref

from . import _gpu as G

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_expert_count_gb300 import build
    build.build()
    ref.build()
    m.lib()


def _run(w, d, calls, cap=0, out=None):
    dd = G.to_dev(d)
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, cap=cap)
    G.fill_sentinels(buf)
    buf.partial_rows().view(torch.int16).fill_(G.SENT_U16)
    buf.dispatch(dd["x"], dd["topk_idx"])
    buf.expert(1 if w.expert == "scale" else 0)
    res = buf.combine(dd["topk_idx"], dd["topk_w"], calls=calls, out=out)
    torch.cuda.synchronize()
    return buf, res


def _check(w, d, calls, cap=0):
    cap_o = cap or w.default_cap
    o = ref.layer_partial(w.N, w.T, w.E, w.R, w.H, cap_o, d["x"], d["topk_idx"], d["topk_w"],
                          mode=1 if w.expert == "scale" else 0)
    buf, _ = _run(w, d, calls, cap)
    G.assert_eq("part", G.host(buf.part), o["part"])
    G.assert_eq("out", G.host(buf.out), o["out_partial"])
    return buf, o


@pytest.mark.parametrize("calls", ["partial", "partial_separate"])
@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "qwen3_skew", "qwen3_zipf1.5"])
def test_config_parity(name, calls):
    w = W.CONFIGS[name]
    if name == "qwen3_skew":
        w = w.replace(T=128)
    _check(w, W.generate(w), calls)


@pytest.mark.parametrize("N,T,E,R,H", [(1, 3, 2, 2, 128), (2, 5, 8, 3, 256), (4, 16, 16, 4, 384),
                                       (3, 7, 12, 8, 128), (4, 4, 32, 12, 256),
                                       (2, 9, 64, 32, 128), (4, 8, 1024, 32, 128),
                                       (1, 16, 1024, 32, 128), (2, 40, 8, 8, 2048),
                                       (2, 3, 4, 2, 65536), (32, 1, 1024, 32, 128)])
def test_small_shapes_and_many_experts(N, T, E, R, H):
    """Includes R > 8 (the shared-memory slot loop), R = 32, one rank
    holding all 1024 experts, 2048-element rows (the narrow blocks, two per
    token) with every expert of a rank taken by each token, the widest row,
    and one token per rank on 32 ranks with 1024 experts and 32 slots."""
    w = W.Workload("grid", N=N, T=T, H=H, E=E, R=R, seed=41 + N * 100 + T * 10 + R)
    d = W.generate(w)
    for calls in ("partial", "partial_separate"):
        _check(w, d, calls)


def test_bad_ids_duplicates_and_capacity_drops():
    w = W.Workload("edge", N=2, T=12, H=256, E=4, R=3, seed=9)
    d = W.generate(w)
    d["topk_idx"][0, 1, 1] = -1
    d["topk_idx"][1, 5, 0] = 4
    d["topk_idx"][0, 3] = [1, 1, 0]
    d["topk_idx"][1, 2] = [3, 3, 3]
    for cap in (0, 9):
        for calls in ("partial", "partial_separate"):
            _check(w, d, calls, cap)


def test_empty_batch():
    buf = m.MoeBuffers(2, 0, 4, 2, 128, cap=1)
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    zf = torch.zeros(1, dtype=torch.float32, device="cuda")
    buf.dispatch(z, z)
    buf.combine(z, zf, calls="partial")
    buf.combine(z, zf, calls="partial_separate")
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0


def test_pinned_host_out_and_graph_replay():
    w = W.CONFIGS["dsv3_decode"].replace(T=16)
    d = W.generate(w)
    want, _ = _run(w, d, "partial")
    dd = G.to_dev(d)
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H)
    buf.dispatch(dd["x"], dd["topk_idx"])
    buf.expert(1)
    oh = torch.empty(buf.out.shape, dtype=buf.out.dtype, pin_memory=True)
    buf.combine(dd["topk_idx"], dd["topk_w"], calls="partial", out=oh)
    torch.cuda.synchronize()
    assert torch.equal(oh.view(torch.int16), want.out.cpu().view(torch.int16))
    buf.out.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        buf.combine(dd["topk_idx"], dd["topk_w"], calls="partial")
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(buf.out, want.out)
