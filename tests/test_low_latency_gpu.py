"""GPU parity of the low-latency calls (moe_dispatch_ll, moe_expert_standin_ll,
moe_combine_ll) against the oracle's low-latency layout, token by token, and
against the main path's combined output (the same fused multiply-adds in the
same slot order give the same bits)."""
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


def _run_ll(w, d, mode):
    b = m.MoeLLBuffers(w.N, w.T, w.E, w.R, w.H)
    b.ll_q.fill_(G.SENT_U8)
    b.ll_s.fill_(float("nan"))
    b.ll_src.fill_(G.SENT_I32)
    b.ll_row.fill_(G.SENT_I32)
    b.ll_count.fill_(G.SENT_I32)
    b.y_ll.view(torch.int16).fill_(G.SENT_U16)
    b.status.fill_(-1)
    dd = G.to_dev(d)
    b.dispatch(dd["x"], dd["topk_idx"])
    b.expert(mode)
    b.combine(dd["topk_w"])
    torch.cuda.synchronize()
    return b


def _check_ll(w, d, b, mode, tokens=None):
    o = ref.ll_rows(w.N, w.T, w.E, w.R, d["topk_idx"])
    G.assert_eq("ll_row", G.host(b.ll_row), o["ll_row"])
    G.assert_eq("ll_count", G.host(b.ll_count), o["ll_count"])
    assert int(b.status.item()) == o["status"]
    q_all, s_all, src_all = G.host(b.ll_q), G.host(b.ll_s), G.host(b.ll_src)
    y_all, out = G.host(b.y_ll), G.host(b.out)
    written = np.zeros(q_all.shape[0], bool)
    toks = range(w.N * w.T) if tokens is None else tokens
    for flat in toks:
        s, t = divmod(int(flat), w.T)
        q, sc = ref.quant_token(w.H, d["x"][s, t])
        rows, use = [], []
        for k in range(w.R):
            row = int(o["ll_row"][s, t, k])
            if row < 0:
                rows.append(np.zeros(w.H, np.uint16))
                use.append(0)
                continue
            e = int(d["topk_idx"][s, t, k])
            G.assert_eq("ll_q", q_all[row], q)
            G.assert_eq("ll_s", s_all[row], sc)
            assert src_all[row] == t
            yr = ref.standin_row(w.H, mode, e, q, sc)
            G.assert_eq("y_ll", y_all[row], yr)
            written[row] = True
            rows.append(yr)
            use.append(1)
        want = ref.weighted_sum(np.stack(rows), d["topk_w"][s, t], np.array(use, np.int32))
        G.assert_eq("out", out[s, t], want)
    if tokens is None:
        assert np.all(q_all[~written] == G.SENT_U8), "rows outside the layout were written"


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "qwen3_skew", "qwen3_worst"])
def test_ll_config_parity(name):
    w = W.CONFIGS[name]
    d = W.generate(w)
    mode = 1 if w.expert == "scale" else 0
    b = _run_ll(w, d, mode)
    _check_ll(w, d, b, mode, tokens=None if w.N * w.T <= 2048 else
              np.random.default_rng(0).choice(w.N * w.T, 256, replace=False))


def test_ll_output_equals_main_path():
    w = W.CONFIGS["dsv3_decode"]
    d = W.generate(w)
    b = _run_ll(w, d, 1)
    main = G.run_path(w, G.to_dev(d))
    assert torch.equal(b.out.view(torch.int16), main.out.view(torch.int16))


@pytest.mark.parametrize("N,T,E,R,H", [(1, 5, 4, 2, 128), (2, 16, 8, 3, 256), (3, 7, 6, 2, 384),
                                       (4, 33, 16, 4, 640), (2, 3, 4, 2, 8192 + 1024),
                                       (2, 9, 32, 12, 128), (2, 5, 64, 32, 256),
                                       (2, 1024, 8, 2, 128), (4, 8, 1024, 32, 128),
                                       (3, 700, 12, 4, 256), (2, 1024, 64, 32, 128),
                                       (5, 520, 1000, 8, 128), (2, 3, 4, 2, 65536),
                                       (1, 16, 1024, 32, 128), (1, 1024, 64, 4, 128),
                                       (32, 1, 1024, 32, 128)])
def test_ll_small_shapes(N, T, E, R, H):
    """Includes more than eight slots per token (the earlier-id count runs in
    groups of eight), 32 slots, the longest batch (T = 1024) and the most
    experts (1024, the largest region-count histogram); the last three have
    more than 2048 ids per rank, so each sender's ids are ranked once in the
    same launch (more experts than the CTA has threads in the last); the
    widest row the ABI takes (65536 elements); one rank holding all 1024
    experts, and one rank ranking 4096 ids."""
    w = W.Workload("llgrid", N=N, T=T, H=H, E=E, R=R, seed=N * 100 + T)
    d = W.generate(w)
    b = _run_ll(w, d, 0)
    _check_ll(w, d, b, 0)


def test_ll_duplicates_overflow_and_bad_ids():
    w = W.Workload("lldup", N=2, T=4, H=256, E=4, R=3, seed=9)
    d = W.generate(w)
    d["topk_idx"][0, :, :] = 1          # 12 rows for expert 1 from rank 0: 4 fit
    d["topk_idx"][1, 2, 1] = -3
    b = _run_ll(w, d, 0)
    o = ref.ll_rows(w.N, w.T, w.E, w.R, d["topk_idx"])
    assert o["status"] == ref.ST_CAPACITY | ref.ST_BAD_EXPERT
    _check_ll(w, d, b, 0)


def test_ll_ranked_duplicates_overflow_and_bad_ids():
    """The ranked form (more than 2048 ids per rank): regions that overflow
    their T rows, duplicate experts inside a token and bad ids."""
    w = W.Workload("llrank", N=2, T=600, H=256, E=4, R=4, seed=19)
    d = W.generate(w)
    d["topk_idx"][0, :, 0] = 1           # 600 rows of sender 0 for expert 1, plus duplicates
    d["topk_idx"][0, :300, 1] = 1
    d["topk_idx"][1, 7, 2] = -1
    d["topk_idx"][1, 9, 3] = 4
    b = _run_ll(w, d, 0)
    o = ref.ll_rows(w.N, w.T, w.E, w.R, d["topk_idx"])
    assert o["status"] == ref.ST_CAPACITY | ref.ST_BAD_EXPERT
    _check_ll(w, d, b, 0)


def test_ll_rejects_long_batches():
    sh = m.make_shape(2, 1025, 8, 2, 256)
    z = m.sizes_query(sh)
    p = torch.zeros(16, dtype=torch.int32, device="cuda")
    import ctypes
    rc = m.lib().moe_dispatch_ll(ctypes.byref(sh), *([ctypes.c_void_p(p.data_ptr())] * 8), None)
    assert rc == m.MOE_ENOTSUP and z.ll_rows == 2 * 8 * 1025


def _fill_sentinels(b):
    b.ll_q.fill_(G.SENT_U8)
    b.ll_s.fill_(float("nan"))
    b.ll_src.fill_(G.SENT_I32)
    b.ll_row.fill_(G.SENT_I32)
    b.ll_count.fill_(G.SENT_I32)
    b.y_ll.view(torch.int16).fill_(G.SENT_U16)
    b.status.fill_(-1)


@pytest.mark.parametrize("N,T,E,R,H", [(4, 32, 64, 8, 1024),     # per-token row search
                                       (2, 1024, 16, 4, 512)])   # senders ranked first
def test_ll_graph_replay_with_new_inputs(N, T, E, R, H):
    """The three low-latency calls captured once in a CUDA graph and replayed
    on two different inputs copied into the captured tensors: each replay
    equals the oracle on its own inputs (rows, counts, payload, output), and
    rows outside the second input's layout keep their sentinels."""
    w = W.Workload("llgraph", N=N, T=T, H=H, E=E, R=R, seed=N * 1000 + T)
    d_a = W.generate(w)
    d_b = W.generate(w.replace(seed=w.seed + 1))
    b = m.MoeLLBuffers(w.N, w.T, w.E, w.R, w.H)
    st = G.to_dev(d_a)
    x, idx, wt = st["x"].clone(), st["topk_idx"].clone(), st["topk_w"].clone()
    b.dispatch(x, idx)   # load the kernels before capture
    b.expert(1)
    b.combine(wt)
    torch.cuda.synchronize()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b.dispatch(x, idx)
        b.expert(1)
        b.combine(wt)
    for d in (d_a, d_b):
        dd = G.to_dev(d)
        x.copy_(dd["x"])
        idx.copy_(dd["topk_idx"])
        wt.copy_(dd["topk_w"])
        _fill_sentinels(b)
        torch.cuda.synchronize()
        g.replay()
        torch.cuda.synchronize()
        _check_ll(w, d, b, 1)


@pytest.mark.parametrize("N,T,E,R,H", [(16, 32, 256, 8, 7168),   # per-token row search
                                       (2, 1024, 16, 4, 512)])   # senders ranked first
def test_ll_pinned_host_x(N, T, E, R, H):
    """x read from pinned host memory by the low-latency dispatch gives the
    same rows, counts and output as x in device memory."""
    w = W.Workload("llhost", N=N, T=T, H=H, E=E, R=R, seed=N * 10 + T)
    d = W.generate(w)
    ref_b = _run_ll(w, d, 1)
    dd = G.to_dev(d)
    b = m.MoeLLBuffers(w.N, w.T, w.E, w.R, w.H)
    _fill_sentinels(b)
    xh = torch.empty(dd["x"].shape, dtype=dd["x"].dtype, pin_memory=True)
    xh.copy_(dd["x"])
    b.dispatch(xh, dd["topk_idx"])
    b.expert(1)
    b.combine(dd["topk_w"])
    torch.cuda.synchronize()
    for k in ("ll_row", "ll_count", "status", "out"):
        assert torch.equal(getattr(b, k).view(torch.uint8), getattr(ref_b, k).view(torch.uint8)), k
    rows = ref_b.ll_row.flatten()
    rows = rows[rows >= 0].long()
    for k in ("ll_q", "ll_s", "ll_src"):
        assert torch.equal(getattr(b, k)[rows].view(torch.uint8),
                           getattr(ref_b, k)[rows].view(torch.uint8)), k


def test_ll_empty_batch():
    """No tokens: every region count is zero, the status clear, and the
    stand-in and combine have nothing to do."""
    w = W.Workload("llempty", N=4, T=0, H=256, E=8, R=2)
    b = m.MoeLLBuffers(w.N, w.T, w.E, w.R, w.H)
    b.ll_count.fill_(G.SENT_I32)
    b.status.fill_(-1)
    x = torch.zeros(16, dtype=torch.int16, device="cuda")
    idx = torch.zeros(16, dtype=torch.int32, device="cuda")
    wt = torch.zeros(16, dtype=torch.float32, device="cuda")
    b.dispatch(x, idx)
    b.expert(1)
    b.combine(wt)
    torch.cuda.synchronize()
    assert int(b.status.item()) == 0
    assert torch.all(b.ll_count == 0)
