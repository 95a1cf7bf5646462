"""GPU parity of moe_dispatch_signalled: the dispatch send and the receive
shuffle in one kernel whose CTAs hand rows over by per-(sender, receiver)
arrival flags (the one-GPU form of the decoupled signalling on the Perseus
page, section 3).  Its outputs are those of moe_dispatch, so every test
compares the whole path with the CPU oracle; the flag scratch must come back
zero, and a flag that nothing sets must end in MOE_ST_TIMEOUT, not a hang."""
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


def _oracle(w, d, cap):
    return ref.layer(w.N, w.T, w.E, w.R, w.H, cap, d["x"], d["topk_idx"], d["topk_w"],
                     mode=1 if w.expert == "scale" else 0)


def _exact_cap(w, d):
    rc = ref.route_count(w.N, w.T, w.E, w.R, d["topk_idx"])
    ex = ref.exchange(w.N, w.E, 1 << 30, rc["expert_count"], rc["send_off"])
    return max(1, int(ex["grp_off"][:, -1].max()))


def _run(w, d, cap=0):
    buf = G.run_path(w, G.to_dev(d), cap=cap, calls="signalled")
    assert int(buf.sig.abs().sum().item()) == 0, "flag scratch not cleared"
    return buf


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "kimi_k2_decode", "qwen3_skew",
                                  "qwen3_zipf1.5"])
def test_config_full_parity(name):
    w = W.CONFIGS[name]
    d = W.generate(w)
    G.compare_with_oracle(w, _run(w, d), _oracle(w, d, _exact_cap(w, d)))


def test_worst_case_all_tokens_to_one_rank():
    w = W.CONFIGS["qwen3_worst"].replace(T=64)
    d = W.generate(w)
    G.compare_with_oracle(w, _run(w, d), _oracle(w, d, w.default_cap))


@pytest.mark.parametrize("H", [128, 640, 8192 + 1024, 20480])
def test_row_pieces_and_odd_scale_rows(H):
    """Rows of several shared-memory pieces (each piece counts in its group)
    and scale rows that are not whole 16-byte vectors."""
    w = W.Workload("pieces", N=2, T=3, H=H, E=4, R=2, seed=H)
    d = W.generate(w)
    G.compare_with_oracle(w, _run(w, d), _oracle(w, d, w.default_cap))


@pytest.mark.parametrize("N,T,E,R,H", [(1, 1, 1, 1, 128), (1, 16, 4, 3, 256), (3, 5, 6, 2, 384),
                                       (4, 16, 16, 4, 128), (4, 1, 4, 4, 256),
                                       (2, 16, 8, 4, 384), (16, 7, 64, 8, 256)])
def test_small_shapes(N, T, E, R, H):
    w = W.Workload("grid", N=N, T=T, H=H, E=E, R=R, seed=17 + N * 1000 + T * 100 + E * 10 + R)
    d = W.generate(w)
    G.compare_with_oracle(w, _run(w, d), _oracle(w, d, w.default_cap))


def test_bad_ids_capacity_and_duplicates():
    w = W.Workload("bad", N=2, T=8, H=256, E=8, R=2, seed=3)
    d = W.generate(w)
    d["topk_idx"][0, 1, 1] = -1
    d["topk_idx"][1, 5, 0] = 8
    o = _oracle(w, d, w.default_cap)
    assert o["status"] == ref.ST_BAD_EXPERT
    G.compare_with_oracle(w, _run(w, d), o)

    w = W.Workload("cap", N=2, T=16, H=256, E=4, R=2, seed=11)
    d = W.generate(w)
    o = _oracle(w, d, 7)
    assert o["status"] & ref.ST_CAPACITY
    G.compare_with_oracle(w, _run(w, d, cap=7), o)

    w = W.Workload("dup", N=2, T=6, H=128, E=4, R=3, seed=5)
    d = W.generate(w)
    d["topk_idx"][0, 2] = [1, 1, 3]
    d["topk_idx"][1, 0] = [2, 2, 2]
    G.compare_with_oracle(w, _run(w, d, cap=w.N * w.T * w.R),
                          _oracle(w, d, w.N * w.T * w.R))


def test_pinned_host_x():
    w = W.CONFIGS["dsv3_decode"].replace(T=24)
    d = W.generate(w)
    dd = G.to_dev(d)
    want = G.run_path(w, dd, calls="fused")
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H)
    G.fill_sentinels(buf)
    xh = torch.empty(dd["x"].shape, dtype=dd["x"].dtype, pin_memory=True)
    xh.copy_(dd["x"])
    buf.dispatch(xh, dd["topk_idx"], calls="signalled")
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    n = G.host(want.grp_off)[:, -1]
    for r in range(w.N):
        assert torch.equal(buf.grp_q[r, :n[r]], want.grp_q[r, :n[r]])
        assert torch.equal(buf.grp_src[r, :n[r]], want.grp_src[r, :n[r]])
    assert torch.equal(buf.send_q, want.send_q)


def test_empty_batch():
    buf = m.MoeBuffers(4, 0, 8, 2, 256, cap=1)
    G.fill_sentinels(buf)
    z = torch.zeros(1, dtype=torch.int32, device="cuda")
    buf.dispatch(z, z, calls="signalled")
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    assert np.all(G.host(buf.grp_off) == 0)


def test_unset_flag_times_out_and_scratch_recovers():
    """Group counters that do not start at zero mean no group ever reaches
    its size, so no flag is set: every receiving warp gives up after its
    bounded wait, MOE_ST_TIMEOUT is raised, the call returns, and the kernel
    still clears the scratch, so the next call is exact again."""
    w = W.Workload("timeout", N=2, T=8, H=256, E=4, R=2, seed=23)
    d = W.generate(w)
    dd = G.to_dev(d)
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H)
    G.fill_sentinels(buf)
    buf.sig[: w.N * w.N] = 1 << 30  # counters far past any group's size
    buf.dispatch(dd["x"], dd["topk_idx"], calls="signalled")
    torch.cuda.synchronize()
    assert int(buf.status.item()) & m.MOE_ST_TIMEOUT
    assert int(buf.sig.abs().sum().item()) == 0
    G.fill_sentinels(buf)
    buf.dispatch(dd["x"], dd["topk_idx"], calls="signalled")
    buf.expert(0)
    buf.combine(dd["topk_idx"], dd["topk_w"])
    torch.cuda.synchronize()
    G.compare_with_oracle(w, buf, _oracle(w, d, w.default_cap))


def test_repeat_and_graph_replay_are_identical():
    """Repeated calls and a CUDA-graph replay give the same bytes (the
    scratch is reset by every call, so replays need no extra node)."""
    w = W.CONFIGS["dsv3_decode"].replace(T=32)
    d = W.generate(w)
    dd = G.to_dev(d)
    want = G.run_path(w, dd, calls="fused")
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H)
    buf.dispatch(dd["x"], dd["topk_idx"], calls="signalled")
    torch.cuda.synchronize()
    buf.grp_q.zero_()
    buf.send_q.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        buf.dispatch(dd["x"], dd["topk_idx"], calls="signalled")
    for _ in range(3):
        g.replay()
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    assert int(buf.sig.abs().sum().item()) == 0
    n = G.host(want.grp_off)[:, -1]
    for r in range(w.N):
        assert torch.equal(buf.grp_q[r, :n[r]], want.grp_q[r, :n[r]])
        assert torch.equal(buf.grp_s[r, :n[r]], want.grp_s[r, :n[r]])
    assert torch.equal(buf.send_q, want.send_q)
