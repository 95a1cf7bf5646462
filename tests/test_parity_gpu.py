"""GPU parity: the CUDA path through the C ABI against the CPU oracle.

Bit-exact for counts, offsets, slots, packed and grouped layouts, fp8 bytes,
scales and metadata; the combine is graded at one bf16 step
(|gpu - oracle| <= 2^-7 |oracle| + 1e-6) and, since both sides run the same
fused multiply-adds in the same slot order, also checked bit for bit.
"""
from __future__ import annotations

import itertools

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


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "kimi_k2_decode", "qwen3_skew",
                                  "qwen3_zipf0", "qwen3_zipf1.5"])
def test_config_full_parity(name):
    """Every output of the path at the config's full size, default capacity
    on the GPU (the benchmark's launch), exact-fit capacity in the oracle."""
    w = W.CONFIGS[name]
    d = W.generate(w)
    buf = G.run_path(w, G.to_dev(d))
    o = _oracle(w, d, _exact_cap(w, d))
    G.compare_with_oracle(w, buf, o)


@pytest.mark.parametrize("calls", ["separate", "fused_route"])
@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "kimi_k2_decode", "qwen3_skew"])
def test_other_call_forms(name, calls):
    """The per-step calls (moe_route_count, moe_exchange, moe_dispatch_send,
    moe_dispatch_recv, moe_combine_send, moe_combine_recv), and the same with
    moe_route, give the oracle's outputs like the fused calls."""
    w = W.CONFIGS[name]
    d = W.generate(w)
    buf = G.run_path(w, G.to_dev(d), calls=calls)
    G.compare_with_oracle(w, buf, _oracle(w, d, _exact_cap(w, d)))


@pytest.mark.parametrize("H", [128, 640, 8192 + 1024, 20480])
def test_fused_and_separate_identical_across_row_pieces(H):
    """Rows longer than one shared-memory piece (8192 elements), and scale
    rows that are not whole 16-byte vectors (H/128 not a multiple of 4), give
    the oracle's outputs in both call forms."""
    w = W.Workload("pieces", N=2, T=3, H=H, E=4, R=2, seed=H)
    d = W.generate(w)
    o = _oracle(w, d, w.default_cap)
    for calls in ("fused", "separate"):
        G.compare_with_oracle(w, G.run_path(w, G.to_dev(d), calls=calls), o)


@pytest.mark.parametrize("T", [24, 128])
@pytest.mark.parametrize("calls", ["fused", "separate"])
def test_pinned_host_x_and_out(calls, T):
    """x read from, and out written to, pinned host memory by the kernels give
    the same bytes as device buffers (at 128 tokens per rank the fused
    dispatch's CTAs take more pieces than the ones they copy from host
    memory while the routing kernel runs)."""
    w = W.CONFIGS["dsv3_decode"].replace(T=T)
    d = W.generate(w)
    dd = G.to_dev(d)
    ref_buf = G.run_path(w, dd, calls=calls)
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H)
    G.fill_sentinels(buf)
    xh = torch.empty(dd["x"].shape, dtype=dd["x"].dtype, pin_memory=True)
    xh.copy_(dd["x"])
    oh = torch.empty(buf.out.shape, dtype=buf.out.dtype, pin_memory=True)
    buf.dispatch(xh, dd["topk_idx"], calls=calls)
    buf.expert(1)
    buf.combine(dd["topk_idx"], dd["topk_w"], out=oh, calls=calls)
    torch.cuda.synchronize()
    assert torch.equal(oh.view(torch.int16), ref_buf.out.cpu().view(torch.int16))
    n = G.host(ref_buf.grp_off)[:, -1]
    for r in range(w.N):
        assert torch.equal(buf.grp_q[r, :n[r]], ref_buf.grp_q[r, :n[r]])
    assert int(buf.status.item()) == 0


@pytest.mark.slow
@pytest.mark.parametrize("name", ["prefill", "qwen3_worst"])
def test_config_full_size_every_element(name):
    """The two largest workloads at their configured sizes (prefill: 8 ranks
    x 4096 tokens; the worst case: 16 ranks x 512 tokens all routed to rank
    0's experts, the receive bound of the EFA page's "Send and receive
    buffers"), in the launch the benchmark times (default capacity), every
    output element against the oracle, compared rank by rank."""
    w = W.CONFIGS[name]
    d = W.generate(w)
    buf = G.run_path(w, G.to_dev(d))
    o = _oracle(w, d, _exact_cap(w, d))
    G.compare_with_oracle_by_rank(w, buf, o)
    if name == "qwen3_worst":
        recv = G.host(buf.grp_off)[:, -1]
        assert recv[0] == w.N * w.T * min(w.R, w.Er) and np.all(recv[1:] == 0)


def test_worst_case_reduced_t_full_parity():
    """All tokens routed to rank 0's experts, compared in full."""
    w = W.CONFIGS["qwen3_worst"].replace(T=64)
    d = W.generate(w)
    buf = G.run_path(w, G.to_dev(d))
    o = _oracle(w, d, w.default_cap)
    G.compare_with_oracle(w, buf, o)
    recv = G.host(buf.grp_off)[:, -1]
    assert recv[0] == w.N * w.T * min(w.R, w.Er) and np.all(recv[1:] == 0)


def _sampled_check(w, d, buf, ntok=48, seed=0):
    """Full-size check on sampled tokens: integer layouts in full, payload,
    grouped rows, expert outputs, combine rows and outputs token by token."""
    rc = ref.route_count(w.N, w.T, w.E, w.R, d["topk_idx"])
    ex = ref.exchange(w.N, w.E, buf.cap, rc["expert_count"], rc["send_off"])
    for k in ("expert_count", "send_off", "expert_send_off", "slot_row"):
        G.assert_eq(k, G.host(getattr(buf, k)), rc[k])
    for k in ("grp_off", "seg_off", "csend_off", "m_sizes"):
        G.assert_eq(k, G.host(getattr(buf, k)), ex[k])
    assert int(buf.status.item()) == (rc["status"] | ex["status"])
    mode = 1 if w.expert == "scale" else 0
    rng = np.random.default_rng(seed)
    Er = w.Er
    for flat in rng.choice(w.N * w.T, ntok, replace=False):
        s, t = divmod(int(flat), w.T)
        q, sc = ref.quant_token(w.H, d["x"][s, t])
        rows, use = [], []
        for k in range(w.R):
            e = int(d["topk_idx"][s, t, k])
            slot = int(rc["slot_row"][s, t, k])
            G.assert_eq("send_q", G.host(buf.send_q[s, slot]), q)
            G.assert_eq("send_s", G.host(buf.send_s[s, slot]), sc)
            assert int(buf.send_tok[s, slot]) == t
            r, j = e // Er, e % Er
            g = int(ex["seg_off"][r, j, s]) + slot - int(rc["expert_send_off"][s, e])
            c = int(ex["csend_off"][r, s]) + slot - int(rc["send_off"][s, r])
            G.assert_eq("grp_q", G.host(buf.grp_q[r, g]), q)
            G.assert_eq("grp_s", G.host(buf.grp_s[r, g]), sc)
            assert tuple(G.host(buf.grp_src[r, g])) == (s, t)
            yr = ref.standin_row(w.H, mode, e, q, sc)
            G.assert_eq("y", G.host(buf.y[r, g]), yr)
            G.assert_eq("csend", G.host(buf.csend[r, c]), yr)
            rows.append(yr)
            use.append(1)
        want = ref.weighted_sum(np.stack(rows), d["topk_w"][s, t], np.array(use, np.int32))
        G.assert_eq("out", G.host(buf.out[s, t]), want)


@pytest.mark.parametrize("name", ["prefill", "qwen3_worst"])
def test_config_full_size_sampled(name):
    w = W.CONFIGS[name]
    d = W.generate(w)
    buf = G.run_path(w, G.to_dev(d), sentinels=False)
    _sampled_check(w, d, buf)


def _grid():
    cases = []
    for N, Er, T, H in itertools.product([1, 2, 3, 4], [1, 2, 4], [1, 5, 16], [128, 256, 384]):
        E = N * Er
        for R in range(1, min(E, 4) + 1):
            cases.append((N, T, E, R, H))
    return cases


@pytest.mark.parametrize("N,T,E,R,H", _grid())
def test_small_shape_grid(N, T, E, R, H):
    w = W.Workload("grid", N=N, T=T, H=H, E=E, R=R, seed=7 + N * 1000 + T * 100 + E * 10 + R)
    d = W.generate(w)
    o = _oracle(w, d, w.default_cap)
    for calls in ("fused", "separate", "fused_route"):
        buf = G.run_path(w, G.to_dev(d), calls=calls)
        G.compare_with_oracle(w, buf, o)


def test_empty_batch():
    w = W.Workload("empty", N=4, T=0, H=256, E=8, R=2)
    d = {"x": np.zeros((4, 0, 256), np.uint16), "topk_idx": np.zeros((4, 0, 2), np.int32),
         "topk_w": np.zeros((4, 0, 2), np.float32)}
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, cap=1)
    G.fill_sentinels(buf)
    dd = {"x": torch.zeros(1, dtype=torch.int16, device="cuda"),
          "topk_idx": torch.zeros(1, dtype=torch.int32, device="cuda"),
          "topk_w": torch.zeros(1, dtype=torch.float32, device="cuda")}
    buf.dispatch(dd["x"], dd["topk_idx"])
    buf.expert(0)
    buf.combine(dd["topk_idx"], dd["topk_w"])
    torch.cuda.synchronize()
    assert int(buf.status.item()) == 0
    o = ref.route_count(4, 0, 8, 2, d["topk_idx"])
    G.assert_eq("expert_count", G.host(buf.expert_count), o["expert_count"])
    G.assert_eq("send_off", G.host(buf.send_off), o["send_off"])
    assert np.all(G.host(buf.grp_off) == 0) and np.all(G.host(buf.csend_off) == 0)


@pytest.mark.parametrize("calls", ["fused", "separate", "fused_route"])
def test_bad_expert_ids_are_skipped_and_flagged(calls):
    w = W.Workload("bad", N=2, T=8, H=256, E=8, R=2, seed=3)
    d = W.generate(w)
    d["topk_idx"][0, 1, 1] = -1
    d["topk_idx"][1, 5, 0] = 8
    d["topk_idx"][1, 6, 1] = 1 << 30
    buf = G.run_path(w, G.to_dev(d), calls=calls)
    o = _oracle(w, d, w.default_cap)
    assert o["status"] == ref.ST_BAD_EXPERT
    G.compare_with_oracle(w, buf, o)
    assert G.host(buf.slot_row)[0, 1, 1] == -1


@pytest.mark.parametrize("E", [1, 7, 8, 64, 255, 256, 1023, 1024])
@pytest.mark.parametrize("calls", ["fused", "separate"])
def test_ranking_keys_at_bit_boundaries(E, calls):
    """The routing kernels find equal ids with one warp ballot per bit of a
    key (expert id, or E for an id outside [0, E)): expert counts just below
    and at a power of two, bad ids of every kind, and whole warps of one
    expert give the oracle's counts, slots and layouts."""
    R = min(3, E)
    w = W.Workload("keys", N=1, T=96, H=128, E=E, R=R, seed=E)
    d = W.generate(w)
    ids = d["topk_idx"]
    ids[0, 0:11, 0] = E - 1              # a run of the highest expert
    ids[0, 40:72, :] = 0                 # whole warps of expert 0 (repeated slots)
    for t, v in ((3, -1), (17, E), (29, E + 1), (50, 2 * E), (77, 1 << 30), (90, -(1 << 30))):
        ids[0, t, R - 1] = v
    o = _oracle(w, d, w.N * w.T * w.R)
    assert o["status"] == ref.ST_BAD_EXPERT
    buf = G.run_path(w, G.to_dev(d), cap=w.N * w.T * w.R, calls=calls)
    G.compare_with_oracle(w, buf, o)


@pytest.mark.parametrize("cap", [1, 7, 20])
@pytest.mark.parametrize("calls", ["fused", "separate", "fused_route"])
def test_capacity_overflow_drops_and_flags(cap, calls):
    w = W.Workload("cap", N=2, T=16, H=256, E=4, R=2, seed=11)
    d = W.generate(w)
    buf = G.run_path(w, G.to_dev(d), cap=cap, calls=calls)
    o = _oracle(w, d, cap)
    assert o["status"] & ref.ST_CAPACITY
    G.compare_with_oracle(w, buf, o)


def test_duplicate_experts_in_a_token():
    w = W.Workload("dup", N=2, T=6, H=128, E=4, R=3, seed=5)
    d = W.generate(w)
    d["topk_idx"][0, 2] = [1, 1, 3]
    d["topk_idx"][1, 0] = [2, 2, 2]
    buf = G.run_path(w, G.to_dev(d), cap=w.N * w.T * w.R)
    G.compare_with_oracle(w, buf, _oracle(w, d, w.N * w.T * w.R))


def test_zero_blocks_and_signed_zero():
    w = W.Workload("zeros", N=2, T=4, H=384, E=4, R=2, seed=13)
    d = W.generate(w)
    d["x"][0, 0, :] = 0                # whole token zero
    d["x"][0, 1, 128:256] = 0x8000     # one block of -0
    d["x"][1, 2, 5] = 0x8000           # a -0 inside a non-zero block
    d["x"][1, 3, :128] = 0x0001        # smallest bf16 subnormal everywhere
    buf = G.run_path(w, G.to_dev(d))
    G.compare_with_oracle(w, buf, _oracle(w, d, w.default_cap))


def test_repeat_and_graph_replay_are_identical():
    """Two eager runs and a CUDA-graph replay of the six calls agree bit for
    bit (no state survives between calls; the sequence captures)."""
    w = W.CONFIGS["tiny"].replace(T=64, H=512)
    d = W.generate(w)
    dd = G.to_dev(d)
    b1 = G.run_path(w, dd)
    b2 = G.run_path(w, dd)
    for k in ("slot_row", "grp_q", "grp_s", "csend", "out"):
        assert torch.equal(getattr(b1, k).view(torch.uint8), getattr(b2, k).view(torch.uint8))
    b3 = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H)
    b3.dispatch(dd["x"], dd["topk_idx"])
    b3.expert(0)
    b3.combine(dd["topk_idx"], dd["topk_w"])
    torch.cuda.synchronize()
    b3.out.zero_()
    b3.grp_q.zero_()
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        b3.dispatch(dd["x"], dd["topk_idx"])
        b3.combine(dd["topk_idx"], dd["topk_w"])
        b3.dispatch(dd["x"], dd["topk_idx"], calls="separate")
        b3.combine(dd["topk_idx"], dd["topk_w"], calls="separate")
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(b3.out, b1.out)
    n = G.host(b1.grp_off)[:, -1]
    for r in range(w.N):
        assert torch.equal(b3.grp_q[r, :n[r]], b1.grp_q[r, :n[r]])


@pytest.mark.slow
def test_e4m3_encoder_matches_oracle_exhaustively():
    """The GPU conversion (the quantiser's) equals the oracle's encoder for
    every fp32 bit pattern with |v| <= 480, both signs."""
    import concurrent.futures as cf
    top = int(np.float32(480.0).view(np.uint32))
    chunk = 1 << 25
    dev_in = torch.empty(chunk, dtype=torch.int32, device="cuda")
    dev_out = torch.empty(chunk, dtype=torch.uint8, device="cuda")
    pool = cf.ThreadPoolExecutor(8)

    def ora(v):
        parts = np.array_split(v, 8)
        return np.concatenate(list(pool.map(ref.e4m3_encode, parts)))

    for sign in (0, 0x80000000):
        for start in range(0, top + 1, chunk):
            n = min(chunk, top + 1 - start)
            pats = (np.arange(start, start + n, dtype=np.uint64) | sign).astype(np.uint32)
            dev_in[:n].copy_(torch.from_numpy(pats.view(np.int32)))
            m.moe_e4m3_encode(dev_in[:n].view(torch.float32), dev_out[:n])
            got = dev_out[:n].cpu().numpy()
            want = ora(pats.view(np.float32))
            bad = np.nonzero(got != want)[0]
            assert bad.size == 0, (f"{bad.size} mismatches, first pattern "
                                   f"{pats[bad[0]]:#010x}: gpu {got[bad[0]]:#04x} "
                                   f"oracle {want[bad[0]]:#04x}")
    # beyond the range: saturation on both sides
    v = np.array([480.0, 1e4, np.inf, -1e30, -np.inf], np.float32)
    t = torch.from_numpy(v).cuda()
    o = torch.empty(5, dtype=torch.uint8, device="cuda")
    m.moe_e4m3_encode(t, o)
    assert list(o.cpu().numpy()) == list(ref.e4m3_encode(v))


@pytest.mark.parametrize("N,T,E,R,H", [(2, 9, 32, 12, 128), (2, 5, 64, 32, 256),
                                       (3, 4, 24, 9, 384), (4, 6, 32, 32, 256)])
@pytest.mark.parametrize("calls", ["fused", "separate", "fused_route", "signalled"])
def test_many_experts_per_token(N, T, E, R, H, calls):
    """More than eight slots per token (the quantiser stores to every slot's
    rows from registers; the combine's slot table leaves registers), every
    output against the oracle."""
    w = W.Workload("wide", N=N, T=T, H=H, E=E, R=R, seed=1000 + N * 10 + R)
    d = W.generate(w)
    G.compare_with_oracle(w, G.run_path(w, G.to_dev(d), calls=calls),
                          _oracle(w, d, w.default_cap))


@pytest.mark.parametrize("N,T,E,R,H", [(4, 8, 1024, 32, 128), (64, 4, 128, 2, 256),
                                       (1, 1024, 16, 4, 128), (2, 3, 4, 2, 65536),
                                       (20, 256, 40, 8, 128), (16, 300, 32, 8, 128),
                                       (32, 128, 32, 8, 128), (1, 64, 1024, 32, 128),
                                       (32, 1, 1024, 32, 128)])
@pytest.mark.parametrize("calls", ["fused", "separate", "signalled"])
def test_limits(N, T, E, R, H, calls):
    """At the ABI's limits: the most experts (1024, the route's largest
    shared-memory tables) with the most slots (32), 64 ranks (the route
    without a cluster, many blocks), one rank with the longest batch, the
    widest row (65536 elements: many pieces per row, 512 scales); and the
    routing kernel's forms with many ids per rank: 20 and 32 ranks (the
    grid-barrier route) and 16 ranks with 2400 ids each (the cluster
    route); one rank holding all 1024 experts with 32 slots (as many local
    experts as the routing block has threads); one token per rank on 32
    ranks with 1024 experts and 32 slots."""
    w = W.Workload("limits", N=N, T=T, H=H, E=E, R=R, seed=2000 + N + E)
    d = W.generate(w)
    G.compare_with_oracle(w, G.run_path(w, G.to_dev(d), calls=calls),
                          _oracle(w, d, w.default_cap))


def test_dispatch_reads_x_written_just_before():
    """moe_dispatch's quantiser starts loading x while its routing kernel runs
    (programmatic dependent launch). x written by a kernel issued just
    before the call on the same stream, eagerly and inside a CUDA graph, must
    still be the x it reads: the grouped rows match the oracle on the new x."""
    w = W.CONFIGS["dsv3_decode"].replace(T=32)
    d_a = W.generate(w)
    d_b = W.generate(w.replace(seed=w.seed + 99))
    dd_a, dd_b = G.to_dev(d_a), G.to_dev(d_b)
    x = dd_a["x"].clone()
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H)
    idx = dd_a["topk_idx"]
    o_b = ref.layer(w.N, w.T, w.E, w.R, w.H, buf.cap, d_b["x"], d_a["topk_idx"], d_a["topk_w"],
                    mode=1)
    recv = o_b["grp_off"][:, -1]

    def check():
        torch.cuda.synchronize()
        gq, sq = G.host(buf.grp_q), G.host(buf.send_q)
        for r in range(w.N):
            G.assert_eq(f"grp_q[{r}]", gq[r, :recv[r]], o_b["grp_q"][r, :recv[r]])
            n = int(o_b["send_off"][r, -1])
            G.assert_eq(f"send_q[{r}]", sq[r, :n], o_b["send_q"][r, :n])
        assert int(buf.status.item()) == 0

    buf.dispatch(x, idx)             # x = A
    x.copy_(dd_b["x"])               # a kernel writes x = B ...
    buf.dispatch(x, idx)             # ... and the next call must see it
    check()
    # the same inside a graph: the copy node right before the dispatch nodes
    s = torch.cuda.Stream()
    g = torch.cuda.CUDAGraph()
    x.copy_(dd_a["x"])
    torch.cuda.synchronize()
    with torch.cuda.graph(g, stream=s):
        x.copy_(dd_b["x"])
        buf.dispatch(x, idx)
    buf.grp_q.zero_()
    buf.send_q.zero_()
    x.copy_(dd_a["x"])
    torch.cuda.synchronize()
    g.replay()
    check()
