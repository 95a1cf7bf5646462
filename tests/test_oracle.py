"""Pins of the CPU oracle to things other than itself (no GPU needed).

What pins each oracle function:
  ref_e4m3_decode    page-independent facts of the OCP E4M3 format (named
                     codes), monotonicity and spacing, and torch's own
                     float8_e4m3fn decoding of all 256 codes.
  ref_e4m3_encode    torch's float8_e4m3fn cast (an independent library
                     encoder, RNE) on a dense sweep below 464, plus a brute
                     force nearest-code search with ties to even; satfinite
                     above.
  ref_f32_to_bf16_rn torch's bfloat16 cast on a dense sweep.
  ref_quant_token    closed forms: the amax element encodes to +-448, every
                     element is within half an e4m3 step of x/scale, zero
                     blocks give zero bytes and scale 0.
  ref_route_count    invariants (counts sum to T*R, exclusive-scan identity,
                     slot_row a permutation, send_off nested in
                     expert_send_off) and brute force by sorting.
  ref_exchange       brute force by sorting, receive bound N*T*max(R,E/N)
                     from the pages, worst case reaching N*T*min(R,E/N).
  ref_dispatch_send/recv, ref_combine_send/recv
                     brute-force positions (grp_src, tagged combine rows) on
                     every routing of tiny shapes; round trip through the
                     identity expert with weights summing to 1.
  ref_weighted_sum   exact rational sum: result within one bf16 step; every
                     element equal, bit for bit, to a chain of fused
                     multiply-adds in ascending slot order rounded by an
                     exact-fraction fp32 rounder; hand cases where descending
                     or pairwise order, or a separate multiply and add, give
                     other bits.
  ref_standin_row    exact product in fractions, rounded by torch's bf16 cast.
  ref_expert_standin / ref_standin_ll (per-expert scale)
                     every grouped and low-latency row equals the stand-in of
                     the expert its brute-force position says it belongs to
                     (expert id from topk_idx), computed with numpy products
                     and torch's bf16 cast.
  ref_combine_partial_send / _recv (send-side reduction)
                     exact rational sums on every routing of a tiny shape
                     and on random shapes with duplicates, bad ids and drops;
                     hand cases fixing where the per-group rounding happens
                     and the ascending-rank order of the final sum; one
                     expert per rank reduces to torch's rounded products; the
                     two-rounding error bound against the exact sum.
"""
from __future__ import annotations

import itertools
from fractions import Fraction

import numpy as np
import pytest
import torch

from combine_expert_count_gb300 import workloads as W
from oracle import brute, ref

# ----------------------------------------------------------------- e4m3 / bf16


def test_e4m3_named_codes():
    d = ref.e4m3_decode(np.arange(256, dtype=np.uint8))
    assert d[0x00] == 0.0 and not np.signbit(d[0x00])
    assert d[0x80] == 0.0 and np.signbit(d[0x80])
    assert d[0x01] == 2.0 ** -9          # smallest subnormal
    assert d[0x07] == 7 * 2.0 ** -9      # largest subnormal
    assert d[0x08] == 2.0 ** -6          # smallest normal
    assert d[0x38] == 1.0
    assert d[0x7E] == 448.0              # largest finite
    assert d[0xFE] == -448.0
    assert np.isnan(d[0x7F]) and np.isnan(d[0xFF])
    assert np.isnan(d).sum() == 2        # no infinities, two NaN codes


def test_e4m3_decode_monotone_and_spaced():
    d = ref.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    assert np.all(np.diff(d) > 0)
    # 8 equal steps per binade above the subnormals
    for ef in range(1, 16):
        codes = [ef * 8 + m for m in range(8) if ef * 8 + m < 0x7F]
        steps = np.diff(d[codes])
        assert np.all(steps == 2.0 ** (ef - 7 - 3))
    # negative codes mirror positive ones
    dn = ref.e4m3_decode(np.arange(0x80, 0xFF, dtype=np.uint8))
    assert np.array_equal(dn, -d)


def test_e4m3_decode_matches_torch():
    codes = torch.arange(256, dtype=torch.uint8)
    t = codes.view(torch.float8_e4m3fn).double().numpy()
    d = ref.e4m3_decode(codes.numpy())
    fin = ~np.isnan(t)
    assert np.array_equal(np.isnan(d), np.isnan(t))
    assert np.array_equal(d[fin], t[fin])


def _sweep_below_464(stride: int = 97) -> np.ndarray:
    """fp32 values with |v| < 464: a strided walk over bit patterns plus every
    e4m3 midpoint and its fp32 neighbours."""
    top = np.float32(464.0).view(np.uint32)
    pats = np.arange(0, int(top), stride, dtype=np.uint32)
    v = pats.view(np.float32)
    d = ref.e4m3_decode(np.arange(0x7F, dtype=np.uint8))
    mids = ((d[:-1] + d[1:]) / 2).astype(np.float32)
    near = np.concatenate([mids, np.nextafter(mids, np.float32(0)), np.nextafter(mids, np.float32(1e9))])
    v = np.concatenate([v, near, d.astype(np.float32)])
    return np.concatenate([v, -v])


def test_e4m3_encode_matches_torch_rne():
    v = _sweep_below_464()
    ours = ref.e4m3_encode(v)
    theirs = torch.from_numpy(v).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = np.nonzero(ours != theirs)[0]
    assert bad.size == 0, f"{bad.size} mismatches, first v={v[bad[0]]!r}"


def test_e4m3_encode_nearest_code_bruteforce():
    rng = np.random.default_rng(5)
    v = np.concatenate([
        rng.uniform(-448, 448, 4000),
        rng.uniform(-0.02, 0.02, 4000),
        np.ldexp(rng.uniform(-1, 1, 4000), rng.integers(-12, 9, 4000)),
    ]).astype(np.float32)
    codes = np.arange(0x7F, dtype=np.uint8)          # finite non-negative codes
    vals = ref.e4m3_decode(codes)
    got = ref.e4m3_encode(v)
    for x, c in zip(v.tolist(), got.tolist()):
        a = abs(Fraction(x))
        dist = [abs(Fraction(float(q)) - a) for q in vals]
        best = min(dist)
        cands = [i for i, dd in enumerate(dist) if dd == best]
        want = cands[0] if len(cands) == 1 else [i for i in cands if i % 2 == 0][0]
        want |= 0x80 if np.signbit(np.float32(x)) else 0
        assert c == want, (x, c, want)


def test_e4m3_satfinite_and_nan():
    v = np.array([448.0, 463.99, 464.0, 1e6, np.inf, -1e6, -np.inf], np.float32)
    assert list(ref.e4m3_encode(v)) == [0x7E] * 5 + [0xFE] * 2
    assert ref.e4m3_encode(np.array([np.nan], np.float32))[0] & 0x7F == 0x7F


def test_bf16_rn_matches_torch():
    rng = np.random.default_rng(11)
    pats = np.concatenate([
        rng.integers(0, 2 ** 32, 200000, dtype=np.uint64).astype(np.uint32),
        # exact ties and their neighbours
        (rng.integers(0, 2 ** 16, 20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8000,
        (rng.integers(0, 2 ** 16, 20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x7FFF,
        (rng.integers(0, 2 ** 16, 20000, dtype=np.uint64).astype(np.uint32) << 16) | 0x8001,
    ])
    v = pats.view(np.float32)
    v = v[~np.isnan(v)]
    theirs = torch.from_numpy(v.copy()).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(ref.f32_to_bf16_array(v), theirs)
    ours = np.array([ref.f32_to_bf16(float(x)) for x in v[::97]], np.uint16)
    assert np.array_equal(ours, theirs[::97])


# ----------------------------------------------------------------- quantisation


def _bf16(x: np.ndarray) -> np.ndarray:
    return W.bf16_bits(np.asarray(x, np.float32))


def _f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def test_quant_closed_forms():
    rng = np.random.default_rng(3)
    H = 1024
    for trial in range(20):
        x = _bf16(rng.standard_normal(H) * np.exp(rng.uniform(-30, 30)))
        q, sc = ref.quant_token(H, x)
        xf = _f32(x).reshape(-1, 128).astype(np.float64)
        amax = np.abs(xf).max(axis=1)
        # scale = amax / 448 in fp32
        assert np.array_equal(sc, (amax.astype(np.float32) / np.float32(448.0)).astype(np.float32))
        # the bytes are torch's RNE e4m3 cast of the fp32 quotient x / scale
        xs = (_f32(x).reshape(-1, 128) / sc[:, None]).astype(np.float32)
        lib_q = torch.from_numpy(xs.ravel()).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        assert np.array_equal(q, lib_q)
        dq = ref.e4m3_decode(q).reshape(-1, 128)
        for b in range(H // 128):
            i = int(np.argmax(np.abs(xf[b])))
            assert abs(dq[b, i]) == 448.0 and np.sign(dq[b, i]) == np.sign(xf[b, i])
            v = xf[b] / np.float64(sc[b])
            # half an e4m3 step: 2^-10 below 2^-6, else 2^-4 relative
            bound = np.maximum(2.0 ** -10, np.abs(v) * 2.0 ** -4) * (1 + 1e-6)
            assert np.all(np.abs(v - dq[b]) <= bound)


def test_quant_zero_block_and_signed_zero():
    H = 256
    x = np.zeros(H, np.float32)
    x[128] = -0.0
    x[129] = 3.0
    x[130] = -0.0
    xb = _bf16(x)
    xb[0] = 0x8000  # -0 in an all-zero block
    q, sc = ref.quant_token(H, xb)
    assert sc[0] == 0.0 and np.all(q[:128] == 0)
    assert q[129] == 0x7E and q[128] == 0x80 and q[130] == 0x80 and q[131] == 0x00


# ----------------------------------------------------------------- layouts


def _check_route_invariants(N, T, E, R, idx, rc):
    Er = E // N
    cnt, so, eso, slot = rc["expert_count"], rc["send_off"], rc["expert_send_off"], rc["slot_row"]
    idx = idx.reshape(N, T, R)
    for s in range(N):
        valid = (idx[s] >= 0) & (idx[s] < E)
        assert np.array_equal(cnt[s], np.bincount(idx[s][valid], minlength=E))
        assert eso[s, 0] == 0 and np.array_equal(np.diff(eso[s]), cnt[s])
        assert so[s, 0] == 0 and np.array_equal(np.diff(so[s]), cnt[s].reshape(N, Er).sum(1))
        assert np.array_equal(so[s], eso[s, ::Er])       # peers nest inside experts
        sl = slot[s][valid]
        assert np.array_equal(np.sort(sl), np.arange(valid.sum()))
        assert np.all(slot[s][~valid] == -1)


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "kimi_k2_decode", "qwen3_skew",
                                  "qwen3_worst"])
def test_route_and_exchange_invariants(name):
    w = W.CONFIGS[name]
    d = W.generate(w, with_x=False)
    rc = ref.route_count(w.N, w.T, w.E, w.R, d["topk_idx"])
    assert rc["status"] == 0
    assert np.all(rc["expert_count"].sum(1) == w.T * w.R)
    _check_route_invariants(w.N, w.T, w.E, w.R, d["topk_idx"], rc)
    ex = ref.exchange(w.N, w.E, w.default_cap, rc["expert_count"], rc["send_off"])
    recv = ex["grp_off"][:, -1]
    assert recv.sum() == w.A
    assert np.all(recv <= w.N * w.T * max(w.R, w.Er))              # the pages' bound
    assert np.all(np.diff(ex["grp_off"], axis=1) == ex["m_sizes"])
    assert np.array_equal(ex["csend_off"][:, -1], recv)
    if w.routing == "worst":
        assert recv[0] == w.N * w.T * min(w.R, w.Er) and np.all(recv[1:] == 0)


def test_receive_bound_from_page(golden):
    """The pages' bound N*T*max(R,E/N) holds for every routing of small shapes,
    and all-to-one routing reaches N*T*min(R,E/N)."""
    assert golden["receive_bound"]["formula"] == "N*T*max(R,E/N)"
    for N, T, E, R in [(2, 3, 4, 2), (2, 2, 8, 3), (4, 2, 4, 2), (3, 2, 6, 1)]:
        Er = E // N
        rng = np.random.default_rng(N * 100 + E)
        worst = 0
        for _ in range(200):
            idx = np.stack([rng.permutation(E)[:R] for _ in range(N * T)]).astype(np.int32)
            rc = ref.route_count(N, T, E, R, idx)
            ex = ref.exchange(N, E, N * T * R, rc["expert_count"], rc["send_off"])
            worst = max(worst, int(ex["grp_off"][:, -1].max()))
        idx = np.tile(np.arange(min(R, Er), dtype=np.int32), (N * T, 1))
        if min(R, Er) < R:
            # R > E/N: a token can put at most E/N copies on one rank
            idx = np.concatenate([idx, np.tile(np.arange(Er, Er + R - Er, dtype=np.int32),
                                                (N * T, 1))], axis=1)
        rc = ref.route_count(N, T, E, R, idx)
        ex = ref.exchange(N, E, N * T * R, rc["expert_count"], rc["send_off"])
        assert ex["grp_off"][0, -1] == N * T * min(R, Er)
        assert worst <= N * T * max(R, Er)


def test_page_copy_counts(golden):
    """Each GPU sends T*R token copies (2K tokens x top-8 = 16K), one row per
    (token, expert) assignment, over E/N = 32 experts per GPU."""
    g = golden["prefill_ep8"]
    w = W.Workload("ep8", N=g["N"], T=g["T"], H=128, E=g["E"], R=g["R"], seed=99)
    d = W.generate(w, with_x=False)
    rc = ref.route_count(w.N, w.T, w.E, w.R, d["topk_idx"])
    assert np.all(rc["send_off"][:, -1] == g["copies_per_rank"])
    assert w.Er == g["experts_per_rank"]
    assert W.CONFIGS["dsv3_decode"].Er == golden["decode_ep16"]["experts_per_rank"]
    assert W.CONFIGS["dsv3_decode"].T == golden["decode_ep16"]["max_dispatch_tokens_per_rank"]


def test_page_transfers_per_pe(golden):
    """Qwen3-30B on 16 PEs: each sender's layout has E/P = 8 expert runs per
    peer; toward the 12 off-node PEs that is 96 runs."""
    g = golden["qwen3_transfers"]
    w = W.CONFIGS["qwen3_skew"]
    assert (w.N, w.E) == (g["PEs"], g["E"]) and w.Er == g["experts_per_pe"]
    d = W.generate(w, with_x=False)
    rc = ref.route_count(w.N, w.T, w.E, w.R, d["topk_idx"])
    eso, so = rc["expert_send_off"], rc["send_off"]
    for s in range(w.N):
        node = s // g["gpus_per_node"]
        remote = [p for p in range(w.N) if p // g["gpus_per_node"] != node]
        assert len(remote) == g["remote_pes"]
        runs = 0
        for p in remote:
            # runs of peer p are exactly experts p*Er .. p*Er+Er-1 and tile send_off[p]..[p+1]
            starts = eso[s, p * w.Er:(p + 1) * w.Er + 1]
            assert starts[0] == so[s, p] and starts[-1] == so[s, p + 1]
            runs += len(starts) - 1
        assert runs == g["transfers_per_pe"]


def test_zipf_share_from_page(golden):
    g = golden["zipf_skew"]
    p = W.zipf_popularity(g["E"], g["s"])
    assert abs(np.sort(p)[::-1][: g["top"]].sum() - g["share"]) < 0.005
    assert np.allclose(W.zipf_popularity(g["E"], 0.0), 1.0 / g["E"])


def test_skew_recipe_share():
    w = W.CONFIGS["qwen3_skew"]
    d = W.generate(w, with_x=False)
    share = np.isin(d["topk_idx"], W.hot_experts(w.E, w.seed)).mean()
    assert abs(share - 0.5) < 0.03, share


def _layout_vs_brute(N, T, E, R, idx):
    Er = E // N
    rc = ref.route_count(N, T, E, R, idx)
    ex = ref.exchange(N, E, N * T * R, rc["expert_count"], rc["send_off"])
    send_row, grp_row, csend_row = brute.layouts(N, T, E, R, idx)
    slot, eso, so = rc["slot_row"], rc["expert_send_off"], rc["send_off"]
    for (s, t, k), pos in send_row.items():
        e = int(idx.reshape(N, T, R)[s, t, k])
        r, j = e // Er, e % Er
        assert slot[s, t, k] == pos
        assert ex["seg_off"][r, j, s] + (pos - eso[s, e]) == grp_row[(s, t, k)]
        assert ex["csend_off"][r, s] + (pos - so[s, r]) == csend_row[(s, t, k)]
    return rc, ex


def test_layouts_bruteforce_all_routings_2x2x4x2():
    n = 0
    for idx in brute.all_routings(2, 2, 4, 2):
        _layout_vs_brute(2, 2, 4, 2, idx)
        n += 1
    assert n == 12 ** 4


@pytest.mark.parametrize("R", [1, 2])
def test_layouts_bruteforce_all_routings_3x1x3(R):
    for idx in brute.all_routings(3, 1, 3, R):
        _layout_vs_brute(3, 1, 3, R, idx)


def _tiny_x(N, T, H, seed):
    rng = np.random.default_rng(seed)
    return _bf16(rng.standard_normal((N, T, H)))


def _full_path_vs_brute(N, T, E, R, H, idx, x, cap=None):
    """Run every oracle step and check positions against brute force; the
    combine is checked with tagged rows and one-hot weights.  With a small
    ``cap``, an assignment whose grouped or combine row is at or beyond cap is
    dropped and contributes zero."""
    Er = E // N
    cap = N * T * R if cap is None else cap
    rc = ref.route_count(N, T, E, R, idx)
    ex = ref.exchange(N, E, cap, rc["expert_count"], rc["send_off"])
    ds = ref.dispatch_send(N, T, R, H, x, rc["slot_row"])
    dr = ref.dispatch_recv(N, T, E, R, H, cap, ds["send_q"], ds["send_s"], ds["send_tok"],
                           rc["expert_count"], rc["expert_send_off"], ex["seg_off"])
    send_row, grp_row, csend_row = brute.layouts(N, T, E, R, idx)
    recv = np.bincount([int(e) // Er for e in idx.ravel()], minlength=N)
    assert ex["status"] == (ref.ST_CAPACITY if recv.max() > cap else 0)
    idx3 = idx.reshape(N, T, R)
    y = np.zeros((N, cap, H), np.uint16)
    tags = {}
    for (s, t, k), g in grp_row.items():
        r = int(idx3[s, t, k]) // Er
        tag = float(1 + s * 64 + t * 4 + k)   # exact in bf16 for these sizes
        tags[(s, t, k)] = tag
        if g >= cap:
            continue
        q, sc = ref.quant_token(H, x[s, t])
        assert np.array_equal(dr["grp_q"][r, g], q)
        assert np.array_equal(dr["grp_s"][r, g], sc)
        assert tuple(dr["grp_src"][r, g]) == (s, t)
        y[r, g] = _bf16(np.full(H, tag))
    csend = ref.combine_send(N, T, E, R, H, cap, y, rc["expert_count"], rc["expert_send_off"],
                             rc["send_off"], ex["seg_off"], ex["csend_off"])
    for (s, t, k), c in csend_row.items():
        r = int(idx3[s, t, k]) // Er
        if c < cap:
            want = tags[(s, t, k)] if grp_row[(s, t, k)] < cap else 0.0
            assert np.all(_f32(csend[r, c]) == want)
    for k in range(R):
        w = np.zeros((N, T, R), np.float32)
        w[:, :, k] = 1.0
        out = ref.combine_recv(N, T, E, R, H, cap, csend, idx, w, rc["slot_row"], rc["send_off"],
                               ex["csend_off"])
        for s, t in itertools.product(range(N), range(T)):
            kept = grp_row[(s, t, k)] < cap and csend_row[(s, t, k)] < cap
            assert _f32(out[s, t, :1])[0] == (tags[(s, t, k)] if kept else 0.0)


def test_full_path_bruteforce_sampled_2x2x4x2():
    rng = np.random.default_rng(1)
    x = _tiny_x(2, 2, 128, 2)
    allr = list(brute.all_routings(2, 2, 4, 2))
    for i in rng.choice(len(allr), 300, replace=False):
        _full_path_vs_brute(2, 2, 4, 2, 128, allr[i], x)


def test_full_path_capacity_drops():
    rng = np.random.default_rng(21)
    x = _tiny_x(2, 3, 128, 5)
    for cap in (1, 2, 3, 5):
        for _ in range(40):
            idx = np.stack([rng.permutation(4)[:2] for _ in range(6)]).astype(np.int32)
            _full_path_vs_brute(2, 3, 4, 2, 128, idx.reshape(2, 3, 2), x, cap=cap)


@pytest.mark.parametrize("R", [1, 2])
def test_full_path_bruteforce_all_3x1x3(R):
    x = _tiny_x(3, 1, 128, 4)
    for idx in brute.all_routings(3, 1, 3, R):
        _full_path_vs_brute(3, 1, 3, R, 128, idx, x)


def test_bad_expert_and_capacity_flags():
    N, T, E, R, H = 2, 4, 4, 2, 128
    idx = np.array([[[0, 1], [2, -1], [9, 3], [1, 0]],
                    [[3, 2], [0, 1], [1, 2], [3, 0]]], np.int32)
    rc = ref.route_count(N, T, E, R, idx)
    assert rc["status"] == ref.ST_BAD_EXPERT
    assert rc["slot_row"][0, 1, 1] == -1 and rc["slot_row"][0, 2, 0] == -1
    assert rc["send_off"][0, -1] == T * R - 2
    ex = ref.exchange(N, E, 4, rc["expert_count"], rc["send_off"])
    assert ex["status"] == ref.ST_CAPACITY
    x = _tiny_x(N, T, H, 9)
    w = np.full((N, T, R), 0.5, np.float32)
    o = ref.layer(N, T, E, R, H, 4, x, idx, w)
    assert o["status"] == ref.ST_BAD_EXPERT | ref.ST_CAPACITY
    # a rank that received more than cap rows dropped the rest: grouped rows stay < cap
    assert o["grp_q"].shape[1] == 4


# ----------------------------------------------------------------- combine numerics


def test_weighted_sum_exact_within_one_bf16_step():
    rng = np.random.default_rng(8)
    for _ in range(200):
        R, H = int(rng.integers(1, 9)), 64
        rows = _bf16(rng.standard_normal((R, H)))
        w = rng.dirichlet(np.ones(R)).astype(np.float32)
        out = _f32(ref.weighted_sum(rows, w)).astype(np.float64)
        rf = _f32(rows).astype(np.float64)
        exact = np.array([float(sum(Fraction(float(w[k])) * Fraction(float(rf[k, h]))
                                    for k in range(R))) for h in range(H)])
        ex_bf = _f32(_bf16(exact)).astype(np.float64)
        step = np.abs(ex_bf) * 2.0 ** -7 + 1e-30
        assert np.all(np.abs(out - ex_bf) <= step)
    # dropping a term is caught
    rows = _bf16(np.ones((2, 4)))
    assert _f32(ref.weighted_sum(rows, np.array([0.5, 0.5], np.float32)))[0] == 1.0
    assert _f32(ref.weighted_sum(rows, np.array([0.5, 0.5], np.float32),
                                 np.array([1, 0], np.int32)))[0] == 0.5


def _rn32(v: Fraction) -> Fraction:
    """v rounded to the nearest fp32 value, ties to even (normal and subnormal
    ranges; no overflow in these cases), in exact fractions."""
    if v == 0:
        return Fraction(0)
    a = abs(v)
    e = a.numerator.bit_length() - a.denominator.bit_length()
    if Fraction(2) ** e > a:
        e -= 1
    e = max(e, -126)                      # 2^e <= a < 2^(e+1), or the subnormal quantum
    ulp = Fraction(2) ** (e - 23)
    n, rest = divmod(a, ulp)
    n = int(n)
    if rest > ulp / 2 or (rest == ulp / 2 and n % 2 == 1):
        n += 1
    return (n * ulp) if v > 0 else -(n * ulp)


def _fma_chain(w, y, order, fused=True) -> float:
    """acc = 0; for k in order: acc = rn32(w_k * y_k + acc) (one rounding per
    slot), or with fused=False rn32(rn32(w_k * y_k) + acc)."""
    acc = Fraction(0)
    for k in order:
        p = Fraction(float(w[k])) * Fraction(float(y[k]))
        acc = _rn32((p if fused else _rn32(p)) + acc)
    return float(acc)


def _bf16_of(v: float) -> int:
    return int(torch.tensor([v], dtype=torch.float32).to(torch.bfloat16).view(torch.int16)
               .item()) & 0xFFFF


def test_weighted_sum_is_fma_chain_in_ascending_slot_order():
    """Every output element is bf16_rn of the fp32 fused multiply-add chain
    over the used slots in ascending order (fp32 accumulation in a fixed
    top-k slot order of the weighted average the combine takes: "Enabling
    trillion-parameter models on AWS EFA", "Dispatch and combine"), bit for
    bit."""
    rng = np.random.default_rng(31)
    for _ in range(60):
        R, H = int(rng.integers(1, 9)), 16
        rows = _bf16(rng.standard_normal((R, H)) * np.exp2(rng.integers(-6, 7, size=(R, 1))))
        w = rng.dirichlet(np.ones(R)).astype(np.float32)
        use = (rng.random(R) < 0.8).astype(np.int32)
        got = ref.weighted_sum(rows, w, use)
        y = _f32(rows).astype(np.float64)
        order = [k for k in range(R) if use[k]]
        for h in range(H):
            assert int(got[h]) == _bf16_of(_fma_chain(w, y[:, h], order)), (R, h)


def test_weighted_sum_order_hand_case():
    """Rows 1, 2^-24, 2^-24, -1 with unit weights.  In ascending slot order
    each 1 + 2^-24 is an fp32 tie that rounds to 1, so the result is 0;
    descending order keeps both small terms (2^-23), and a pairwise tree
    (1 + 2^-24) + (2^-24 - 1) keeps one (2^-24)."""
    y = np.array([1.0, 2.0 ** -24, 2.0 ** -24, -1.0])
    rows = _bf16(np.repeat(y[:, None], 4, axis=1))
    w = np.ones(4, np.float32)
    assert _fma_chain(w, y, [0, 1, 2, 3]) == 0.0
    assert _fma_chain(w, y, [3, 2, 1, 0]) == 2.0 ** -23
    pair = float(_rn32(_rn32(Fraction(1) + Fraction(2) ** -24) +
                       _rn32(Fraction(2) ** -24 - 1)))
    assert pair == 2.0 ** -24
    assert np.all(_f32(ref.weighted_sum(rows, w)) == 0.0)


def test_weighted_sum_fuses_multiply_and_add():
    """Slot 0 gives -1, slot 1 adds w*y.  For seeded weights where rounding
    the product to fp32 before the addition changes the bf16 result, the
    oracle gives the fused result."""
    rng = np.random.default_rng(77)
    y = np.array([-1.0, 1.0 + 2.0 ** -7])
    rows = _bf16(np.repeat(y[:, None], 2, axis=1))
    hits = 0
    for m in rng.integers(1, 2 ** 16, size=4000):
        w = np.array([1.0, 1.0 + float(m) * 2.0 ** -23], np.float32)
        fused, split = _fma_chain(w, y, [0, 1]), _fma_chain(w, y, [0, 1], fused=False)
        if _bf16_of(fused) == _bf16_of(split):
            continue
        hits += 1
        assert int(ref.weighted_sum(rows, w)[0]) == _bf16_of(fused)
    assert hits >= 5


def _standin_want(H, xrow, e, mode):
    """The stand-in output of expert e for token row x: fp32 product of the
    decoded code and its block scale (numpy, exact in float64 then one cast),
    times s_e = 2^((e mod 3) - 1) (mode 1) or 1, rounded by torch's bf16 cast."""
    q, sc = ref.quant_token(H, xrow)
    dq = (ref.e4m3_decode(q) * np.repeat(sc.astype(np.float64), 128)).astype(np.float32)
    se = np.float32(2.0 ** (e % 3 - 1)) if mode == 1 else np.float32(1.0)
    return _bf16(dq * se)


def _check_standin_lookup(N, T, E, R, H, idx, x, wt):
    """Every grouped row (main layout) and every low-latency row holds the
    stand-in of the expert that topk_idx names for it, found by brute force."""
    Er = E // N
    o = ref.layer(N, T, E, R, H, N * T * min(R, Er), x, idx, wt, mode=1)
    ll = ref.layer_ll(N, T, E, R, H, x, idx, wt, mode=1)
    _, grp, _ = brute.layouts(N, T, E, R, idx)
    llr = brute.ll_rows(N, T, E, R, idx)
    idx3 = np.asarray(idx).reshape(N, T, R)
    for (s, t, k), g in grp.items():
        e = int(idx3[s, t, k])
        want = _standin_want(H, x[s, t], e, 1)
        assert np.array_equal(o["y"][e // Er, g], want), (s, t, k)
        assert np.array_equal(ll["y_ll"][llr[(s, t, k)]], want), (s, t, k)


def test_standin_expert_lookup_mode1_all_routings_sampled():
    rng = np.random.default_rng(41)
    x = _tiny_x(2, 2, 128, 6)
    allr = list(brute.all_routings(2, 2, 4, 2))
    wt = np.full((2, 2, 2), 0.5, np.float32)
    for i in rng.choice(len(allr), 120, replace=False):
        _check_standin_lookup(2, 2, 4, 2, 128, allr[i], x, wt)


@pytest.mark.parametrize("name", ["tiny", "qwen3_worst"])
def test_standin_expert_lookup_mode1_configs(name):
    w = W.CONFIGS[name]
    if name == "qwen3_worst":
        w = w.replace(T=4, H=256)
    d = W.generate(w)
    _check_standin_lookup(w.N, w.T, w.E, w.R, w.H, d["topk_idx"], d["x"], d["topk_w"])


def test_standin_row_exact():
    rng = np.random.default_rng(12)
    H = 256
    x = _bf16(rng.standard_normal(H) * 3)
    q, sc = ref.quant_token(H, x)
    for e, se in [(0, 0.5), (1, 1.0), (2, 2.0), (3, 0.5)]:
        y = ref.standin_row(H, 1, e, q, sc)
        dq = ref.e4m3_decode(q) * np.repeat(sc.astype(np.float64), 128)
        want = _bf16((dq.astype(np.float32) * np.float32(se)))
        assert np.array_equal(y, want)
    assert np.array_equal(ref.standin_row(H, 0, 5, q, sc),
                          _bf16((ref.e4m3_decode(q) * np.repeat(sc.astype(np.float64), 128))
                                .astype(np.float32)))


@pytest.mark.parametrize("name", ["tiny", "qwen3_worst"])
def test_round_trip_identity_expert(name):
    """dispatch -> identity expert -> combine with weights summing to 1 gives
    bf16(dequant(quant(x))) within one bf16 step."""
    w = W.CONFIGS[name]
    if name == "qwen3_worst":
        w = w.replace(T=8, H=256)
    d = W.generate(w)
    o = ref.layer(w.N, w.T, w.E, w.R, w.H, w.default_cap, d["x"], d["topk_idx"], d["topk_w"])
    assert o["status"] == 0
    for s in range(w.N):
        for t in range(w.T):
            q, sc = ref.quant_token(w.H, d["x"][s, t])
            dq = ref.e4m3_decode(q) * np.repeat(sc.astype(np.float64), 128)
            want = _f32(_bf16(dq.astype(np.float32))).astype(np.float64)
            got = _f32(o["out"][s, t]).astype(np.float64)
            assert np.all(np.abs(got - want) <= np.abs(want) * 2.0 ** -7 + 1e-6)


# ----------------------------------------------------------------- low-latency layout


def test_ll_rows_bruteforce_all_routings_2x2x4x2():
    for idx in brute.all_routings(2, 2, 4, 2):
        o = ref.ll_rows(2, 2, 4, 2, idx)
        assert o["status"] == 0
        want = brute.ll_rows(2, 2, 4, 2, idx)
        for (s, t, k), row in want.items():
            assert o["ll_row"][s, t, k] == row
        cnt = np.zeros((2, 2, 2), np.int32)
        for (s, t, k, e) in brute.assignments(2, 2, 4, 2, idx):
            cnt[e // 2, e % 2, s] += 1
        assert np.array_equal(o["ll_count"], cnt)


def test_ll_rows_duplicates_overflow_and_bad_ids():
    N, T, E, R = 2, 2, 4, 3
    idx = np.array([[[1, 1, 1], [1, 2, 9]], [[0, 3, 2], [-1, 0, 1]]], np.int32)
    o = ref.ll_rows(N, T, E, R, idx)
    assert o["status"] == ref.ST_CAPACITY | ref.ST_BAD_EXPERT
    want = brute.ll_rows(N, T, E, R, idx)
    for (s, t, k), row in want.items():
        assert o["ll_row"][s, t, k] == (-1 if row is None else row)
    assert o["ll_row"][0, 1, 2] == -1 and o["ll_row"][1, 1, 0] == -1
    assert o["ll_count"][0, 1, 0] == 4   # expert 1 from sender 0: four rows, two fit


@pytest.mark.parametrize("name", ["tiny", "qwen3_worst"])
def test_ll_layer_matches_main_path(name):
    """The low-latency path places the same quantised rows and, with the same
    slot order of fused multiply-adds, gives the same combined output."""
    w = W.CONFIGS[name]
    if name == "qwen3_worst":
        w = w.replace(T=8, H=256)
    d = W.generate(w)
    main = ref.layer(w.N, w.T, w.E, w.R, w.H, w.default_cap, d["x"], d["topk_idx"], d["topk_w"])
    ll = ref.layer_ll(w.N, w.T, w.E, w.R, w.H, d["x"], d["topk_idx"], d["topk_w"])
    assert ll["status"] == 0
    assert np.array_equal(ll["out"], main["out"])
    for s in range(w.N):
        for t in range(w.T):
            for k in range(w.R):
                row = ll["ll_row"][s, t, k]
                q, sc = ref.quant_token(w.H, d["x"][s, t])
                assert np.array_equal(ll["ll_q"][row], q) and ll["ll_src"][row] == t


# ----------------------------------------------------------------- send-side reduction
#
# ref_combine_partial_send / _recv are pinned by: exact rational sums on
# every routing of a tiny shape and on random shapes with duplicates, bad ids
# and capacity drops (values chosen so that every partial and the result are
# exact in bf16, so any dropped, doubled or mis-weighted term shows); hand
# cases where the place of the extra bf16 rounding (per rank group) and the
# order of the final sum (ascending rank) change the result; the set of
# partial rows written against the brute-force rank sets; and the error
# bound two bf16 roundings imply, against the exact weighted sum.


def _partial_case(N, T, E, R, H, idx, w, yval, cap=None):
    """Routing arrays from the oracle's pinned route_count / exchange; the
    expert outputs placed at each assignment's grouped row by the brute-force
    layout; yval(s, t, k, e) gives the row's H values (exact in bf16)."""
    cap = cap or N * T * R
    idx = np.asarray(idx, np.int32).reshape(N, T, R)
    rc = ref.route_count(N, T, E, R, idx)
    ex = ref.exchange(N, E, cap, rc["expert_count"], rc["send_off"])
    _, grp, _ = brute.layouts(N, T, E, R, idx)
    Er = E // N
    y = np.zeros((N, cap, H), np.uint16)
    for (s, t, k), g in grp.items():
        e = int(idx[s, t, k])
        if g < cap:
            y[e // Er, g] = _bf16(np.broadcast_to(np.float32(yval(s, t, k, e)), (H,)))
    part = ref.combine_partial_send(N, T, E, R, H, cap, y, idx, np.asarray(w, np.float32),
                                    rc["slot_row"], rc["expert_send_off"], ex["seg_off"])
    out = ref.combine_partial_recv(N, T, E, R, H, part, idx, rc["slot_row"])
    return dict(rc=rc, ex=ex, y=y, part=part, out=out, grp=grp, cap=cap, idx=idx)


def _rank_sets(N, T, E, R, idx):
    Er = E // N
    D = {}
    for (s, t, k, e) in brute.assignments(N, T, E, R, idx):
        D.setdefault((s, t), set()).add(e // Er)
    return D


def _check_exact(N, T, E, R, H, idx, w, yv, cap=None):
    c = _partial_case(N, T, E, R, H, idx, w, lambda s, t, k, e: yv[s, t, k], cap)
    Er, D = E // N, _rank_sets(N, T, E, R, c["idx"])
    w = np.asarray(w, np.float32).reshape(N, T, R)
    for s in range(N):
        for t in range(T):
            total = Fraction(0)
            for r in range(N):
                got = c["part"][r, s, t]
                if r not in D.get((s, t), set()):
                    assert np.all(got == ref.FILL_U16), ("row written", r, s, t)
                    continue
                grp_sum = Fraction(0)
                for k in range(R):
                    e = int(c["idx"][s, t, k])
                    if 0 <= e < E and e // Er == r and c["grp"][(s, t, k)] < c["cap"]:
                        grp_sum += Fraction(float(w[s, t, k])) * Fraction(float(yv[s, t, k]))
                assert np.all(_f32(got) == float(grp_sum)), (r, s, t)
                total += grp_sum
            assert np.all(_f32(c["out"][s, t]) == float(total)), (s, t)
    return c


def test_partial_exact_sums_every_routing_2x2x4x2():
    rng = np.random.default_rng(31)
    for idx in brute.all_routings(2, 2, 4, 2):
        w = rng.choice([0.5, 1.0], size=(2, 2, 2))
        yv = rng.integers(-3, 4, size=(2, 2, 2)) / 4.0
        _check_exact(2, 2, 4, 2, 8, idx, w, yv)


@pytest.mark.parametrize("seed", range(12))
def test_partial_exact_sums_duplicates_bad_ids_and_drops(seed):
    rng = np.random.default_rng(100 + seed)
    N = int(rng.integers(1, 5))
    Er = int(rng.integers(1, 4))
    E, T, R, H = N * Er, int(rng.integers(1, 6)), int(rng.integers(1, 5)), 8
    idx = rng.integers(-1, E + 1, size=(N, T, R))     # duplicates and bad ids allowed
    w = rng.choice([0.5, 1.0], size=(N, T, R))
    yv = rng.integers(-3, 4, size=(N, T, R)) / 4.0
    cap = int(rng.integers(1, N * T * R + 1))         # some grouped rows dropped
    _check_exact(N, T, E, R, H, idx, w, yv, cap)


def test_partial_rounds_once_per_rank_group():
    """Two experts on rank 0 (outputs 1 and 2^-8) and one on rank 1 (2^-8):
    the rank-0 partial 1 + 2^-8 is a bf16 tie and rounds to 1, then
    1 + 2^-8 rounds to 1 again; accumulating all three on the receiving side
    gives 1 + 2^-7 instead."""
    N, T, E, R, H = 2, 1, 4, 3, 8
    idx = np.array([[[2, 0, 1]], [[3, 2, 1]]])
    vals = {0: 1.0, 1: 2.0 ** -8, 2: 2.0 ** -8, 3: 0.5}
    c = _partial_case(N, T, E, R, H, idx, np.ones((N, T, R)), lambda s, t, k, e: vals[e])
    assert np.all(_f32(c["part"][0, 0, 0]) == 1.0)
    assert np.all(_f32(c["part"][1, 0, 0]) == 2.0 ** -8)
    assert np.all(_f32(c["out"][0, 0]) == 1.0)
    main = ref.combine_recv(N, T, E, R, H, c["cap"],
                            ref.combine_send(N, T, E, R, H, c["cap"], c["y"],
                                             c["rc"]["expert_count"], c["rc"]["expert_send_off"],
                                             c["rc"]["send_off"], c["ex"]["seg_off"],
                                             c["ex"]["csend_off"]),
                            idx, np.ones((N, T, R), np.float32), c["rc"]["slot_row"],
                            c["rc"]["send_off"], c["ex"]["csend_off"])
    assert np.all(_f32(main[0, 0]) == 1.0 + 2.0 ** -7)


def test_partial_final_sum_in_ascending_rank_order():
    """Partials 1, 3*2^-24 and -1 on ranks 0, 1, 2 (slots in the order 2, 0,
    1): in ascending rank order 1 + 3*2^-24 is an fp32 tie that rounds up to
    1 + 2^-22, leaving 2^-22 after -1; in slot order the result would be
    3*2^-24."""
    N, T, E, R, H = 3, 1, 3, 3, 8
    idx = np.array([[[2, 0, 1]], [[0, 1, 2]], [[1, 2, 0]]])
    vals = {0: 1.0, 1: 3 * 2.0 ** -24, 2: -1.0}
    c = _partial_case(N, T, E, R, H, idx, np.ones((N, T, R)), lambda s, t, k, e: vals[e])
    for s in range(N):
        assert np.all(_f32(c["out"][s, 0]) == 2.0 ** -22), s


@pytest.mark.parametrize("name", ["tiny", "qwen3_skew"])
def test_partial_error_bound_against_exact(name):
    """|out - X| <= 2^-7 * sum_k |w_k y_k| + 2^-126, X the exact weighted sum:
    one bf16 rounding per partial and one at the end (unit roundoff 2^-8
    each), fp32 additions far below that."""
    w = W.CONFIGS[name]
    if name == "qwen3_skew":
        w = w.replace(T=4, H=256)
    d = W.generate(w)
    o = ref.layer_partial(w.N, w.T, w.E, w.R, w.H, w.default_cap, d["x"], d["topk_idx"],
                          d["topk_w"], mode=1)
    _, grp, _ = brute.layouts(w.N, w.T, w.E, w.R, d["topk_idx"])
    Er = w.E // w.N
    worst = 0.0
    for s in range(w.N):
        for t in range(w.T):
            X = np.zeros(w.H)
            A = np.zeros(w.H)
            for k in range(w.R):
                e = int(d["topk_idx"][s, t, k])
                yk = _f32(o["y"][e // Er, grp[(s, t, k)]]).astype(np.float64)
                X += float(d["topk_w"][s, t, k]) * yk
                A += abs(float(d["topk_w"][s, t, k])) * np.abs(yk)
            err = np.abs(_f32(o["out_partial"][s, t]).astype(np.float64) - X)
            assert np.all(err <= A * 2.0 ** -7 + 2.0 ** -126)
            worst = max(worst, float(np.max(err / (A + 1e-30))))
    assert worst > 0.0  # the extra rounding is visible somewhere


def test_partial_one_expert_per_rank_reduces_to_products():
    """E == N: every rank group holds one assignment, so each partial is the
    fp32 product w*y rounded to bf16 (torch's casts) and the result is their
    sum in ascending rank order."""
    N, T, R, H = 4, 3, 3, 16
    rng = np.random.default_rng(5)
    idx = np.stack([np.stack([rng.permutation(N)[:R] for _ in range(T)]) for _ in range(N)])
    w = rng.random((N, T, R)).astype(np.float32)
    yv = _f32(_bf16(rng.standard_normal((N, T, R))))
    c = _partial_case(N, T, N, R, H, idx, w, lambda s, t, k, e: yv[s, t, k])
    for s in range(N):
        for t in range(T):
            acc = np.float32(0.0)
            for r in range(N):
                ks = [k for k in range(R) if idx[s, t, k] == r]
                if not ks:
                    continue
                p = (torch.tensor(w[s, t, ks[0]]) * torch.tensor(yv[s, t, ks[0]])).to(
                    torch.bfloat16).float().item()
                assert np.all(_f32(c["part"][r, s, t]) == p)
                acc = np.float32(acc + np.float32(p))
            want = torch.tensor(float(acc), dtype=torch.float32).to(torch.bfloat16).float().item()
            assert np.all(_f32(c["out"][s, t]) == want)
