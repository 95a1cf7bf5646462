"""Helpers for the GPU parity tests: run the CUDA path through the C ABI and
compare it with the CPU oracle.  Output buffers are pre-filled with sentinel
patterns so a row the kernels never write (or write by mistake) shows up."""
from __future__ import annotations

import numpy as np
import torch

from combine_expert_count_gb300 import moeroute as m
from combine_expert_count_gb300 import workloads as W

SENT_U8 = 0xA5
SENT_I32 = -12345
SENT_U16 = 0x7FA5


def to_dev(d: dict, dev="cuda") -> dict:
    out = {}
    if "x" in d:
        out["x"] = torch.from_numpy(np.ascontiguousarray(d["x"]).view(np.int16)).to(dev)
    out["topk_idx"] = torch.from_numpy(np.ascontiguousarray(d["topk_idx"])).to(dev)
    out["topk_w"] = torch.from_numpy(np.ascontiguousarray(d["topk_w"])).to(dev)
    return out


def fill_sentinels(buf: m.MoeBuffers) -> None:
    for name in ("send_q", "grp_q"):
        getattr(buf, name).fill_(SENT_U8)
    for name in ("send_s", "grp_s"):
        getattr(buf, name).fill_(float("nan"))
    for name in ("send_tok", "grp_src", "slot_row", "expert_count", "send_off",
                 "expert_send_off", "grp_off", "seg_off", "csend_off", "m_sizes"):
        getattr(buf, name).fill_(SENT_I32)
    for name in ("y", "csend", "out"):
        getattr(buf, name).view(torch.int16).fill_(SENT_U16)
    buf.status.fill_(-1)


def run_path(w: W.Workload, dd: dict, cap: int = 0, mode: int | None = None,
             sentinels: bool = True, calls: str = "fused") -> m.MoeBuffers:
    """Whole path on the GPU: dispatch, stand-in expert, combine.  ``calls``
    picks the call form (see MoeBuffers.dispatch)."""
    buf = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H, cap=cap, device="cuda")
    if sentinels:
        fill_sentinels(buf)
    buf.dispatch(dd["x"], dd["topk_idx"], calls=calls)
    buf.expert(mode if mode is not None else (1 if w.expert == "scale" else 0))
    buf.combine(dd["topk_idx"], dd["topk_w"], calls="fused" if calls == "signalled" else calls)
    torch.cuda.synchronize()
    return buf


def host(t: torch.Tensor) -> np.ndarray:
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).cpu().numpy().view(np.uint16)
    return t.cpu().numpy()


def bf16_f32(b: np.ndarray) -> np.ndarray:
    return (np.asarray(b, np.uint16).astype(np.uint32) << 16).view(np.float32)


def assert_eq(name: str, got: np.ndarray, want: np.ndarray) -> None:
    got = np.asarray(got)
    want = np.asarray(want)
    assert got.shape == want.shape, (name, got.shape, want.shape)
    if got.dtype.kind == "f":
        same = (got.view(np.uint32) == want.view(np.uint32))
    else:
        same = got == want
    if not np.all(same):
        bad = np.argwhere(~same)
        i = tuple(bad[0])
        raise AssertionError(f"{name}: {bad.shape[0]} of {same.size} differ; first at {i}: "
                             f"gpu={got[i]!r} oracle={want[i]!r}")


def assert_combine_close(got_bits: np.ndarray, want_bits: np.ndarray) -> int:
    """The combine tolerance: |gpu - oracle| <= 2^-7 |oracle| + 1e-6 (one bf16
    step).  Returns how many elements are not bit-identical."""
    g = bf16_f32(got_bits).astype(np.float64)
    r = bf16_f32(want_bits).astype(np.float64)
    err = np.abs(g - r)
    tol = np.abs(r) * 2.0 ** -7 + 1e-6
    ok = err <= tol
    if not np.all(ok):
        i = tuple(np.argwhere(~ok)[0])
        raise AssertionError(f"combine: {int((~ok).sum())} elements beyond one bf16 step; "
                             f"first at {i}: gpu={g[i]} oracle={r[i]}")
    return int((got_bits != want_bits).sum())


def compare_with_oracle(w: W.Workload, buf: m.MoeBuffers, o: dict, exact_combine: bool = True):
    """Element-by-element comparison of every output the oracle produced."""
    N, E = w.N, w.E
    assert_eq("expert_count", host(buf.expert_count), o["expert_count"])
    assert_eq("send_off", host(buf.send_off), o["send_off"])
    assert_eq("expert_send_off", host(buf.expert_send_off), o["expert_send_off"])
    assert_eq("slot_row", host(buf.slot_row), o["slot_row"])
    assert_eq("grp_off", host(buf.grp_off), o["grp_off"])
    assert_eq("seg_off", host(buf.seg_off), o["seg_off"])
    assert_eq("csend_off", host(buf.csend_off), o["csend_off"])
    assert_eq("m_sizes", host(buf.m_sizes), o["m_sizes"])
    assert int(buf.status.item()) == o["status"], (int(buf.status.item()), o["status"])
    sq, ss, st = host(buf.send_q), host(buf.send_s), host(buf.send_tok)
    for s in range(N):
        n = int(o["send_off"][s, -1])
        assert_eq(f"send_q[{s}]", sq[s, :n], o["send_q"][s, :n])
        assert_eq(f"send_s[{s}]", ss[s, :n], o["send_s"][s, :n])
        assert_eq(f"send_tok[{s}]", st[s, :n], o["send_tok"][s, :n])
        assert np.all(sq[s, n:] == SENT_U8), f"send_q[{s}] rows past {n} were written"
    cap_g, cap_o = buf.cap, o["grp_q"].shape[1]
    gq, gs, gsrc = host(buf.grp_q), host(buf.grp_s), host(buf.grp_src)
    y, cs = host(buf.y), host(buf.csend)
    for r in range(N):
        n = min(int(o["grp_off"][r, -1]), cap_g, cap_o)
        assert_eq(f"grp_q[{r}]", gq[r, :n], o["grp_q"][r, :n])
        assert_eq(f"grp_s[{r}]", gs[r, :n], o["grp_s"][r, :n])
        assert_eq(f"grp_src[{r}]", gsrc[r, :n], o["grp_src"][r, :n])
        assert_eq(f"y[{r}]", y[r, :n], o["y"][r, :n])
        if n < cap_g:
            assert np.all(gq[r, n:] == SENT_U8), f"grp_q[{r}] rows past {n} were written"
        nc = min(int(o["csend_off"][r, -1]), cap_g, cap_o)
        assert_eq(f"csend[{r}]", cs[r, :nc], o["csend"][r, :nc])
    out = host(buf.out)
    if exact_combine:
        assert_eq("out", out, o["out"])
    return assert_combine_close(out, o["out"])


def compare_with_oracle_by_rank(w: W.Workload, buf: m.MoeBuffers, o: dict) -> None:
    """compare_with_oracle for workloads whose device buffers are too large to
    copy to the host at once: every output element the oracle produced,
    compared rank by rank (only each rank's written rows are copied), the
    rows just past each count checked for the sentinel, and the combine bit
    for bit and at one bf16 step."""
    N = w.N
    for k in ("expert_count", "send_off", "expert_send_off", "slot_row", "grp_off", "seg_off",
              "csend_off", "m_sizes"):
        assert_eq(k, host(getattr(buf, k)), o[k])
    assert int(buf.status.item()) == o["status"], (int(buf.status.item()), o["status"])
    for s in range(N):
        n = int(o["send_off"][s, -1])
        assert_eq(f"send_q[{s}]", host(buf.send_q[s, :n]), o["send_q"][s, :n])
        assert_eq(f"send_s[{s}]", host(buf.send_s[s, :n]), o["send_s"][s, :n])
        assert_eq(f"send_tok[{s}]", host(buf.send_tok[s, :n]), o["send_tok"][s, :n])
        if n < buf.send_q.shape[1]:
            assert np.all(host(buf.send_q[s, n:n + 4]) == SENT_U8), f"send_q[{s}] past {n}"
    cap_g, cap_o = buf.cap, o["grp_q"].shape[1]
    for r in range(N):
        n = min(int(o["grp_off"][r, -1]), cap_g, cap_o)
        assert_eq(f"grp_q[{r}]", host(buf.grp_q[r, :n]), o["grp_q"][r, :n])
        assert_eq(f"grp_s[{r}]", host(buf.grp_s[r, :n]), o["grp_s"][r, :n])
        assert_eq(f"grp_src[{r}]", host(buf.grp_src[r, :n]), o["grp_src"][r, :n])
        assert_eq(f"y[{r}]", host(buf.y[r, :n]), o["y"][r, :n])
        if n < cap_g:
            assert np.all(host(buf.grp_q[r, n:n + 4]) == SENT_U8), f"grp_q[{r}] past {n}"
        nc = min(int(o["csend_off"][r, -1]), cap_g, cap_o)
        assert_eq(f"csend[{r}]", host(buf.csend[r, :nc]), o["csend"][r, :nc])
    for s in range(N):
        got = host(buf.out[s])
        assert_eq(f"out[{s}]", got, o["out"][s])
        assert_combine_close(got, o["out"][s])
