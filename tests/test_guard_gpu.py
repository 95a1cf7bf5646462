"""Writes past the end of a buffer: every output buffer is allocated with a
guard band after the size the library asks for, filled with a pattern, and
every entry point runs on small odd shapes; the guard bands must come back
untouched (with memcheck closed on this pool, this is how a stray write at
the end of a buffer shows up)."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from combine_expert_count_gb300 import moeroute as m
from combine_expert_count_gb300 import workloads as W

pytestmark = pytest.mark.gpu

GUARD = 65536
PAT = 0x5A


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_expert_count_gb300 import build
    build.build()
    m.lib()


class Guarded:
    """Byte buffers of exactly `nbytes` followed by a guard band."""

    def __init__(self):
        self.bufs = {}

    def __call__(self, name, nbytes, dtype=torch.uint8):
        raw = torch.full((int(nbytes) + GUARD,), PAT, dtype=torch.uint8, device="cuda")
        self.bufs[name] = (raw, int(nbytes))
        view = raw[:int(nbytes)]
        return view.view(dtype) if nbytes % torch.tensor([], dtype=dtype).element_size() == 0 \
            else view

    def check(self):
        torch.cuda.synchronize()
        for name, (raw, n) in self.bufs.items():
            tail = raw[n:]
            assert bool((tail == PAT).all()), f"{name}: write past its end"


def _inputs(w):
    d = W.generate(w)
    return (torch.from_numpy(d["x"].view(np.int16)).cuda(),
            torch.from_numpy(d["topk_idx"]).cuda(), torch.from_numpy(d["topk_w"]).cuda())


@pytest.mark.parametrize("N,T,E,R,H", [(2, 16, 8, 2, 256), (3, 5, 12, 9, 640),
                                       (2, 3, 4, 2, 8192 + 1024), (4, 7, 32, 32, 128),
                                       (1, 64, 1024, 32, 128), (2, 40, 8, 8, 2048),
                                       (2, 600, 8, 4, 256), (2, 3, 4, 2, 65536)])
def test_no_write_past_any_buffer(N, T, E, R, H):
    w = W.Workload("guard", N=N, T=T, H=H, E=E, R=R, seed=71)
    x, idx, wt = _inputs(w)
    sh = m.make_shape(N, T, E, R, H)
    z = m.sizes_query(sh)
    g = Guarded()
    t = {"x": x, "topk_idx": idx, "topk_w": wt}
    for name, key, dt in [("expert_count", "bytes_expert_count", torch.int32),
                          ("send_off", "bytes_send_off", torch.int32),
                          ("expert_send_off", "bytes_expert_send_off", torch.int32),
                          ("slot_row", "bytes_topk_idx", torch.int32),
                          ("grp_off", "bytes_grp_off", torch.int32),
                          ("seg_off", "bytes_seg_off", torch.int32),
                          ("csend_off", "bytes_send_off", torch.int32),
                          ("m_sizes", "bytes_m_sizes", torch.int32),
                          ("send_q", "bytes_send_q", torch.uint8),
                          ("send_s", "bytes_send_s", torch.float32),
                          ("send_tok", "bytes_send_tok", torch.int32),
                          ("grp_q", "bytes_grp_q", torch.uint8),
                          ("grp_s", "bytes_grp_s", torch.float32),
                          ("grp_src", "bytes_grp_src", torch.int32),
                          ("y", "bytes_y", torch.bfloat16),
                          ("csend", "bytes_y", torch.bfloat16),
                          ("out", "bytes_x", torch.bfloat16)]:
        t[name] = g(name, getattr(z, key), dt)
    t["status"] = g("status", 4, torch.int32)
    sig = g("sig", z.bytes_sig, torch.int32)
    sig.zero_()
    part = g("part", z.bytes_part, torch.bfloat16)

    # the whole path in every call form
    m.moe_dispatch(sh, t)
    m.moe_expert_standin(sh, 1, t["grp_q"], t["grp_s"], t["grp_off"], t["y"])
    m.moe_combine(sh, t)
    m.moe_dispatch_signalled(sh, t, sig)
    m.moe_combine_partial(sh, t, part)
    m.moe_combine_partial_send(sh, t["y"], idx, wt, t["slot_row"], t["expert_send_off"],
                               t["seg_off"], part)
    m.moe_combine_partial_recv(sh, part, idx, t["slot_row"], t["out"])
    m.moe_route_count(sh, idx, t["expert_count"], t["send_off"], t["expert_send_off"],
                      t["slot_row"], t["status"])
    m.moe_exchange(sh, t["expert_count"], t["send_off"], t["grp_off"], t["seg_off"],
                   t["csend_off"], t["m_sizes"], t["status"])
    m.moe_dispatch_send(sh, x, t["slot_row"], t["send_q"], t["send_s"], t["send_tok"],
                        t["status"])
    m.moe_dispatch_recv(sh, t["send_q"], t["send_s"], t["send_tok"], t["expert_count"],
                        t["expert_send_off"], t["seg_off"], t["grp_q"], t["grp_s"],
                        t["grp_src"], t["status"])
    m.moe_combine_send(sh, t["y"], t["expert_count"], t["expert_send_off"], t["send_off"],
                       t["seg_off"], t["csend_off"], t["csend"], t["status"])
    m.moe_combine_recv(sh, t["csend"], idx, wt, t["slot_row"], t["send_off"], t["csend_off"],
                       t["out"], t["status"])
    g.check()
    assert int(t["status"].item()) == 0

    # the low-latency layout
    ll = {name: g("ll_" + name, getattr(z, key), dt) for name, key, dt in
          [("q", "bytes_ll_q", torch.uint8), ("s", "bytes_ll_s", torch.float32),
           ("src", "bytes_ll_src", torch.int32), ("count", "bytes_ll_count", torch.int32),
           ("row", "bytes_topk_idx", torch.int32), ("y", "bytes_ll_y", torch.bfloat16)]}
    m.moe_dispatch_ll(sh, x, idx, ll["q"], ll["s"], ll["src"], ll["count"], ll["row"],
                      t["status"])
    m.moe_expert_standin_ll(sh, 1, ll["q"], ll["s"], ll["count"], ll["y"])
    m.moe_combine_ll(sh, ll["y"], wt, ll["row"], t["out"], t["status"])
    g.check()
