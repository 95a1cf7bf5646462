"""moe_dispatch_signalled_static against moe_dispatch_signalled, through the
C ABI, over two calls in a row with different inputs.

The static entry keeps the signalled dispatch's flag scratch in a device
array of the library, for callers that cannot allocate that buffer: a
serving process that fixes its device-memory plan at start-up and must not
allocate while serving, or a C caller that only holds the buffers another
framework allocated.  Its outputs must equal the caller-scratch entry's bit
for bit.  This file is collected last, so a run that stops at the first
failure has already run every other test; it also passes on its own."""
from __future__ import annotations

import numpy as np
import pytest
import torch

from combine_expert_count_gb300 import moeroute as m
from combine_expert_count_gb300 import workloads as W

pytestmark = pytest.mark.gpu

OUTPUTS = ("expert_count", "send_off", "expert_send_off", "slot_row", "grp_off", "seg_off",
           "csend_off", "m_sizes", "send_q", "send_s", "send_tok", "grp_q", "grp_s", "grp_src")


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_expert_count_gb300 import build
    build.build()
    m.lib()


def _bufs(w):
    b = m.MoeBuffers(w.N, w.T, w.E, w.R, w.H)
    for name in OUTPUTS:
        t = getattr(b, name)
        if t.dtype == torch.float32:
            t.fill_(float("nan"))
        else:
            t.view(torch.uint8).fill_(0xA5)
    return b


def _inputs(w, seed):
    d = W.generate(w.replace(seed=seed))
    return (torch.from_numpy(d["x"].view(np.int16)).cuda(),
            torch.from_numpy(d["topk_idx"]).cuda())


@pytest.mark.parametrize("name,T", [("tiny", 16), ("dsv3_decode", 32), ("qwen3_skew", 48)])
def test_static_scratch_matches_caller_scratch_two_calls(name, T):
    w = W.CONFIGS[name].replace(T=T)
    want, got = _bufs(w), _bufs(w)
    sig = torch.zeros(int(want.sizes.bytes_sig) // 4, dtype=torch.int32, device="cuda")
    for seed in (101, 202):
        x, idx = _inputs(w, seed)
        m.moe_dispatch_signalled(want.shape, want.tensors(x=x, topk_idx=idx), sig)
        m.moe_dispatch_signalled_static(got.shape, got.tensors(x=x, topk_idx=idx))
        torch.cuda.synchronize()
        assert int(want.status.item()) == 0 and int(got.status.item()) == 0
        for name_ in OUTPUTS:
            a, b = getattr(want, name_), getattr(got, name_)
            assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), (name_, seed)


def test_static_scratch_at_its_limit():
    """64 ranks, the most the static scratch holds: the same outputs as the
    caller's scratch."""
    w = W.Workload("static64", N=64, T=4, H=256, E=128, R=2, seed=64)
    want, got = _bufs(w), _bufs(w)
    sig = torch.zeros(int(want.sizes.bytes_sig) // 4, dtype=torch.int32, device="cuda")
    x, idx = _inputs(w, 303)
    m.moe_dispatch_signalled(want.shape, want.tensors(x=x, topk_idx=idx), sig)
    m.moe_dispatch_signalled_static(got.shape, got.tensors(x=x, topk_idx=idx))
    torch.cuda.synchronize()
    assert int(want.status.item()) == 0 and int(got.status.item()) == 0
    for name_ in OUTPUTS:
        a, b = getattr(want, name_), getattr(got, name_)
        assert torch.equal(a.view(torch.uint8), b.view(torch.uint8)), name_


def test_beyond_the_static_limit_is_rejected():
    sh = m.make_shape(128, 4, 128, 2, 256)
    z = m.sizes_query(sh)
    b = m.moe_buffers(*([0x10000] * len(m._BUFFER_FIELDS)))
    import ctypes
    rc = m.lib().moe_dispatch_signalled_static(ctypes.byref(sh), ctypes.byref(b), None)
    assert rc == m.MOE_ENOTSUP and z.bytes_sig > (2 * 64 * 64 + 4) * 4
