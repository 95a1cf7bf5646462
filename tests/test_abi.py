"""C-ABI checks that need no GPU: the library loads, exports every function
``include/*.h`` declares, sizes buffers as documented, and rejects bad
arguments on the host before anything touches CUDA.  The product package
never reaches the CPU oracle."""
from __future__ import annotations

import ctypes
import glob
import os
import re
import subprocess

import pytest

from combine_expert_count_gb300 import moeroute as m
from combine_expert_count_gb300 import workloads as W

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def lib():
    from combine_expert_count_gb300 import build
    build.build()
    return m.lib()


def _declared() -> set[str]:
    names = set()
    for h in glob.glob(os.path.join(ROOT, "include", "*.h")):
        src = open(h).read()
        src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
        names |= set(re.findall(r"^\s*(?:const\s+)?\w+\s*\**\s*(moe_\w+)\s*\(", src, flags=re.M))
    return names


def test_exports_every_declared_symbol(lib):
    declared = _declared()
    assert {"moe_route_count", "moe_exchange", "moe_dispatch_send", "moe_dispatch_recv",
            "moe_combine_send", "moe_combine_recv"} <= declared
    out = subprocess.run(["nm", "-D", "--defined-only", m.library_path()], capture_output=True,
                         text=True, check=True).stdout
    exported = set(re.findall(r"\sT\s(moe_\w+)$", out, flags=re.M))
    assert declared <= exported, declared - exported
    for name in declared:
        getattr(lib, name)
    assert set(m.EXPORTS) <= declared


def test_version_and_strerror(lib):
    assert m.lib().moe_version() >> 16 == 1
    for code in (m.MOE_OK, m.MOE_EINVAL, m.MOE_ENOTSUP, m.MOE_ECUDA, m.MOE_ST_BAD_EXPERT,
                 m.MOE_ST_CAPACITY, m.MOE_ST_TIMEOUT):
        assert m.strerror(code) and "unknown" not in m.strerror(code)


@pytest.mark.parametrize("name", ["tiny", "dsv3_decode", "kimi_k2_decode", "prefill",
                                  "qwen3_skew"])
def test_sizes_query_matches_layout(lib, name):
    w = W.CONFIGS[name]
    z = m.sizes_query(m.make_shape(w.N, w.T, w.E, w.R, w.H))
    N, T, E, R, H, Er, Sb = w.N, w.T, w.E, w.R, w.H, w.Er, w.H // 128
    cap = N * T * min(R, Er)
    assert z.cap == cap == w.default_cap
    assert z.send_rows == T * R
    assert z.bytes_x == N * T * H * 2
    assert z.bytes_send_q == N * T * R * H and z.bytes_send_s == N * T * R * Sb * 4
    assert z.bytes_grp_q == N * cap * H and z.bytes_grp_s == N * cap * Sb * 4
    assert z.bytes_grp_src == N * cap * 8 and z.bytes_y == N * cap * H * 2
    assert z.bytes_seg_off == N * Er * N * 4 and z.bytes_grp_off == N * (Er + 1) * 4
    assert z.ll_rows == N * E * T and z.bytes_ll_q == N * E * T * H
    assert z.bytes_ll_count == N * E * 4 and z.bytes_ll_y == N * E * T * H * 2
    assert z.bytes_sig == (2 * N * N + 4) * 4
    assert z.bytes_part == N * N * T * H * 2
    z2 = m.sizes_query(m.make_shape(w.N, w.T, w.E, w.R, w.H, 100))
    assert z2.cap == 100 and z2.bytes_grp_q == N * 100 * H


@pytest.mark.parametrize("shape,code", [
    ((0, 4, 8, 2, 256, 0), m.MOE_EINVAL),       # N <= 0
    ((2, -1, 8, 2, 256, 0), m.MOE_EINVAL),      # T < 0
    ((2, 4, 8, 2, 200, 0), m.MOE_EINVAL),       # H % 128
    ((3, 4, 8, 2, 256, 0), m.MOE_EINVAL),       # E % N
    ((2, 4, 8, 9, 256, 0), m.MOE_EINVAL),       # R > E
    ((2, 4, 8, 0, 256, 0), m.MOE_EINVAL),       # R <= 0
    ((2, 4, 8, 2, 256, -5), m.MOE_EINVAL),      # cap < 0
    ((2, 4, 2048, 2, 256, 0), m.MOE_ENOTSUP),   # E beyond the limit
    ((2, 4, 64, 33, 256, 0), m.MOE_ENOTSUP),    # R beyond the limit
    ((2, 4, 8, 2, 65664, 0), m.MOE_ENOTSUP),    # H beyond the limit
])
def test_bad_shapes_rejected(lib, shape, code):
    sh = m.moe_shape(*shape)
    z = m.moe_sizes()
    assert m.lib().moe_sizes_query(ctypes.byref(sh), ctypes.byref(z)) == code
    p = ctypes.c_void_p(0x1000)
    assert m.lib().moe_route_count(ctypes.byref(sh), p, p, p, p, p, p, None) == code


def test_null_and_misaligned_pointers_rejected(lib):
    sh = m.moe_shape(2, 4, 8, 2, 256, 0)
    good, bad, null = ctypes.c_void_p(0x10000), ctypes.c_void_p(0x10004), None
    L = m.lib()
    # every pointer slot of every entry point, one at a time
    calls = {
        "moe_route_count": 6, "moe_exchange": 7, "moe_route": 10, "moe_dispatch_send": 6,
        "moe_dispatch_recv": 10, "moe_combine_send": 8, "moe_combine_recv": 8,
        "moe_dispatch_ll": 8, "moe_combine_ll": 5, "moe_combine_partial_send": 7,
        "moe_combine_partial_recv": 4,
    }
    for name, nptr in calls.items():
        fn = getattr(L, name)
        for i in range(nptr):
            for p in (bad, null):
                args = [good] * nptr
                args[i] = p
                assert fn(ctypes.byref(sh), *args, None) == m.MOE_EINVAL, (name, i, p)
    for fn in (L.moe_dispatch, L.moe_dispatch_send_recv, L.moe_combine):
        assert fn(ctypes.byref(sh), None, None) == m.MOE_EINVAL
        needs = m._COMBINE_NEEDS if fn is L.moe_combine else m._DISPATCH_NEEDS
        for field in list(needs) + ["status"]:
            b = m.moe_buffers(*([0x10000] * len(m._BUFFER_FIELDS)))
            setattr(b, field, 0x10004)
            assert fn(ctypes.byref(sh), ctypes.byref(b), None) == m.MOE_EINVAL, field
    full = m.moe_buffers(*([0x10000] * len(m._BUFFER_FIELDS)))
    for part in (bad, null):
        assert L.moe_combine_partial(ctypes.byref(sh), ctypes.byref(full), part,
                                     None) == m.MOE_EINVAL
    for field in list(m._PARTIAL_NEEDS):
        b = m.moe_buffers(*([0x10000] * len(m._BUFFER_FIELDS)))
        setattr(b, field, 0x10004)
        assert L.moe_combine_partial(ctypes.byref(sh), ctypes.byref(b), good,
                                     None) == m.MOE_EINVAL, field
    for sig in (bad, null):
        assert L.moe_dispatch_signalled(ctypes.byref(sh), ctypes.byref(full), sig,
                                        None) == m.MOE_EINVAL
    assert L.moe_dispatch_signalled(ctypes.byref(sh), None, good, None) == m.MOE_EINVAL
    for field in list(m._DISPATCH_NEEDS) + ["status"]:
        b = m.moe_buffers(*([0x10000] * len(m._BUFFER_FIELDS)))
        setattr(b, field, 0x10004)
        assert L.moe_dispatch_signalled(ctypes.byref(sh), ctypes.byref(b), good,
                                        None) == m.MOE_EINVAL, field
    assert L.moe_expert_standin(ctypes.byref(sh), 2, good, good, good, good, None) == m.MOE_EINVAL
    assert L.moe_expert_standin(ctypes.byref(sh), 0, bad, good, good, good, None) == m.MOE_EINVAL
    assert L.moe_expert_standin_ll(ctypes.byref(sh), 2, good, good, good, good,
                                   None) == m.MOE_EINVAL
    for i in range(4):
        for p in (bad, null):
            args = [good] * 4
            args[i] = p
            assert L.moe_expert_standin_ll(ctypes.byref(sh), 0, *args, None) == m.MOE_EINVAL
    assert L.moe_e4m3_encode(null, good, 4, None) == m.MOE_EINVAL
    assert L.moe_e4m3_encode(good, good, -1, None) == m.MOE_EINVAL
    assert L.moe_route_count(None, good, good, good, good, good, good, None) == m.MOE_EINVAL


def test_binding_raises_and_checks_sizes(lib):
    with pytest.raises(m.MoeError) as ei:
        m.sizes_query(m.make_shape(2, 4, 8, 2, 100))
    assert ei.value.code == m.MOE_EINVAL
    import torch
    with pytest.raises(ValueError):
        m.moe_route_count(m.make_shape(2, 4, 8, 2, 256), torch.zeros(16, dtype=torch.int32),
                          None, None, None, None, None)


@pytest.mark.gpu
def test_binding_accepts_pinned_host_only_for_x_and_out(lib):
    import torch
    if not torch.cuda.is_available():
        pytest.skip("pinned host memory needs a CUDA driver")
    t = torch.zeros(64, dtype=torch.int32).pin_memory()
    assert m._p(t, 4, "x") is not None
    with pytest.raises(ValueError):
        m._p(t, 4, "topk_idx")
    with pytest.raises(ValueError):
        m._p(torch.zeros(64, dtype=torch.int32), 4, "x")


def test_missing_library_fails_loudly(monkeypatch):
    monkeypatch.setattr(m, "_LIB_PATH", "/nonexistent/libmoeroute.so")
    monkeypatch.setattr(m, "_lib", None)
    with pytest.raises(RuntimeError, match="not built"):
        m.lib()


def test_product_never_imports_oracle():
    pkg = os.path.join(ROOT, "combine_expert_count_gb300")
    for f in glob.glob(os.path.join(pkg, "**", "*"), recursive=True):
        if f.endswith((".py", ".cu", ".cuh", ".h")):
            src = open(f).read()
            assert not re.search(r"^\s*(from|import)\s+oracle", src, flags=re.M), f
            assert "moe_ref" not in src and "libmoe_ref" not in src, f
