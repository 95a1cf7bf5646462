"""GPU parity on small decode batches of the DSv3 EP16 shape (16 ranks, 256
experts, top-8, rows of 7168 elements), where the token-block kernels give
a token's rows to several blocks because the batch alone cannot fill the
GPU.  Every call form is compared with the CPU oracle bit for bit, on row
lengths whose 16-byte chunks do and do not divide evenly between the blocks
of a token."""
from __future__ import annotations

import pytest
import torch

from combine_expert_count_gb300 import moeroute as m
from combine_expert_count_gb300 import workloads as W
from oracle import ref

from . import _gpu as G
from .test_low_latency_gpu import _check_ll, _run_ll
from .test_partial_gpu import _check as _check_partial

pytestmark = pytest.mark.gpu

SHAPES = [(1, 7168), (3, 7296), (16, 7168), (2, 1152)]  # (tokens per rank, H)


@pytest.fixture(scope="module", autouse=True)
def _built():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from combine_expert_count_gb300 import build
    build.build()
    ref.build()
    m.lib()


def _workload(T, H):
    base = W.CONFIGS["dsv3_decode"]
    return base.replace(T=T, H=H, seed=base.seed + 500 + 7 * T + H)


@pytest.mark.parametrize("calls", ["fused", "separate", "fused_route", "signalled"])
@pytest.mark.parametrize("T,H", SHAPES)
def test_main_path(T, H, calls):
    w = _workload(T, H)
    d = W.generate(w)
    buf = G.run_path(w, G.to_dev(d), calls=calls)
    o = ref.layer(w.N, w.T, w.E, w.R, w.H, w.default_cap, d["x"], d["topk_idx"],
                  d["topk_w"], mode=1)
    G.compare_with_oracle(w, buf, o)


@pytest.mark.parametrize("calls", ["partial", "partial_separate"])
@pytest.mark.parametrize("T,H", SHAPES)
def test_send_side_reduction(T, H, calls):
    w = _workload(T, H)
    _check_partial(w, W.generate(w), calls)


@pytest.mark.parametrize("T,H", SHAPES)
def test_low_latency(T, H):
    w = _workload(T, H)
    d = W.generate(w)
    b = _run_ll(w, d, 1)
    _check_ll(w, d, b, 1)
