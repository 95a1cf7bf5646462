"""Seeded synthetic MoE layer inputs shaped like the models the pages measure.

This module only synthesises inputs: activations ``x`` (bf16 bits), the router's
top-R expert ids and their weights. It holds none of the dispatch/combine
arithmetic (no counting, scanning, quantisation, packing or reduction), so it
may feed both the CUDA path and the CPU oracle.

Shapes follow the pages:
  * "Enabling trillion-parameter models on AWS EFA" (Perplexity), section
    "Evaluation: dispatch/combine latency": hidden 7168, DeepSeek-V3 and Kimi-K2
    configurations, dispatch batch 128, combine batch 4096.
  * "750B MoE model from RoCE to AWS EFA" (AWS China blog), section 4.4: 256
    experts over 16 GPUs (16 per GPU), top-8.
  * "Perseus" article (itsolotime), section 2.1 (Qwen3-30B: 128 experts,
    16 PEs, 8 experts per PE) and section 4.5 (Zipf-skewed routing, exponent
    0..1.5; at 1.5 the top 10 experts receive 82% of tokens).

No dataset, trace or model weight is involved: every value is drawn from a
``numpy.random.Generator(PCG64(seed))`` stream.

Router recipe (input synthesis only): logits ~ N(0,1) [N*T, E]; probabilities
= softmax over E (float64); the R experts with the largest probability are
chosen, ties going to the lower expert id, stored in descending-probability
order; weights = the chosen probabilities renormalised to sum to 1, cast to
float32.
"""
from __future__ import annotations

import dataclasses
import functools
import math

import numpy as np
import torch

SEED_BASE = 20261202


@dataclasses.dataclass(frozen=True)
class Workload:
    """One MoE layer configuration.

    N ranks (expert-parallel group), T tokens per rank, H hidden size, E experts,
    R experts per token.  ``expert`` selects the grouped-GEMM stand-in
    ("identity" or "scale"), ``routing`` the router recipe ("softmax", "skew",
    "worst", "zipf"), ``zipf_s`` the Zipf exponent for "zipf".
    """

    name: str
    N: int
    T: int
    H: int
    E: int
    R: int
    expert: str = "identity"
    routing: str = "softmax"
    seed: int = SEED_BASE
    zipf_s: float = 0.0

    @property
    def Er(self) -> int:
        return self.E // self.N

    @property
    def A(self) -> int:
        """Total (token, expert) assignments over all ranks."""
        return self.N * self.T * self.R

    @property
    def default_cap(self) -> int:
        """Grouped rows per rank that hold any routing with distinct experts per token."""
        return self.N * self.T * min(self.R, self.Er)

    def replace(self, **kw) -> "Workload":
        return dataclasses.replace(self, **kw)


CONFIGS: dict[str, Workload] = {
    "tiny": Workload("tiny", N=2, T=16, H=256, E=8, R=2, expert="identity",
                     routing="softmax", seed=SEED_BASE + 0),
    "dsv3_decode": Workload("dsv3_decode", N=16, T=128, H=7168, E=256, R=8,
                            expert="scale", routing="softmax", seed=SEED_BASE + 1),
    "kimi_k2_decode": Workload("kimi_k2_decode", N=32, T=128, H=7168, E=384, R=8,
                               expert="identity", routing="softmax", seed=SEED_BASE + 2),
    "prefill": Workload("prefill", N=8, T=4096, H=7168, E=256, R=8,
                        expert="identity", routing="softmax", seed=SEED_BASE + 3),
    "qwen3_skew": Workload("qwen3_skew", N=16, T=512, H=2048, E=128, R=8,
                           expert="identity", routing="skew", seed=SEED_BASE + 4),
    "qwen3_worst": Workload("qwen3_worst", N=16, T=512, H=2048, E=128, R=8,
                            expert="identity", routing="worst", seed=SEED_BASE + 4),
}

# Zipf-skewed Qwen3-30B-shaped routing (Perseus article, section 4.5).
for _s in (0.0, 0.5, 1.0, 1.5):
    _n = f"qwen3_zipf{_s:g}"
    CONFIGS[_n] = Workload(_n, N=16, T=512, H=2048, E=128, R=8, expert="identity",
                           routing="zipf", seed=SEED_BASE + 5, zipf_s=_s)

SKEW_HOT_FRACTION = 0.10     # top 10% of experts ...
SKEW_TARGET_SHARE = 0.50     # ... take about half of all assignments


def bf16_bits(a: np.ndarray) -> np.ndarray:
    """float32 array -> bf16 bit patterns (uint16), round to nearest even (torch)."""
    t = torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def _softmax64(logits: np.ndarray) -> np.ndarray:
    z = logits.astype(np.float64)
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    return p / p.sum(axis=1, keepdims=True)


def _top_r(prob: np.ndarray, R: int) -> tuple[np.ndarray, np.ndarray]:
    # stable sort of -prob: equal probabilities keep ascending expert id
    order = np.argsort(-prob, axis=1, kind="stable")[:, :R]
    chosen = np.take_along_axis(prob, order, axis=1)
    w = chosen / chosen.sum(axis=1, keepdims=True)
    return order.astype(np.int32), w.astype(np.float32)


def hot_experts(E: int, seed: int) -> np.ndarray:
    """The hot set of the skewed recipe: first ceil(0.1 E) of a seeded permutation."""
    rng = np.random.Generator(np.random.PCG64(seed + 7919))
    return rng.permutation(E)[: math.ceil(SKEW_HOT_FRACTION * E)]


def hot_share(logits: np.ndarray, hot: np.ndarray, bias: float, R: int) -> float:
    """Fraction of top-R assignments that land on ``hot`` when its logits get ``bias``."""
    z = logits.astype(np.float64).copy()
    z[:, hot] += bias
    top, _ = _top_r(_softmax64(z), R)
    return float(np.isin(top, hot).mean())


@functools.lru_cache(maxsize=None)
def skew_bias(E: int, R: int, seed: int) -> float:
    """Logit bias that gives the hot set ~50% of top-R assignments.

    Found by bisection on a separate seeded calibration sample of 8192 tokens.
    """
    rng = np.random.Generator(np.random.PCG64(seed + 104729))
    cal = rng.standard_normal((8192, E), dtype=np.float32)
    hot = hot_experts(E, seed)
    lo, hi = 0.0, 8.0
    for _ in range(40):
        mid = 0.5 * (lo + hi)
        if hot_share(cal, hot, mid, R) < SKEW_TARGET_SHARE:
            lo = mid
        else:
            hi = mid
    return 0.5 * (lo + hi)


def zipf_popularity(E: int, s: float) -> np.ndarray:
    """Zipf law over expert popularity rank k = 1..E: p_k proportional to k^-s."""
    k = np.arange(1, E + 1, dtype=np.float64)
    p = k ** (-s)
    return p / p.sum()


def generate(w: Workload, with_x: bool = True) -> dict[str, np.ndarray]:
    """Synthesise one layer's inputs.

    Returns ``x`` uint16 bf16 bits [N,T,H], ``topk_idx`` int32 [N,T,R],
    ``topk_w`` float32 [N,T,R].
    """
    out: dict[str, np.ndarray] = {}
    if with_x:
        xrng = np.random.Generator(np.random.PCG64(w.seed))
        x32 = xrng.standard_normal((w.N * w.T, w.H), dtype=np.float32)
        out["x"] = bf16_bits(x32).reshape(w.N, w.T, w.H)
        del x32
    # routing draws come from a stream of their own, so with_x=False
    # yields the same routing as with_x=True
    rng = np.random.Generator(np.random.PCG64(w.seed + 1_000_003))
    logits = rng.standard_normal((w.N * w.T, w.E), dtype=np.float32)
    if w.routing == "softmax":
        idx, wt = _top_r(_softmax64(logits), w.R)
    elif w.routing == "skew":
        z = logits.astype(np.float64)
        z[:, hot_experts(w.E, w.seed)] += skew_bias(w.E, w.R, w.seed)
        idx, wt = _top_r(_softmax64(z), w.R)
    elif w.routing == "worst":
        # every token's top-R is experts 0..R-1, all hosted by rank 0
        if w.R > w.Er:
            raise ValueError("worst-case routing needs R <= E/N")
        idx = np.tile(np.arange(w.R, dtype=np.int32), (w.N * w.T, 1))
        p = _softmax64(logits[:, : w.R])
        wt = (p / p.sum(axis=1, keepdims=True)).astype(np.float32)
    elif w.routing == "zipf":
        # Expert popularity follows a Zipf law over a seeded popularity order;
        # each token draws R distinct experts without replacement in proportion
        # to popularity (Gumbel-top-R), weights from a softmax of N(0,1) logits
        # over the chosen R.
        perm = np.random.Generator(np.random.PCG64(w.seed + 31337)).permutation(w.E)
        pop = np.empty(w.E)
        pop[perm] = zipf_popularity(w.E, w.zipf_s)
        g = rng.gumbel(size=(w.N * w.T, w.E))
        key = np.log(pop)[None, :] + g
        idx = np.argsort(-key, axis=1, kind="stable")[:, : w.R].astype(np.int32)
        sel = np.take_along_axis(logits.astype(np.float64), idx, axis=1)
        p = _softmax64(sel)
        wt = p.astype(np.float32)
    else:
        raise ValueError(f"unknown routing {w.routing!r}")
    out["topk_idx"] = np.ascontiguousarray(idx.reshape(w.N, w.T, w.R), dtype=np.int32)
    out["topk_w"] = np.ascontiguousarray(wt.reshape(w.N, w.T, w.R), dtype=np.float32)
    return out
