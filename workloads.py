"""Seeded synthetic inputs for the five MoE routing / dispatch workloads.

This module only draws random inputs; it holds none of the routing or
planning arithmetic.  Both the CPU oracle (through the tests) and the GPU
library (through the tests, the smoke check and the benchmark) consume what
it returns, so the two sides always see identical inputs.

Recipe (numpy ``default_rng(seed)``, draws in this order):
  1. logits  float32[N, E] ~ N(0, 1)
  2. shaping of the logits, by workload:
     - ``zipf``: a random permutation of the experts gives expert e the
       popularity rank rank(e) in 1..E; -1.1 * ln(rank(e)) is added to every
       logit of expert e, so softmax popularity falls off as rank^-1.1
       (Zipf s = 1.1, hot experts at random positions);
     - ``rank_boost``: each token draws one logical rank uniformly and +1.5
       is added to the logits of all E/R experts of that rank, so many tokens
       send two or more pairs to the same rank.
  3. correction bias float32[E] ~ U(-0.1, 0.1) (sigmoid workloads only)
  4. hidden states: float32 ~ N(0, 1) drawn in blocks of 4096 rows, each
     rounded to bf16 (nearest, ties to even, by torch's conversion) and
     returned as uint16 bit patterns [N, H].
"""
from __future__ import annotations

import dataclasses

import numpy as np

__all__ = ["Workload", "CONFIGS", "get", "make_inputs", "make_x_bits", "random_topk"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    N: int           # tokens
    E: int           # experts
    K: int           # experts per token
    R: int           # logical ranks (E/R experts each)
    H: int           # hidden size (bf16 elements per row)
    alignment: int   # per-expert row alignment of the permuted buffer
    scoring: int     # 0 softmax, 1 sigmoid
    renormalize: bool
    n_group: int = 1
    topk_group: int = 1
    routed_scaling: float = 1.0
    bias: bool = False
    shaping: str = "none"   # none | zipf | rank_boost

    def describe(self) -> str:
        return ("%s: N=%d E=%d K=%d R=%d H=%d a=%d %s%s" % (
            self.name, self.N, self.E, self.K, self.R, self.H, self.alignment,
            "softmax" if self.scoring == 0 else "sigmoid",
            "" if self.n_group == 1 else " group-limited %d/%d" % (self.topk_group, self.n_group)))


CONFIGS = {
    "tiny": Workload("tiny", N=256, E=8, K=2, R=2, H=128, alignment=8,
                     scoring=0, renormalize=True),
    "mixtral": Workload("mixtral", N=16384, E=8, K=2, R=4, H=4096, alignment=16,
                        scoring=0, renormalize=True),
    "qwen3": Workload("qwen3", N=8192, E=128, K=8, R=8, H=2048, alignment=128,
                      scoring=0, renormalize=True, shaping="zipf"),
    "dsv3": Workload("dsv3", N=4096, E=256, K=8, R=8, H=7168, alignment=128,
                     scoring=1, renormalize=True, n_group=8, topk_group=4,
                     routed_scaling=2.5, bias=True),
    "large": Workload("large", N=65536, E=256, K=8, R=64, H=7168, alignment=128,
                      scoring=1, renormalize=True, n_group=8, topk_group=4,
                      routed_scaling=2.5, bias=True, shaping="rank_boost"),
}


def get(name: str) -> Workload:
    return CONFIGS[name]


def _bf16_bits(a32: np.ndarray) -> np.ndarray:
    import torch
    t = torch.from_numpy(np.ascontiguousarray(a32, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def make_x_bits(rng: np.random.Generator, N: int, H: int, block: int = 4096) -> np.ndarray:
    out = np.empty((N, H), dtype=np.uint16)
    for r0 in range(0, N, block):
        r1 = min(N, r0 + block)
        out[r0:r1] = _bf16_bits(rng.standard_normal((r1 - r0, H), dtype=np.float32))
    return out


def make_inputs(w: Workload | str, seed: int = 0, with_x: bool = True, N: int | None = None):
    """Return dict(logits, bias, x_bits) for a workload (optionally with N overridden)."""
    if isinstance(w, str):
        w = CONFIGS[w]
    n = w.N if N is None else N
    rng = np.random.default_rng(seed)
    logits = rng.standard_normal((n, w.E), dtype=np.float32)
    if w.shaping == "zipf":
        perm = rng.permutation(w.E)
        rank = np.empty(w.E, dtype=np.float64)
        rank[perm] = np.arange(1, w.E + 1, dtype=np.float64)
        logits += (-1.1 * np.log(rank)).astype(np.float32)[None, :]
    elif w.shaping == "rank_boost":
        epn = w.E // w.R
        chosen = rng.integers(0, w.R, size=n)
        cols = chosen[:, None] * epn + np.arange(epn)[None, :]
        np.add.at(logits, (np.arange(n)[:, None], cols), np.float32(1.5))
    bias = rng.uniform(-0.1, 0.1, size=w.E).astype(np.float32) if w.bias else None
    x = make_x_bits(rng, n, w.H) if with_x else None
    return {"logits": logits, "bias": bias, "x_bits": x}


def random_topk(rng: np.random.Generator, N: int, E: int, K: int, distinct: bool = True,
                hot: float = 0.0) -> np.ndarray:
    """Random expert ids int32[N, K]; distinct per token like a router's output.

    ``hot`` > 0 sends that fraction of the first picks to expert 0 (skew)."""
    if distinct:
        keys = rng.random((N, E))
        if hot > 0:
            keys[:, 0] += (rng.random(N) < hot) * 2.0
        ids = np.argsort(-keys, axis=1, kind="stable")[:, :K]
    else:
        ids = rng.integers(0, E, size=(N, K))
    return np.ascontiguousarray(ids, dtype=np.int32)
