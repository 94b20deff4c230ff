"""Seeded synthetic workloads for the MoE dispatch/combine path.

This module only draws inputs; it holds none of the path's arithmetic. Both
the CUDA library's tests and the CPU oracle's tests take their inputs from
here, so that the two sides see identical bytes.

Recipe (shapes follow the pages' workloads: hidden size 7168 in BF16, Top-8
routing, up to 128 expert-parallel ranks):

* ``x``            -- N(0, 1) samples in binary32, rounded to bfloat16 by
                      torch's conversion; kept as uint16 bit patterns.
* ``topk_idx``     -- K distinct experts per token, drawn without replacement
                      with the Gumbel-top-K trick. ``uniform`` gives every
                      expert the same weight; ``zipf`` gives the expert at
                      position i of a seeded permutation weight 1/(i+1)^alpha,
                      which makes hot ranks and a long tail.
* masking          -- exactly floor(mask_frac * S * K) slots, chosen
                      uniformly, are set to -1.
* ``topk_weights`` -- softmax over the K slots of N(0, 1) logits (computed in
                      binary64, stored as binary32); masked slots keep their
                      weight.

Independent streams come from ``numpy.random.SeedSequence(seed).spawn(4)``:
hidden rows, expert keys, logits, and permutation + mask.
"""

from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

NUM_CHANNELS = 16
EXPERT_ALIGNMENT = 1

# name -> shape of the workload. T is tokens per source rank; S = P * T.
WORKLOADS = {
    # P=4 virtual ranks, E=16, 64 tokens per rank, H=256, Top-2, uniform.
    "tiny_p4_e16_h256": dict(P=4, E=16, T=64, H=256, K=2, routing="uniform", quant=0),
    # P=8, E=256, 4096 tokens per rank, H=7168, Top-8, uniform, BF16 payload.
    "p8_e256_t4096_h7168": dict(P=8, E=256, T=4096, H=7168, K=8, routing="uniform", quant=0),
    # Same routing, dispatch applies per-token dynamic int8 quantisation.
    "p8_e256_t4096_h7168_int8": dict(P=8, E=256, T=4096, H=7168, K=8, routing="uniform", quant=1),
    # P=128, E=256, 512 tokens per rank, Zipf(1.2) routing, 10% of slots masked.
    "p128_e256_t512_h7168_zipf": dict(P=128, E=256, T=512, H=7168, K=8, routing="zipf",
                                      zipf_alpha=1.2, mask_frac=0.1, quant=0),
    # Small-message regime: P=32, E=256, 128 tokens per rank.
    "p32_e256_t128_h7168": dict(P=32, E=256, T=128, H=7168, K=8, routing="uniform", quant=0),
    "p32_e256_t128_h4096": dict(P=32, E=256, T=128, H=4096, K=8, routing="uniform", quant=0),
    "p32_e256_t128_h2048": dict(P=32, E=256, T=128, H=2048, K=8, routing="uniform", quant=0),
    "p32_e256_t128_h1024": dict(P=32, E=256, T=128, H=1024, K=8, routing="uniform", quant=0),
}

BENCH_WORKLOAD = "p8_e256_t4096_h7168"


@dataclass
class Workload:
    name: str
    P: int
    E: int
    T: int
    H: int
    K: int
    quant: int
    C: int = NUM_CHANNELS
    expert_alignment: int = EXPERT_ALIGNMENT
    x_bits: np.ndarray | None = None      # uint16 [S, H]
    topk_idx: np.ndarray | None = None    # int32  [S, K]
    topk_weights: np.ndarray | None = None  # float32 [S, K]
    meta: dict = field(default_factory=dict)

    @property
    def S(self) -> int:
        return self.P * self.T


def _streams(seed: int):
    return [np.random.default_rng(s) for s in np.random.SeedSequence(seed).spawn(4)]


def draw_hidden(S: int, H: int, rng: np.random.Generator) -> np.ndarray:
    """N(0,1) rows rounded to bfloat16 (torch's conversion), as uint16 bits."""
    import torch

    out = np.empty((S, H), np.uint16)
    rows = max(1, (1 << 24) // max(H, 1))
    for r0 in range(0, S, rows):
        r1 = min(S, r0 + rows)
        f = rng.standard_normal((r1 - r0, H), dtype=np.float32)
        out[r0:r1] = torch.from_numpy(f).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return out


def draw_routing(S: int, E: int, K: int, rng_keys: np.random.Generator,
                 rng_perm: np.random.Generator, routing: str = "uniform",
                 zipf_alpha: float = 1.2) -> np.ndarray:
    """K distinct experts per token by Gumbel-top-K; ordered by decreasing key."""
    if K > E:
        raise ValueError("K must not exceed E")
    logw = np.zeros(E, np.float64)
    if routing == "zipf":
        perm = rng_perm.permutation(E)
        logw[perm] = -zipf_alpha * np.log(np.arange(1, E + 1, dtype=np.float64))
    elif routing != "uniform":
        raise ValueError(f"unknown routing {routing!r}")
    out = np.empty((S, K), np.int32)
    rows = max(1, (1 << 22) // E)
    for r0 in range(0, S, rows):
        r1 = min(S, r0 + rows)
        u = rng_keys.random((r1 - r0, E))
        keys = logw[None, :] - np.log(-np.log(np.clip(u, 1e-300, 1.0)))
        top = np.argpartition(-keys, K - 1, axis=1)[:, :K]
        order = np.argsort(-np.take_along_axis(keys, top, axis=1), axis=1, kind="stable")
        out[r0:r1] = np.take_along_axis(top, order, axis=1)
    return out


def draw_weights(S: int, K: int, rng: np.random.Generator) -> np.ndarray:
    logits = rng.standard_normal((S, K)).astype(np.float64)
    logits -= logits.max(axis=1, keepdims=True)
    e = np.exp(logits)
    return (e / e.sum(axis=1, keepdims=True)).astype(np.float32)


def apply_mask(topk_idx: np.ndarray, frac: float, rng: np.random.Generator) -> np.ndarray:
    if frac <= 0:
        return topk_idx
    S, K = topk_idx.shape
    m = int(np.floor(frac * S * K))
    flat = topk_idx.reshape(-1).copy()
    flat[rng.choice(S * K, size=m, replace=False)] = -1
    return flat.reshape(S, K)


def make(P: int, E: int, T: int, H: int, K: int, *, routing: str = "uniform",
         zipf_alpha: float = 1.2, mask_frac: float = 0.0, quant: int = 0, seed: int = 0,
         with_x: bool = True, name: str = "custom", C: int = NUM_CHANNELS,
         expert_alignment: int = EXPERT_ALIGNMENT) -> Workload:
    S = P * T
    rng_x, rng_keys, rng_logits, rng_perm = _streams(seed)
    idx = draw_routing(S, E, K, rng_keys, rng_perm, routing, zipf_alpha)
    idx = apply_mask(idx, mask_frac, rng_perm)
    w = draw_weights(S, K, rng_logits)
    x = draw_hidden(S, H, rng_x) if with_x else None
    return Workload(name=name, P=P, E=E, T=T, H=H, K=K, quant=quant, C=C,
                    expert_alignment=expert_alignment, x_bits=x, topk_idx=idx, topk_weights=w,
                    meta=dict(routing=routing, zipf_alpha=zipf_alpha, mask_frac=mask_frac,
                              seed=seed))


def workload(name: str, *, seed: int = 0, with_x: bool = True, T: int | None = None) -> Workload:
    """A named workload; ``T`` overrides tokens per rank (a bounded sample)."""
    cfg = dict(WORKLOADS[name])
    if T is not None:
        cfg["T"] = T
    return make(seed=seed, with_x=with_x, name=name, **cfg)
