"""Seeded synthetic workloads shared by the tests, the smoke check and the benchmark.

This module holds input generation only (shapes, seeds, value scales, chunk
sizes, row/head samples) and none of the attention arithmetic; both the CUDA
path and the CPU oracle receive the tensors it makes.

The five workloads are the long-context prefill shapes of the SLOPE prefill
engine (Moreh, "Optimizing long-context prefill on multiple older-generation
GPU nodes": context lengths 32K/64K/100K in its evaluation section; GQA and
MLA named in its context-parallelism section) and the 12K chunked-prefill size
of the SGLang pipeline-parallelism article (TL;DR: chunked prefill size 12K,
dynamic chunking with a 0.65 smoothing factor).  No model weights or prompt
datasets exist here; Q, K and V are random bf16 tensors of those shapes.

Recipe: Q, K, V are drawn in that order from one seeded torch generator as
fp32 N(0, 1), multiplied by the workload's value scale and rounded to bf16
(round-to-nearest-even).  Layout is token-major ``[S, H, d]`` (batch 1).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np

SEED_BASE = 20261202
CHUNK_12K = 12288


@dataclass(frozen=True)
class Workload:
    name: str
    S: int
    Hq: int
    Hkv: int
    dqk: int
    dv: int
    value_scale: float
    layout: str  # "zigzag" | "contiguous" | "chunked"
    n_chunks: int  # ring ranks for ring layouts; number of chunks for "chunked"
    windows: tuple = (0,)  # attention variants run on the same inputs (0 = full causal)
    index: int = 0
    chunk_factor_lo: float = 1.0  # chunked: per-chunk size factor range [lo, 1]
    extra: dict = field(default_factory=dict)

    @property
    def seed(self) -> int:
        return SEED_BASE + self.index


WORKLOADS = [
    Workload("tiny_causal_gqa_s1k", 1024, 4, 1, 64, 64, 1.0, "zigzag", 4, index=0),
    Workload("causal_gqa_s32k_zigzag8", 32768, 64, 8, 64, 64, 0.5, "zigzag", 8, index=1),
    Workload("chunked_prefill_s64k_c12k", 65536, 64, 8, 64, 64, 0.5, "chunked", 6, index=2),
    Workload("long_s100k_zigzag16_full_and_w128", 102400, 64, 8, 64, 64, 0.5, "zigzag", 16,
             windows=(0, 128), index=3),
    Workload("mla_s64k_d192_192_128_chunked_var", 65536, 128, 128, 192, 128, 0.3, "chunked", 0,
             index=4, chunk_factor_lo=0.65),
]
# Smaller case of the same shape family, for profiler captures (inputs still larger than L2).
PROFILE_WORKLOADS = [
    Workload("profile_s16k_zigzag8", 16384, 64, 8, 64, 64, 0.5, "zigzag", 8, index=5),
    Workload("profile_mla_s16k_d192_128_chunked", 16384, 128, 128, 192, 128, 0.3, "chunked", 0, index=6,
             chunk_factor_lo=0.65),
]
BY_NAME = {w.name: w for w in WORKLOADS + PROFILE_WORKLOADS}


def chunk_sizes(w: Workload) -> list[int] | None:
    """Chunk sizes for a chunked workload (None for ring layouts).

    Fixed chunks: ``12288`` each, the last one shorter.  Varying chunks (the
    MLA workload): factors f ~ U[lo, 1] from ``numpy.random.default_rng(seed)``,
    size = round(12288 * f), drawn until the sizes cover S, last clipped to S.
    """
    if w.layout != "chunked":
        return None
    sizes = []
    if w.chunk_factor_lo >= 1.0:
        left = w.S
        while left > 0:
            sizes.append(min(CHUNK_12K, left))
            left -= sizes[-1]
        return sizes
    rng = np.random.default_rng(w.seed)
    total = 0
    while total < w.S:
        f = rng.uniform(w.chunk_factor_lo, 1.0)
        c = int(round(CHUNK_12K * f))
        c = min(c, w.S - total)
        sizes.append(c)
        total += c
    return sizes


def n_chunks(w: Workload) -> int:
    cs = chunk_sizes(w)
    return len(cs) if cs is not None else w.n_chunks


def make_qkv(S, Hq, Hkv, dqk, dv, value_scale, seed, device="cpu", slab_rows=8192):
    """Seeded bf16 Q [S,Hq,dqk], K [S,Hkv,dqk], V [S,Hkv,dv] on ``device``.

    Drawn in slabs of ``slab_rows`` tokens (Q first, then K, then V) from one
    generator of that device, so that peak fp32 scratch stays bounded.
    """
    import torch

    gen = torch.Generator(device=device)
    gen.manual_seed(int(seed))

    def draw(H, d):
        t = torch.empty((S, H, d), dtype=torch.bfloat16, device=device)
        for r0 in range(0, S, slab_rows):
            r1 = min(S, r0 + slab_rows)
            x = torch.randn((r1 - r0, H, d), generator=gen, dtype=torch.float32, device=device)
            t[r0:r1] = (x * value_scale).to(torch.bfloat16)
        return t

    q = draw(Hq, dqk)
    k = draw(Hkv, dqk)
    v = draw(Hkv, dv)
    return q, k, v


def workload_qkv(w: Workload, device="cpu"):
    return make_qkv(w.S, w.Hq, w.Hkv, w.dqk, w.dv, w.value_scale, w.seed, device=device)


def segment_bounds(w: Workload) -> list[tuple[int, int]]:
    """[start, end) of every sub-chunk (ring layouts: S/(2N) or S/N tokens) or chunk."""
    cs = chunk_sizes(w)
    if cs is None:
        parts = 2 * w.n_chunks if w.layout == "zigzag" else w.n_chunks
        c = w.S // parts
        return [(i * c, (i + 1) * c) for i in range(parts)]
    out, s0 = [], 0
    for c in cs:
        out.append((s0, s0 + c))
        s0 += c
    return out


def sample_rows(w: Workload, n_random: int = 4096, edge: int = 128) -> np.ndarray:
    """Query rows checked at full size: the first and last ``edge`` rows of every
    sub-chunk/chunk, plus ``n_random`` rows drawn with the workload's seed."""
    rows = set()
    for s0, s1 in segment_bounds(w):
        rows.update(range(s0, min(s1, s0 + edge)))
        rows.update(range(max(s0, s1 - edge), s1))
    rng = np.random.default_rng(w.seed + 7)
    rows.update(int(x) for x in rng.integers(0, w.S, size=n_random))
    return np.array(sorted(rows), dtype=np.int64)


def sample_heads(w: Workload) -> list[int]:
    """Heads checked at full size: one whole KV group for GQA, two heads otherwise."""
    G = w.Hq // w.Hkv
    if G > 1:
        g = (w.seed % w.Hkv)
        return list(range(g * G, (g + 1) * G))
    return [0, w.Hq - 1]


def causal_pairs(S: int, window: int = 0) -> int:
    """Visible (query, key) pairs per head of causal attention over S tokens."""
    if window <= 0 or window >= S:
        return S * (S + 1) // 2
    return window * (window + 1) // 2 + (S - window) * window


def flops(w: Workload, window: int = 0) -> float:
    """Algorithmic FLOPs: visible pairs x Hq x 2 x (dqk + dv)."""
    return float(causal_pairs(w.S, window)) * w.Hq * 2 * (w.dqk + w.dv)
