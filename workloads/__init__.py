"""Seeded synthetic workloads for block-wise variable-length attention.

This module is shared by the CUDA path's tests/benchmark and by the oracle's
tests. It holds only input generation: sequence-length draws, tensor draws and
the named workload presets. It contains none of the method's arithmetic (no
partitioning, no assignment, no attention), so that the oracle and the CUDA
path stay independent.

Length distributions follow the pages' description of the training corpus
(long-tailed, roughly lognormal, up to 512K tokens; "Unleashing Scalable Context
Parallelism for Foundation Models Pre-Training via FCP", Section 2.1, Figure 2).
The internal traces themselves are not available; the lognormal draws below
stand in for them.
"""
from __future__ import annotations

from dataclasses import dataclass, field
from typing import List, Optional

import numpy as np

__all__ = [
    "Workload",
    "tiny_causal",
    "full_mask",
    "causal_mixed",
    "long_causal",
    "block_sweep",
    "small_cases",
    "cluster_batch",
    "make_qkv",
    "make_dout",
    "make_partials",
]


@dataclass
class Workload:
    """A named batch: sequence lengths, block size, head shape, workers."""

    name: str
    seqlens: List[int]
    block_size: int
    hq: int
    hkv: int
    head_dim: int
    n_workers: int
    causal: bool
    token_cap: Optional[int] = None  # None: the planner's default cap
    std: float = 1.0  # standard deviation of Q/K/V draws
    backward: bool = True
    seed: int = 0
    coalesce: int = 16
    extra: dict = field(default_factory=dict)

    @property
    def total_tokens(self) -> int:
        return int(sum(self.seqlens))


def tiny_causal() -> Workload:
    """3 causal sequences (300/1024/1800 tokens), 512-token blocks, 4/2 heads, D=64, 4 workers."""
    return Workload("tiny causal", [300, 1024, 1800], 512, 4, 2, 64, 4, True)


def _full_mask_lengths(seed: int, n: int = 16, total: int = 65536) -> List[int]:
    """16 lengths ~ lognormal(ln 4096, 1.0), clipped to [128, 32768], rescaled to `total`.

    Rescaling floors each length; the remainder goes to the longest (lowest index on ties).
    """
    rng = np.random.default_rng(seed)
    x = np.clip(rng.lognormal(mean=np.log(4096.0), sigma=1.0, size=n), 128.0, 32768.0)
    lens = np.floor(x * (total / x.sum())).astype(np.int64)
    lens[int(np.argmax(lens))] += total - int(lens.sum())
    return [int(v) for v in lens]


def full_mask(seed: int = 0) -> Workload:
    """16 lognormal sequences, 65536 tokens, full (non-causal) mask, 1024-token blocks, 64/8 heads, D=128."""
    return Workload("full mask", _full_mask_lengths(seed), 1024, 64, 8, 128, 8, False,
                    backward=False, seed=seed)


def _mixed_lengths(seed: int, budget: int = 32768, outlier: int = 32768) -> List[int]:
    """lognormal(ln 2048, 1.5) lengths clipped to [64, 65536] drawn until `budget` tokens.

    The draw that crosses the budget is truncated to fit (the packer rule of the
    forum post "Another View on Context Parallel for LLMs", Computational
    Simulation); one `outlier`-token sequence is appended.
    """
    rng = np.random.default_rng(seed)
    lens: List[int] = []
    total = 0
    while total < budget:
        v = int(np.clip(rng.lognormal(mean=np.log(2048.0), sigma=1.5), 64.0, 65536.0))
        if total + v > budget:
            v = budget - total
        lens.append(v)
        total += v
    lens.append(outlier)
    return lens


def causal_mixed(seed: int = 0) -> Workload:
    """Lognormal short/long mix plus a 32768-token outlier, 65536 tokens, 4096-token blocks, 16 workers."""
    return Workload("causal mixed", _mixed_lengths(seed), 4096, 64, 8, 128, 16, True, seed=seed)


def long_causal() -> Workload:
    """One 524288-token causal sequence in 64 blocks of 8192 (2N blocks, N=32), inputs N(0, 0.5)."""
    return Workload("long causal", [524288], 8192, 64, 8, 128, 32, True, token_cap=16384, std=0.5)


def block_sweep(block_size: int) -> Workload:
    """One 32768-token causal sequence at the given block size, N = blocks/2 workers (zig-zag)."""
    nblocks = 32768 // block_size
    return Workload(f"sweep b={block_size}", [32768], block_size, 64, 8, 128, max(1, nblocks // 2), True,
                    token_cap=2 * block_size)


SWEEP_BLOCK_SIZES = (512, 1024, 2048, 4096, 8192)


def cluster_batch(n_workers: int = 256, tokens_per_worker: int = 32768, seed: int = 0) -> Workload:
    """A cluster-scale batch in the pages' evaluation setting (Section 6.1: 32K tokens per GPU,
    causal, 4K blocks, lengths long-tailed up to 512K): lognormal(ln 8192, 1.5) lengths
    clipped to [128, 524288], drawn until n_workers * tokens_per_worker tokens (the last draw
    truncated). Used for plan-level measurements (solver, balance), not for kernels."""
    rng = np.random.default_rng(seed)
    total = n_workers * tokens_per_worker
    lens: List[int] = []
    t = 0
    while t < total:
        v = int(np.clip(rng.lognormal(mean=np.log(8192.0), sigma=1.5), 128.0, 524288.0))
        v = min(v, total - t)
        lens.append(v)
        t += v
    return Workload(f"cluster {n_workers}x{tokens_per_worker}", lens, 4096, 64, 8, 128, n_workers, True,
                    backward=False, seed=seed)


def small_cases() -> List[Workload]:
    """Small batches whose full oracle runs in seconds but that still span several tiles,
    ragged tails, packed short sequences, both masks and D in {64, 128}."""
    return [
        tiny_causal(),
        Workload("small full d128", [700, 129, 1500, 64], 512, 8, 2, 128, 3, False),
        Workload("small causal d128 gqa8", [1000, 2300, 77, 200, 1], 1024, 16, 2, 128, 5, True, coalesce=2),
        Workload("small causal c1", [1537, 255, 256], 256, 4, 1, 64, 3, True, coalesce=1),
        Workload("small causal mha", [640, 190], 256, 3, 3, 64, 2, True),
    ]


def make_qkv(w: Workload, device="cpu", seed: Optional[int] = None):
    """Q [Hq,T,D], K and V [Hkv,T,D] in bf16, entries ~ N(0, std^2), from a seeded generator."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(w.seed if seed is None else seed)
    T = w.total_tokens
    out = []
    for heads in (w.hq, w.hkv, w.hkv):
        t = torch.randn((heads, T, w.head_dim), generator=g, device=device, dtype=torch.float32)
        out.append((t * w.std).to(torch.bfloat16))
    return tuple(out)


def make_dout(w: Workload, device="cpu", seed: Optional[int] = None):
    """dO [Hq,T,D] in bf16, entries ~ N(0, 1), from a seeded generator distinct from make_qkv's."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed((w.seed if seed is None else seed) + 1_000_003)
    t = torch.randn((w.hq, w.total_tokens, w.head_dim), generator=g, device=device, dtype=torch.float32)
    return t.to(torch.bfloat16)


def make_partials(n_parts: int, hq: int, rows: int, head_dim: int, seed: int = 0, device="cpu",
                  neg_inf_frac: float = 0.0):
    """Random partial outputs [n_parts, Hq, rows, D] (fp32) and log-sum-exps [n_parts, Hq, rows]
    (fp32, spread over [-4, 12)), with an optional fraction of -inf entries."""
    import torch

    g = torch.Generator(device=device)
    g.manual_seed(seed)
    o = torch.randn((n_parts, hq, rows, head_dim), generator=g, device=device, dtype=torch.float32)
    lse = torch.rand((n_parts, hq, rows), generator=g, device=device, dtype=torch.float32) * 16.0 - 4.0
    if neg_inf_frac > 0:
        m = torch.rand((n_parts, hq, rows), generator=g, device=device) < neg_inf_frac
        lse = torch.where(m, torch.full_like(lse, float("-inf")), lse)
    return o, lse
