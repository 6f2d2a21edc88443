"""Plan-level balance report: FCP's block distributor against the ring-attention baseline.

For a batch, both plans come from the library (fcp_partition + fcp_distribute, and
fcp_partition_ring); the figures are the pages' imbalance ratio (max - mean) / max
("Unleashing Scalable Context Parallelism for Foundation Models Pre-Training via FCP",
Section 6.2, Figure 9) over each worker's compute (unmasked score pairs), memory (tokens)
and communication (tokens of KV blocks sent plus received, from the congestion-free solver),
the number of congestion-free sub-stages, and the share of compute that sits in blocks
shorter than 2K tokens, where attention kernels lose efficiency (Section 3.1, Figure 3).
"""
from __future__ import annotations

from typing import Optional, Sequence

from . import Plan

SMALL_BLOCK_TOKENS = 2048


def imbalance(values: Sequence[int]) -> float:
    mx = max(values) if len(values) else 0
    return 0.0 if mx == 0 else (mx - sum(values) / len(values)) / mx


def plan_report(plan: Plan, kv_bytes_per_token: int = 8 * 128 * 2 * 2) -> dict:
    """Balance figures of a distributed plan; kv_bytes_per_token prices a transferred KV token
    (default: 8 KV heads x D 128 x K and V x bf16)."""
    v = plan.view()
    res = plan.solve()
    n = v["n_workers"]
    comm = [0] * n
    for kv, src, dst, stage, tokens in res["transfers"]:
        comm[int(src)] += int(tokens)
        comm[int(dst)] += int(tokens)
    blocks = v["blocks"]
    cost = [int(b[7]) for b in blocks]
    small = sum(c for b, c in zip(blocks, cost) if int(b[2]) < SMALL_BLOCK_TOKENS)
    total = sum(cost)
    sizes = sorted(int(b[2]) for b in blocks)
    return {
        "workers": n,
        "blocks": v["n_blocks"],
        "median_block_tokens": sizes[len(sizes) // 2] if sizes else 0,
        "compute_imbalance": round(imbalance([int(x) for x in v["load"]]), 6),
        "memory_imbalance": round(imbalance([int(x) for x in v["tokens"]]), 6),
        "comm_imbalance": round(imbalance(comm), 6),
        "comm_gb": round(sum(int(t[4]) for t in res["transfers"]) * kv_bytes_per_token / 1e9, 4),
        "stages": res["n_stages"],
        "small_block_compute_share": round(small / total, 6) if total else 0.0,
    }


def compare(seqlens: Sequence[int], block_size: int, n_workers: int, causal: bool,
            token_cap: Optional[int] = None) -> dict:
    """FCP (fixed blocks, LPT under the token cap) against ring (2N blocks per sequence)."""
    fcp_plan = Plan(seqlens, block_size, causal).distribute(n_workers, token_cap)
    ring_plan = Plan.ring(seqlens, n_workers, causal)
    return {"fcp": plan_report(fcp_plan), "ring": plan_report(ring_plan)}
