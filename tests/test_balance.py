"""Balance report (FCP vs ring baseline): figures agree with the oracle's plans, and the
pages' qualitative claims hold on their kind of batch."""
import pytest

import workloads as W
from oracle import plan as P


def _oracle_comm(part, dist, n):
    comm = [0] * n
    for kv, src, dst, tokens in P.transfers(part, dist):
        comm[src] += tokens
        comm[dst] += tokens
    return comm


@pytest.mark.parametrize("make", [W.tiny_causal, W.causal_mixed, W.full_mask])
def test_report_matches_oracle(fcp, make):
    from context_parallelism_fcp_gb300 import balance

    w = make()
    rep = balance.compare(w.seqlens, w.block_size, w.n_workers, w.causal, w.token_cap)
    part = P.partition(w.seqlens, w.block_size, w.causal)
    dist = P.distribute(part, w.n_workers, w.token_cap)
    f = rep["fcp"]
    assert f["compute_imbalance"] == pytest.approx(P.imbalance(dist["load"]), abs=1e-6)
    assert f["memory_imbalance"] == pytest.approx(P.imbalance(dist["tokens"]), abs=1e-6)
    assert f["comm_imbalance"] == pytest.approx(P.imbalance(_oracle_comm(part, dist, w.n_workers)), abs=1e-6)
    assert f["stages"] == P.max_degree(P.transfers(part, dist), w.n_workers)
    rpart = P.partition_ring(w.seqlens, w.n_workers, w.causal)
    rdist = P.distribute_fixed(rpart, rpart["owner"], w.n_workers)
    r = rep["ring"]
    assert r["compute_imbalance"] == pytest.approx(P.imbalance(rdist["load"]), abs=1e-6)
    assert r["comm_imbalance"] == pytest.approx(P.imbalance(_oracle_comm(rpart, rdist, w.n_workers)), abs=1e-6)


def test_pages_claims_on_a_long_tailed_batch(fcp):
    """On a long-tailed causal batch (Section 2.1) FCP keeps compute and memory balanced
    (Figure 9: < 5%) with far less of its compute in blocks below 2K tokens than ring
    (Section 3.1: over-sharding of short sequences), which balances by construction."""
    from context_parallelism_fcp_gb300 import balance

    w = W.cluster_batch(n_workers=32, tokens_per_worker=32768, seed=3)
    rep = balance.compare(w.seqlens, w.block_size, w.n_workers, w.causal)
    assert rep["fcp"]["compute_imbalance"] < 0.05
    assert rep["ring"]["compute_imbalance"] < 0.05
    assert rep["fcp"]["small_block_compute_share"] < 0.5 * rep["ring"]["small_block_compute_share"]
