"""The C++ host plan (fcp_partition / fcp_distribute / fcp_coalesce) is bit-exact against the
oracle's plain restatement of the block distributor, on the named workloads and on random
batches; invalid inputs return the documented status codes."""
import random

import numpy as np
import pytest

import workloads as W
from oracle import plan as P


def _compare(fcp, seqlens, b, causal, n, cap=None, c=1):
    part = P.partition(seqlens, b, causal)
    plan = fcp.Plan(seqlens, b, causal)
    v = plan.view()
    assert v["n_blocks"] == len(part["blocks"])
    if part["blocks"]:
        assert np.array_equal(v["blocks"], np.array(part["blocks"], dtype=np.int64))
        assert np.array_equal(v["segs"], np.array(part["segs"], dtype=np.int64))
    try:
        dist = P.distribute(part, n, cap)
    except P.CapacityError:
        with pytest.raises(fcp.FcpError) as e:
            plan.distribute(n, cap)
        assert e.value.status == 2
        return None
    plan.distribute(n, cap)
    if c != 1:
        plan.coalesce(c)
    v = plan.view()
    assert v["token_cap"] == dist["cap"]
    assert list(v["worker_of_block"]) == dist["worker_of_block"]
    assert list(v["load"]) == dist["load"]
    assert list(v["tokens"]) == dist["tokens"]
    assert v["n_items"] == len(dist["items"])
    if dist["items"]:
        assert np.array_equal(v["items"], np.array(dist["items"], dtype=np.int64))
    runs = P.coalesce(dist["items"], c)
    assert v["n_runs"] == len(runs)
    if runs:
        assert np.array_equal(v["runs"], np.array(runs, dtype=np.int64))
        want_run = np.zeros(len(dist["items"]), np.int64)
        for ri, r in enumerate(runs):
            want_run[r[4]:r[5]] = ri
        assert np.array_equal(v["item_run"], want_run)
    assert v["partial_rows"] == sum(r[3] for r in runs)
    assert v["total_pairs"] == sum(L * (L + 1) // 2 if causal else L * L for L in seqlens)
    plan.validate()
    return v


@pytest.mark.parametrize("make", [W.tiny_causal, W.full_mask, W.causal_mixed, W.long_causal]
                         + [lambda b=b: W.block_sweep(b) for b in W.SWEEP_BLOCK_SIZES])
@pytest.mark.parametrize("c", [1, 16])
def test_named_workloads_bit_exact(fcp, make, c):
    w = make()
    _compare(fcp, w.seqlens, w.block_size, w.causal, w.n_workers, w.token_cap, c)


@pytest.mark.parametrize("w", W.small_cases(), ids=lambda w: w.name)
def test_small_cases_bit_exact(fcp, w):
    _compare(fcp, w.seqlens, w.block_size, w.causal, w.n_workers, w.token_cap, w.coalesce)


@pytest.mark.parametrize("seed", range(40))
def test_random_batches_bit_exact(fcp, seed):
    r = random.Random(seed)
    b = r.choice([1, 2, 3, 8, 64, 100, 512])
    n_seq = r.randint(0, 12)
    seqlens = [r.choice([0, r.randint(1, b), r.randint(1, 5 * b), b, 2 * b]) for _ in range(n_seq)]
    causal = r.random() < 0.6
    n = r.randint(1, 9)
    cap = r.choice([None, None, b, 2 * b, 3 * b, 10 ** 9])
    c = r.choice([1, 2, 3, 16])
    _compare(fcp, seqlens, b, causal, n, cap, c)


def test_lpt_zigzag_in_the_library(fcp):
    for n in (1, 2, 4, 16, 32):
        plan = fcp.Plan([2 * n * 256], 256, True).distribute(n)
        v = plan.view()
        wob = v["worker_of_block"]
        assert all(wob[j] == wob[2 * n - 1 - j] for j in range(2 * n))
        assert len(set(v["load"].tolist())) == 1


def test_invalid_inputs(fcp):
    with pytest.raises(fcp.FcpError) as e:
        fcp.Plan([4, -1], 2, True)
    assert e.value.status == 1
    with pytest.raises(fcp.FcpError):
        fcp.Plan([4], 0, True)
    p = fcp.Plan([4], 2, True)
    with pytest.raises(fcp.FcpError):
        p.distribute(0)
    with pytest.raises(fcp.FcpError) as e:
        p.coalesce(2)
    assert e.value.status == 5
    with pytest.raises(fcp.FcpError) as e:
        fcp.Plan([1000, 1000], 512, True).distribute(2, 400)
    assert e.value.status == 2
    p.distribute(1)
    with pytest.raises(fcp.FcpError):
        p.coalesce(0)


def test_device_image_sizes(fcp):
    w = W.tiny_causal()
    plan = fcp.Plan(w.seqlens, w.block_size, w.causal).distribute(w.n_workers)
    assert plan.device_bytes() > 0 and plan.device_bytes() % 256 == 0
    o, l = plan.partial_sizes(w.hq, w.head_dim)
    rows = plan.view()["partial_rows"]
    assert o == w.hq * rows * w.head_dim * 4 and l == w.hq * rows * 4
    assert plan.workspace_bytes(w.hq, w.head_dim) >= w.hq * w.total_tokens * (w.head_dim + 1) * 4


def _solver_case(fcp, seqlens, b, causal, n, cap=None):
    part = P.partition(seqlens, b, causal)
    try:
        dist = P.distribute(part, n, cap)
    except P.CapacityError:
        return
    plan = fcp.Plan(seqlens, b, causal).distribute(n, cap)
    res = plan.solve()
    edges = P.transfers(part, dist)
    got = res["transfers"]
    assert len(got) == len(edges)
    if edges:
        assert np.array_equal(got[:, [0, 1, 2, 4]], np.array(edges, dtype=np.int64))
    delta = P.max_degree(edges, n)
    assert res["n_stages"] == delta
    assert P.stages_are_matchings(edges, [int(x) for x in got[:, 3]] if len(got) else [], delta)


@pytest.mark.parametrize("make", [W.tiny_causal, W.full_mask, W.causal_mixed, W.long_causal]
                         + [lambda b=b: W.block_sweep(b) for b in W.SWEEP_BLOCK_SIZES])
def test_solver_on_named_workloads(fcp, make):
    w = make()
    _solver_case(fcp, w.seqlens, w.block_size, w.causal, w.n_workers, w.token_cap)


@pytest.mark.parametrize("seed", range(40))
def test_solver_on_random_batches(fcp, seed):
    r = random.Random(1000 + seed)
    b = r.choice([1, 2, 4, 64, 100])
    seqlens = [r.choice([r.randint(1, b), r.randint(1, 6 * b), 3 * b]) for _ in range(r.randint(1, 10))]
    _solver_case(fcp, seqlens, b, r.random() < 0.6, r.randint(1, 12))


def test_solver_state_errors(fcp):
    p = fcp.Plan([100], 10, True)
    with pytest.raises(fcp.FcpError) as e:
        p.solve()
    assert e.value.status == 5
    p.distribute(1)  # one worker: nothing moves
    res = p.solve()
    assert res["n_stages"] == 0 and len(res["transfers"]) == 0


@pytest.mark.parametrize("seed", range(25))
def test_ring_plan_bit_exact(fcp, seed):
    r = random.Random(2000 + seed)
    n = r.randint(1, 9)
    seqlens = [r.choice([0, r.randint(1, 3 * n), r.randint(1, 500)]) for _ in range(r.randint(1, 8))]
    causal = r.random() < 0.6
    part = P.partition_ring(seqlens, n, causal)
    dist = P.distribute_fixed(part, part["owner"], n)
    plan = fcp.Plan.ring(seqlens, n, causal).validate()
    v = plan.view()
    assert v["n_blocks"] == len(part["blocks"])
    if part["blocks"]:
        assert np.array_equal(v["blocks"], np.array(part["blocks"], dtype=np.int64))
        assert np.array_equal(v["segs"], np.array(part["segs"], dtype=np.int64))
        assert list(v["worker_of_block"]) == part["owner"]
    assert list(v["load"]) == dist["load"] and list(v["tokens"]) == dist["tokens"]
    if dist["items"]:
        assert np.array_equal(v["items"], np.array(dist["items"], dtype=np.int64))
    assert v["token_cap"] == (max(dist["tokens"]) if dist["tokens"] else 0)
    res = plan.solve()
    edges = P.transfers(part, dist)
    assert res["n_stages"] == P.max_degree(edges, n)


def test_validate_cluster_plan_and_state_errors(fcp):
    """The validator accepts the cluster-scale plan (256 workers x 32K tokens) in every form the
    library builds (distributed, coalesced, scheduled), and refuses an undistributed plan."""
    w = W.cluster_batch()
    plan = fcp.Plan(w.seqlens, w.block_size, w.causal)
    with pytest.raises(fcp.FcpError) as e:
        plan.validate()
    assert e.value.status == 5 and "not distributed" in str(e.value) + fcp.lib().fcp_last_error().decode()
    plan.distribute(w.n_workers).validate()
    plan.coalesce(16).validate()
    plan.schedule(16)
    plan.validate()
