"""Block-level pipeline and bottom-up coalescer ("Unleashing Scalable Context Parallelism for
Foundation Models Pre-Training via FCP", Section 4.2, Figures 7 and 8; local computation
first, Section 4.3).

Oracle pins: Koenig's edge colouring gives Delta matchings; a hand-worked schedule; the
partials of a schedule's runs, merged, equal whole-sequence attention. Library parity: with
the oracle's sub-stages installed (fcp_set_stages), fcp_schedule is bit-exact against the
oracle's schedule; with the library's own solver, the schedule obeys the same rule."""
import random

import numpy as np
import pytest

import workloads as W
from oracle import attention as A
from oracle import plan as P


# ---------------------------------------------------------------- oracle pins
def _random_edges(r, n, m):
    return [(i, r.randrange(n), r.randrange(n), 1) for i in range(m)]


@pytest.mark.parametrize("seed", range(30))
def test_koenig_colouring_is_delta_matchings(seed):
    r = random.Random(seed)
    n = r.randint(1, 12)
    edges = _random_edges(r, n, r.randint(0, 60))
    stage = P.solve_stages(edges, n)
    delta = P.max_degree(edges, n)
    assert P.stages_are_matchings(edges, stage, delta)
    if edges:  # the busiest worker needs every one of the Delta colours (Lemma 2)
        assert max(stage) + 1 == delta


def test_koenig_colouring_parallel_edges():
    # four blocks from worker 0 to worker 1: four distinct sub-stages
    edges = [(b, 0, 1, 1) for b in range(4)]
    assert sorted(P.solve_stages(edges, 2)) == [0, 1, 2, 3]
    # a 3-regular bipartite multigraph on 3 + 3 nodes: 3 perfect matchings
    edges = [(0, 0, 0, 1), (1, 0, 1, 1), (2, 0, 1, 1), (3, 1, 1, 1), (4, 1, 2, 1), (5, 1, 2, 1),
             (6, 2, 2, 1), (7, 2, 0, 1), (8, 2, 0, 1)]
    stage = P.solve_stages(edges, 3)
    assert P.stages_are_matchings(edges, stage, 3)
    for s in range(3):
        assert sorted(e[1] for e, x in zip(edges, stage) if x == s) == [0, 1, 2]


def test_schedule_worked_example():
    """One causal 1024-token sequence in four 256-token blocks on two workers. LPT with the
    Zig-Zag pairs gives worker 0 blocks {0, 3} and worker 1 blocks {1, 2}. Worker 0's query
    block 3 pulls KV blocks 1 and 2 from worker 1; worker 1's query blocks 1 and 2 pull KV
    block 0 from worker 0. Edges in work-list order: e0 = (kv 1, 1->0), e1 = (kv 2, 1->0),
    e2 = (kv 0, 0->1). Colouring: e0 takes 0; e1 finds 0 used at both ends and takes 1; e2
    takes 0 (Delta = 2)."""
    part = P.partition([1024], 256, True)
    dist = P.distribute(part, 2, None)
    assert dist["worker_of_block"] == [0, 1, 1, 0]
    edges = P.transfers(part, dist)
    assert [e[:3] for e in edges] == [(1, 1, 0), (2, 1, 0), (0, 0, 1)]
    stage = P.solve_stages(edges, 2)
    assert stage == [0, 1, 0]

    # degree 1: worker 0 runs (q0,kv0) (q3,kv0) (q3,kv3) locally, then (q3,kv1) in stage 1 and
    # (q3,kv2) in stage 2; worker 1 runs (q1,kv1) (q2,kv1) (q2,kv2), then (q1,kv0) (q2,kv0)
    s = P.schedule(part, dist, edges, stage, 1)
    assert [(it[0], it[1], it[2]) for it in s["items"]] == [
        (0, 0, 0), (0, 3, 0), (0, 3, 3), (0, 3, 1), (0, 3, 2),
        (1, 1, 1), (1, 2, 1), (1, 2, 2), (1, 1, 0), (1, 2, 0)]
    assert s["item_stage"] == [0, 0, 0, 1, 2, 0, 0, 0, 1, 1]
    assert s["n_stages"] == 3
    # runs (worker, q_block, item range, stage); partial rows: q0 | q3 x3 | q1 x2 | q2 x2
    assert [(r[0], r[1], r[4], r[5], r[7]) for r in s["runs"]] == [
        (0, 0, 0, 1, 0), (0, 3, 1, 3, 0), (0, 3, 3, 4, 1), (0, 3, 4, 5, 2),
        (1, 1, 5, 6, 0), (1, 2, 6, 8, 0), (1, 1, 8, 9, 1), (1, 2, 9, 10, 1)]
    assert [r[6] for r in s["runs"]] == [0, 256, 512, 768, 1024, 1536, 1280, 1792]
    assert s["partial_rows"] == 2048

    # degree 2: sub-stages 0 and 1 merge into stage 1; worker 0's two remote items share a run
    s = P.schedule(part, dist, edges, stage, 2)
    assert s["item_stage"] == [0, 0, 0, 1, 1, 0, 0, 0, 1, 1]
    assert s["n_stages"] == 2
    assert [(r[4], r[5], r[7]) for r in s["runs"]] == [
        (0, 1, 0), (1, 3, 0), (3, 5, 1), (5, 6, 0), (6, 8, 0), (8, 9, 1), (9, 10, 1)]
    assert s["partial_rows"] == 1792


def _sched_cases():
    out = [(w.seqlens, w.block_size, w.causal, w.n_workers, w.token_cap) for w in W.small_cases()]
    r = random.Random(7)
    for _ in range(20):
        b = r.choice([2, 3, 8, 64, 100])
        seqlens = [r.choice([r.randint(1, b), r.randint(1, 6 * b), 2 * b]) for _ in range(r.randint(1, 8))]
        out.append((seqlens, b, r.random() < 0.6, r.randint(1, 7), None))
    return out


@pytest.mark.parametrize("case", range(len(_sched_cases())))
@pytest.mark.parametrize("degree", [1, 2, 3, 16])
def test_schedule_invariants(case, degree):
    seqlens, b, causal, n, cap = _sched_cases()[case]
    part = P.partition(seqlens, b, causal)
    dist = P.distribute(part, n, cap)
    edges = P.transfers(part, dist)
    stage = P.solve_stages(edges, n)
    s = P.schedule(part, dist, edges, stage, degree)
    owner = dist["worker_of_block"]
    # the same items, each worker's items contiguous and stage-ordered
    assert sorted(s["items"]) == sorted(dist["items"])
    items, st = s["items"], s["item_stage"]
    for i in range(1, len(items)):
        assert (items[i - 1][0], st[i - 1]) <= (items[i][0], st[i])
    # stage 0 is exactly the local computation
    for it, x in zip(items, st):
        assert (x == 0) == (owner[it[2]] == it[0])
    # in each later stage a worker receives and sends at most `degree` distinct blocks
    recv, send = {}, {}
    for it, x in zip(items, st):
        if x:
            recv.setdefault((it[0], x), set()).add(it[2])
            send.setdefault((owner[it[2]], x), set()).add((it[2], it[0]))
    assert all(len(v) <= degree for v in recv.values())
    assert all(len(v) <= degree for v in send.values())
    delta = P.max_degree(edges, n)
    assert s["n_stages"] == 1 + -(-delta // degree)
    # runs cover the items, never cross a stage, and the rows of a range are contiguous
    assert [r[4] for r in s["runs"][1:]] == [r[5] for r in s["runs"][:-1]]
    rows = {}
    for r in s["runs"]:
        assert len({st[i] for i in range(r[4], r[5])}) == 1 and st[r[4]] == r[7]
        rows.setdefault((r[2], r[3]), []).append(r[6])
    for (tok0, qlen), r0 in rows.items():
        assert r0 == [r0[0] + k * qlen for k in range(len(r0))]
    assert s["partial_rows"] == sum(r[3] for r in s["runs"])


def _run_partial(q, k, v, items, scale):
    """fp64 softmax attention of one run: its query rows against the union of its items'
    keys, a CAUSAL_DIAG item masking key > query within the aligned block pair."""
    it0 = items[0]
    qt, ql = it0[3], it0[4]
    Hq, Hkv = q.shape[0], k.shape[0]
    cols, masks = [], []
    for it in items:
        kt, kl, mask = it[5], it[6], it[7]
        cols.append(np.arange(kt, kt + kl))
        allowed = np.ones((ql, kl), bool)
        if mask == 1:
            allowed = np.arange(kl)[None, :] <= np.arange(ql)[:, None]
        masks.append(allowed)
    cols = np.concatenate(cols)
    allowed = np.concatenate(masks, axis=1)
    o = np.zeros((Hq, ql, q.shape[2]))
    lse = np.full((Hq, ql), -np.inf)
    for h in range(Hq):
        g = h // (Hq // Hkv)
        s = q[h, qt:qt + ql] @ k[g, cols].T * scale
        s = np.where(allowed, s, -np.inf)
        m = s.max(axis=1, keepdims=True)
        ok = np.isfinite(m[:, 0])
        p = np.where(ok[:, None], np.exp(s - np.where(ok[:, None], m, 0.0)), 0.0)
        den = p.sum(axis=1)
        o[h, ok] = (p[ok] @ v[g, cols]) / den[ok, None]
        lse[h, ok] = m[ok, 0] + np.log(den[ok])
    return o, lse


@pytest.mark.parametrize("degree", [1, 2])
def test_schedule_partials_merge_to_attention(degree):
    """The pipeline reorders work only: per-run partials of the schedule, merged per query
    range (Section 2.3), give whole-sequence attention."""
    w = W.Workload("sched", [300, 513, 40, 77], 128, 4, 2, 16, 4, True)
    part = P.partition(w.seqlens, w.block_size, w.causal)
    dist = P.distribute(part, w.n_workers, None)
    edges = P.transfers(part, dist)
    s = P.schedule(part, dist, edges, P.solve_stages(edges, w.n_workers), degree)
    assert s["n_stages"] > 1
    q, k, v = (t.double().numpy() for t in W.make_qkv(w))
    scale = 1.0 / np.sqrt(w.head_dim)
    T = w.total_tokens
    po = np.zeros((w.hq, s["partial_rows"], w.head_dim))
    pl = np.full((w.hq, s["partial_rows"]), -np.inf)
    for r in s["runs"]:
        o, lse = _run_partial(q, k, v, s["items"][r[4]:r[5]], scale)
        po[:, r[6]:r[6] + r[3]] = o
        pl[:, r[6]:r[6] + r[3]] = lse
    out = np.zeros((w.hq, T, w.head_dim))
    by_range = {}
    for r in s["runs"]:
        by_range.setdefault((r[2], r[3]), []).append(r[6])
    for (tok0, qlen), r0 in by_range.items():
        rows = np.array(r0)[:, None] + np.arange(qlen)[None, :]
        mo, _ = A.lse_merge(np.moveaxis(po[:, rows], 1, 0), np.moveaxis(pl[:, rows], 1, 0))
        out[:, tok0:tok0 + qlen] = mo
    ref, _ = A.attention_forward(q, k, v, w.seqlens, True)
    assert np.abs(out - ref).max() < 1e-12


# ---------------------------------------------------------------- library parity
def _lib_vs_oracle(fcp, seqlens, b, causal, n, cap, degree):
    part = P.partition(seqlens, b, causal)
    dist = P.distribute(part, n, cap)
    edges = P.transfers(part, dist)
    stage = P.solve_stages(edges, n)
    want = P.schedule(part, dist, edges, stage, degree)
    plan = fcp.Plan(seqlens, b, causal).distribute(n, cap)
    plan.set_stages(stage)
    got_t = plan.transfers()
    assert [tuple(t[:3]) for t in got_t["transfers"]] == [e[:3] for e in edges]
    n_exec = plan.schedule(degree)
    v = plan.view()
    assert n_exec == want["n_stages"] == v["n_exec_stages"]
    assert v["coalesce"] == degree
    assert np.array_equal(v["items"], np.array(want["items"], dtype=np.int64).reshape(-1, 8))
    assert np.array_equal(v["runs"], np.array(want["runs"], dtype=np.int64).reshape(-1, 8))
    assert v["partial_rows"] == want["partial_rows"]
    plan.validate()
    return plan


@pytest.mark.parametrize("case", range(len(_sched_cases())))
@pytest.mark.parametrize("degree", [1, 3, 16])
def test_library_schedule_bit_exact(fcp, case, degree):
    seqlens, b, causal, n, cap = _sched_cases()[case]
    _lib_vs_oracle(fcp, seqlens, b, causal, n, cap, degree)


@pytest.mark.parametrize("make", [W.causal_mixed, W.long_causal, lambda: W.block_sweep(512)])
@pytest.mark.parametrize("degree", [1, 4, 16])
def test_library_schedule_bit_exact_named(fcp, make, degree):
    w = make()
    _lib_vs_oracle(fcp, w.seqlens, w.block_size, w.causal, w.n_workers, w.token_cap, degree)


@pytest.mark.parametrize("make", [W.causal_mixed, W.long_causal, lambda: W.cluster_batch(32)])
@pytest.mark.parametrize("degree", [1, 16])
def test_library_schedule_with_its_own_solver(fcp, make, degree):
    """With the library's Hopcroft-Karp sub-stages (a different valid colouring), the
    schedule follows the same rule: checked item by item against the library's transfers."""
    w = make()
    plan = fcp.Plan(w.seqlens, w.block_size, w.causal).distribute(w.n_workers, w.token_cap)
    base = plan.view()
    n_exec = plan.schedule(degree)
    t = plan.transfers()
    v = plan.view()
    owner = v["worker_of_block"]
    arrive = {(int(r[0]), int(r[2])): int(r[3]) for r in t["transfers"]}
    items = v["items"]
    stage = np.array([0 if owner[it[2]] == it[0] else 1 + arrive[(int(it[2]), int(it[0]))] // degree
                      for it in items])
    assert n_exec == 1 + -(-t["n_stages"] // degree) == stage.max() + 1
    # stable reorder of the work list by (worker, stage)
    key = sorted(range(len(base["items"])), key=lambda i: (base["items"][i][0], (
        0 if owner[base["items"][i][2]] == base["items"][i][0]
        else 1 + arrive[(int(base["items"][i][2]), int(base["items"][i][0]))] // degree), i))
    assert np.array_equal(items, base["items"][key])
    assert all(stage[r[4]:r[5]].min() == stage[r[4]:r[5]].max() == r[7] for r in v["runs"])
    plan.validate()
    # the stage-ordered forward units: unscheduling restores the work list
    plan.coalesce(1)
    assert np.array_equal(plan.view()["items"], base["items"])
    assert plan.view()["n_exec_stages"] == 1


def test_set_stages_rejects_invalid(fcp):
    plan = fcp.Plan([1024], 256, True).distribute(2)
    n = len(plan.solve()["transfers"])
    assert n == 3
    with pytest.raises(fcp.FcpError) as e:
        plan.set_stages([0, 1])  # wrong count
    assert e.value.status == 1
    with pytest.raises(fcp.FcpError) as e:
        plan.set_stages([0, 0, 1])  # worker 1 sends two blocks in sub-stage 0
    assert e.value.status == 1
    with pytest.raises(fcp.FcpError) as e:
        plan.set_stages([0, -1, 1])
    assert e.value.status == 1
    with pytest.raises(fcp.FcpError) as e:
        plan.transfers()  # left unsolved
    assert e.value.status == 5
    plan.set_stages([2, 0, 5])  # a valid, wasteful plan: 6 sub-stages
    assert plan.transfers()["n_stages"] == 6
    assert plan.schedule(2) == 4
    with pytest.raises(fcp.FcpError) as e:
        plan.schedule(0)
    assert e.value.status == 1
    undistributed = fcp.Plan([1024], 256, True)
    with pytest.raises(fcp.FcpError) as e:
        undistributed.schedule(1)
    assert e.value.status == 5


@pytest.mark.parametrize("seqlens,b,causal,n", [
    ([0, 300, 0, 5], 64, True, 3),       # empty sequences and a packed short one
    ([1024], 256, True, 1),               # one worker: every block local, one stage
    ([40, 17, 3, 60], 64, False, 4),      # packed blocks only (full mask)
    ([512, 512], 128, True, 8),           # more workers than blocks
])
@pytest.mark.parametrize("degree", [1, 1000])
def test_library_schedule_edge_cases(fcp, seqlens, b, causal, n, degree):
    plan = _lib_vs_oracle(fcp, seqlens, b, causal, n, None, degree)
    v = plan.view()
    if n == 1:
        assert v["n_exec_stages"] == 1
    if degree >= 1000:
        assert v["n_exec_stages"] <= 2
