"""Pins of the block-distributor oracle against what the pages and the mathematics fix.

* The pages' worked Zig-Zag example (Section 3.2, Figure 4) as a golden fixture.
* The closed form of the Zig-Zag pair cost for any block count and size.
* LPT over the 2N equal-length blocks of one causal sequence reproduces exactly
  the Zig-Zag pairs (an exchange/induction argument: the k-th heaviest block is
  always placed on the worker holding the k-th lightest partial sum).
* Coverage: every token in exactly one block; every unmasked (query, key) pair in
  exactly one work item, and no masked pair in any (brute force on tiny inputs).
* Packing into the fewest blocks: hand-worked First-Fit-Decreasing cases and the
  FFD guarantee FFD <= 11/9 OPT + 6/9 against a brute-force optimum.
"""
import itertools
import os

import pytest

from oracle import plan as P

GOLDEN = os.path.join(os.path.dirname(__file__), "golden", "fig4_zigzag.txt")


def _read_golden():
    meta, rows = {}, []
    with open(GOLDEN) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            if parts[0].isalpha() or "_" in parts[0]:
                meta[parts[0]] = int(parts[1])
            else:
                rows.append(tuple(int(x) for x in parts))
    return meta, rows


def test_figure4_worked_example():
    meta, rows = _read_golden()
    part = P.partition([meta["seqlen"]], meta["block_size"], causal=True)
    blocks = part["blocks"]
    assert len(blocks) == len(rows)
    for blk, (bid, tokens, pairs, partner, pair_total) in zip(blocks, rows):
        assert blk[2] == tokens and blk[7] == pairs and blk[6] == partner
        assert blk[7] + blocks[partner][7] == pair_total
    dist = P.distribute(part, meta["workers"])
    groups = {}
    for b, w in enumerate(dist["worker_of_block"]):
        groups.setdefault(w, set()).add(b)
    assert sorted(map(sorted, groups.values())) == sorted([sorted({r[0], r[3]}) for r in rows][::2])
    assert dist["load"] == [18, 18]


@pytest.mark.parametrize("k,b", [(2, 1), (4, 3), (8, 512), (64, 512), (7, 5), (5, 100)])
def test_zigzag_pair_cost_closed_form(k, b):
    """Block j of a causal sequence of k full blocks of b tokens has b^2 j + b(b+1)/2 unmasked
    pairs, so j and k-1-j together carry b^2 (k-1) + b(b+1), the same for every pair."""
    blocks = P.partition([k * b], b, causal=True)["blocks"]
    for j, blk in enumerate(blocks):
        assert blk[7] == b * b * j + b * (b + 1) // 2
        if blk[6] >= 0:
            assert blk[6] == k - 1 - j
            assert blk[7] + blocks[blk[6]][7] == b * b * (k - 1) + b * (b + 1)
    if k % 2:
        assert blocks[k // 2][6] == -1


@pytest.mark.parametrize("n", [1, 2, 3, 4, 8, 16, 32])
@pytest.mark.parametrize("b", [1, 4, 512])
@pytest.mark.parametrize("capped", [False, True])
def test_lpt_reproduces_zigzag_on_one_causal_sequence(n, b, capped):
    part = P.partition([2 * n * b], b, causal=True)
    dist = P.distribute(part, n, 2 * b if capped else 10 ** 12)
    owner = dist["worker_of_block"]
    for j in range(2 * n):
        assert owner[j] == owner[2 * n - 1 - j]
    assert len(set(dist["load"])) == 1
    assert P.imbalance(dist["load"]) == 0.0


def _tiny_cases():
    return [
        ([300, 1024, 1800], 512, True, 4),
        ([300, 1024, 1800], 512, False, 3),
        ([5, 9, 3, 2, 7, 16, 1], 4, True, 3),
        ([5, 9, 3, 2, 7, 16, 1], 4, False, 2),
        ([13, 8, 8, 0, 2], 8, True, 5),
        ([1], 3, True, 2),
    ]


@pytest.mark.parametrize("seqlens,b,causal,n", _tiny_cases())
def test_coverage_by_brute_force(seqlens, b, causal, n):
    part = P.partition(seqlens, b, causal)
    T = sum(seqlens)
    seq_id, pos = [], []
    for s, L in enumerate(seqlens):
        seq_id += [s] * L
        pos += list(range(L))
    cover = [0] * T
    for seg in part["segs"]:
        for t in range(seg[3], seg[3] + seg[2]):
            cover[t] += 1
            assert seq_id[t] == seg[0] and pos[t] == seg[1] + (t - seg[3])
    assert cover == [1] * T
    for blk in part["blocks"]:
        assert 0 < blk[2] <= b
    dist = P.distribute(part, n)
    hits = {}
    for (w, qb, kb, qt, ql, kt, kl, mask) in dist["items"]:
        assert dist["worker_of_block"][qb] == w
        for i in range(qt, qt + ql):
            for j in range(kt, kt + kl):
                if mask == P.CAUSAL_DIAG and (j - kt) > (i - qt):
                    continue
                hits[(i, j)] = hits.get((i, j), 0) + 1
    want = {(i, j) for i in range(T) for j in range(T)
            if seq_id[i] == seq_id[j] and (not causal or pos[j] <= pos[i])}
    assert set(hits) == want
    assert all(c == 1 for c in hits.values())
    # loads are the unmasked pairs owned, and add up to all of them
    assert sum(dist["load"]) == len(want)
    assert all(t <= dist["cap"] for t in dist["tokens"])


def test_tiny_workload_shape():
    part = P.partition([300, 1024, 1800], 512, True)
    assert len(part["blocks"]) == 7
    dist = P.distribute(part, 4)
    assert len(dist["items"]) == 14
    assert dist["cap"] == 512 * 2


def test_capacity_error_and_cap_respected():
    part = P.partition([1000, 1000], 512, True)
    with pytest.raises(P.CapacityError):
        P.distribute(part, 2, 400)  # no worker can hold a 512-token block
    with pytest.raises(P.CapacityError):
        P.distribute(part, 1, 1024)  # 4 blocks, 2000 tokens, cap 1024 on one worker
    dist = P.distribute(part, 2, 1024)
    assert all(t <= 1024 for t in dist["tokens"])


def test_ffd_hand_worked():
    # lengths 300, 200, 100, 500 into 512-token bins, decreasing order 500, 300, 200, 100:
    # 500 -> bin0; 300 -> bin1; 200 -> bin1 (500); 100 -> bin2 (bins 0 and 1 have 12 left)
    part = P.partition([300, 200, 100, 500], 512, causal=True)
    bins = [[part["segs"][s][0] for s in range(b[0], b[0] + b[1])] for b in part["blocks"]]
    assert bins == [[3], [0, 1], [2]]
    # ties in length keep input order; a length equal to the block size is not packed
    part = P.partition([256, 512, 256, 256], 512, causal=False)
    assert [(b[3], b[1]) for b in part["blocks"]] == [(1, 1), (-1, 2), (-1, 1)]
    bins = [[part["segs"][s][0] for s in range(b[0], b[0] + b[1])] for b in part["blocks"][1:]]
    assert bins == [[0, 2], [3]]


def _opt_bins(lens, cap):
    best = len(lens)
    for assign in itertools.product(range(len(lens)), repeat=len(lens)):
        loads = [0] * len(lens)
        for L, b in zip(lens, assign):
            loads[b] += L
        if max(loads) <= cap:
            best = min(best, len(set(assign)))
    return best


@pytest.mark.parametrize("seed", range(12))
def test_ffd_within_its_guarantee(seed):
    import random

    r = random.Random(seed)
    lens = [r.randint(1, 9) for _ in range(6)]
    part = P.partition(lens, 10, causal=True)
    n_bins = len(part["blocks"])
    opt = _opt_bins(lens, 10)
    assert opt <= n_bins <= (11 * opt + 6) / 9 + 1e-9


def test_cost_totals_match_pair_counts():
    for seqlens, causal in (([7, 3, 12], True), ([7, 3, 12], False)):
        part = P.partition(seqlens, 4, causal)
        want = sum(L * (L + 1) // 2 if causal else L * L for L in seqlens)
        assert sum(b[7] for b in part["blocks"]) == want


def test_coalesce_runs():
    part = P.partition([300, 1024, 1800], 512, True)
    items = P.distribute(part, 4)["items"]
    runs1 = P.coalesce(items, 1)
    assert [(r[4], r[5]) for r in runs1] == [(i, i + 1) for i in range(len(items))]
    for c in (2, 3, 16):
        runs = P.coalesce(items, c)
        assert runs[0][4] == 0 and runs[-1][5] == len(items)
        row = 0
        for a, b in zip(runs[:-1], runs[1:]):
            assert a[5] == b[4]
        for r in runs:
            assert 1 <= r[5] - r[4] <= c
            assert r[6] == row
            row += r[3]
            for it in items[r[4]:r[5]]:
                assert (it[0], it[3], it[4]) == (r[0], r[2], r[3])
    # q block 3 of the 1800-token sequence has 4 items; with c = 3 they split 3 + 1
    runs3 = P.coalesce(items, 3)
    assert sorted(r[5] - r[4] for r in runs3 if r[1] == 5) == [1, 3]


def test_imbalance_ratio():
    assert P.imbalance([10, 10]) == 0.0
    assert abs(P.imbalance([10, 0]) - 0.5) < 1e-15
    assert abs(P.imbalance([4, 2, 3]) - 0.25) < 1e-15


def test_invalid_arguments():
    with pytest.raises(ValueError):
        P.partition([4], 0, True)
    with pytest.raises(ValueError):
        P.partition([-1], 4, True)
    with pytest.raises(ValueError):
        P.distribute(P.partition([4], 2, True), 0)
    empty = P.partition([], 4, True)
    assert empty["blocks"] == [] and P.distribute(empty, 3)["items"] == []


def test_transfers_hand_worked():
    """One causal sequence of 4 blocks on 2 workers: Zig-Zag gives w0 = {0, 3}, w1 = {1, 2}.
    In work-list order (worker 0's items first): block 3 (w0) pulls KV 1 and KV 2 from w1;
    block 1 (w1) pulls KV 0 from w0; block 2 (w1) holds KV 1 and 2 and pulls KV 0, which w1
    already has. Worker 1 sends 2 blocks: Delta = 2."""
    part = P.partition([8], 2, True)
    dist = P.distribute(part, 2)
    assert dist["worker_of_block"] == [0, 1, 1, 0]
    edges = P.transfers(part, dist)
    assert edges == [(1, 1, 0, 2), (2, 1, 0, 2), (0, 0, 1, 2)]
    assert P.max_degree(edges, 2) == 2
    assert P.stages_are_matchings(edges, [0, 1, 0], 2)
    assert not P.stages_are_matchings(edges, [1, 1, 0], 2)  # worker 1 sends twice in stage 1


def _min_matchings(edges, n):
    """Smallest k such that the edges split into k matchings, by exhaustive search."""
    if not edges:
        return 0
    for k in range(1, len(edges) + 1):
        for assign in itertools.product(range(k), repeat=len(edges)):
            if P.stages_are_matchings([(0,) + e for e in edges], assign, k):
                return k
    return len(edges)


@pytest.mark.parametrize("seed", range(25))
def test_min_congestion_free_stages_is_max_degree(seed):
    """Lemmas 1-2 and Konig's theorem: the fewest sub-stages (matchings) covering a bipartite
    multigraph's edges equals its maximum degree -- checked by brute force on tiny graphs."""
    import random

    r = random.Random(seed)
    n = r.randint(2, 4)
    edges = [(r.randrange(n), r.randrange(n)) for _ in range(r.randint(0, 6))]
    edges = [e for e in edges if e[0] != e[1]] or edges[:0]
    assert _min_matchings(edges, n) == P.max_degree([(0,) + e for e in edges], n)


def test_every_remote_pair_has_a_transfer():
    for seqlens, b, causal, n in _tiny_cases():
        part = P.partition(seqlens, b, causal)
        dist = P.distribute(part, n)
        have = {(e[0], e[2]) for e in P.transfers(part, dist)}
        for (w, qb, kb, *_rest) in dist["items"]:
            if dist["worker_of_block"][kb] != w:
                assert (kb, w) in have


def test_worker_order_hand_worked():
    """8-token causal sequence, 2-token blocks, 2 workers: w0 holds blocks 0 and 3 (tokens
    0,1 and 6,7), w1 holds blocks 1 and 2 (tokens 2..5)."""
    part = P.partition([8], 2, True)
    dist = P.distribute(part, 2)
    assert P.worker_order(part, dist, 2) == [0, 1, 6, 7, 2, 3, 4, 5]


@pytest.mark.parametrize("seqlens,b,causal,n", _tiny_cases())
def test_worker_order_is_a_permutation(seqlens, b, causal, n):
    part = P.partition(seqlens, b, causal)
    dist = P.distribute(part, n)
    order = P.worker_order(part, dist, n)
    assert sorted(order) == list(range(sum(seqlens)))
    # contiguous per worker, in token counts equal to the worker's tokens
    sizes = dist["tokens"]
    starts = [sum(sizes[:w]) for w in range(n)]
    for w in range(n):
        chunk = order[starts[w]:starts[w] + sizes[w]]
        for t in chunk:
            seg_block = [bi for bi, blk in enumerate(part["blocks"])
                         for si in range(blk[0], blk[0] + blk[1])
                         if part["segs"][si][3] <= t < part["segs"][si][3] + part["segs"][si][2]]
            assert dist["worker_of_block"][seg_block[0]] == w


@pytest.mark.parametrize("n,b", [(1, 4), (2, 2), (4, 8), (8, 512)])
def test_ring_equals_zigzag_plan_on_one_causal_sequence(n, b):
    """On one causal sequence of 2N*b tokens, ring's 2N equal blocks with worker w holding
    blocks w and 2N-1-w is the same plan as fixed blocks of b tokens with LPT (Zig-Zag)."""
    ring = P.partition_ring([2 * n * b], n, True)
    fcp = P.partition([2 * n * b], b, True)
    assert ring["blocks"] == fcp["blocks"] and ring["segs"] == fcp["segs"]
    assert ring["owner"] == P.distribute(fcp, n)["worker_of_block"]


def test_ring_short_and_uneven_sequences():
    part = P.partition_ring([3, 10], 2, True)  # 2N = 4
    # L=3: j=0 empty, then [0,1), [1,2), [2,3); L=10: [0,2), [2,5), [5,7), [7,10)
    assert [s[1:3] for s in part["segs"]] == [(0, 1), (1, 1), (2, 1), (0, 2), (2, 3), (5, 2), (7, 3)]
    assert part["owner"] == [1, 1, 0, 0, 1, 1, 0]
    dist = P.distribute_fixed(part, part["owner"], 2)
    assert sum(dist["load"]) == 3 * 4 // 2 + 10 * 11 // 2
    assert dist["tokens"] == [1 + 2 + 3, 2 + 3 + 2]


@pytest.mark.parametrize("n", [2, 3, 8])
def test_ring_compute_is_balanced_when_divisible(n):
    part = P.partition_ring([2 * n * 5, 2 * n * 7], n, True)
    dist = P.distribute_fixed(part, part["owner"], n)
    assert len(set(dist["load"])) == 1 and len(set(dist["tokens"])) == 1
