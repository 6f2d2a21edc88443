"""Plain restatement of FCP's block distributor and work list (oracle; test infrastructure).

Source: "Unleashing Scalable Context Parallelism for Foundation Models
Pre-Training via FCP" (arXiv 2605.08524):

* Section 3.3 (problem formulation): a sharding function G maps each sequence to
  blocks, an assignment function M maps each block to a worker, and a worker's
  load is the sum of f(B) over its blocks.
* Section 4.1 (block distributor, sharding policy): every sequence is cut into
  fixed-size blocks; sequences shorter than the block size are packed into the
  fewest blocks and computed with the varlen kernel interface.
* Section 3.2 / Figure 4 (Zig-Zag): for a causal sequence, block i is paired with
  the block at the mirrored position so that every pair carries equal compute.
* Sections 3.2 and 4.1 (assignment policy): a variant of Longest Processing Time
  greedily gives each block to the least-loaded worker, under a strict cap on the
  tokens a worker holds.
* Section 4.2 (bottom-up coalescer): consecutive block-level sub-stages of a
  worker can be merged into one execution stage of up to c blocks.
* Section 4.2 (block-level pipelining, congestion-free solver, Figures 7 and 8) and
  Section 4.3 (local computation first): the execution stage of each work item.

Readings where the pages are silent (Appendix A.1 is not on the pages):

1. Blocks: a sequence of length L >= b gives ceil(L/b) blocks aligned at its
   start; a short final block stays its own block. L == b is one full block.
2. Packing of L < b: First-Fit-Decreasing by length (ties: lower sequence index),
   bins in creation order, segments in insertion order. FFD is not always the
   minimum; the pages' "minimal number of blocks" is bin packing.
3. Block order: unpacked sequences in input order (blocks in order), then bins.
4. Zig-Zag partner of block j of a causal sequence of k blocks: k-1-j (0-based);
   the middle block of an odd k and every packed or full-mask block has none (-1).
   The pages' "i-th with (2N-i)-th" is off by one under either indexing.
5. Cost f(B): unmasked score pairs whose query lies in B. Causal segment at
   offset s of length l: s*l + l(l+1)/2; full mask: l * L_seq. The efficiency
   factor is constant at a fixed block size and is dropped.
6. LPT: blocks by cost descending, ties by block id ascending; each goes to the
   least-loaded worker among those whose tokens + len(B) <= cap, ties by lowest
   worker id. No such worker: capacity error. Default cap: b * ceil(K / N).
7. Work list, per worker, per owned Q-block (ascending id), per segment: an
   unpacked causal block j of a sequence pairs with KV blocks 0..j of it (j is the
   causal diagonal, the rest full); full mask pairs with every block of the
   sequence; a packed segment pairs with itself.
8. Runs (coalescing): consecutive items of one worker with the same query range,
   at most c per run; each run owns one partial (O, LSE) slot.
"""
from __future__ import annotations

from typing import Dict, List, Optional, Sequence

FULL = 0
CAUSAL_DIAG = 1


class CapacityError(Exception):
    """No worker can take a block without exceeding the token cap."""


def segment_cost(start: int, length: int, seq_len: int, causal: bool) -> int:
    """Unmasked score pairs of the queries at positions [start, start+length) of a sequence."""
    if causal:
        return sum(i + 1 for i in range(start, start + length))
    return length * seq_len


def partition(seqlens: Sequence[int], block_size: int, causal: bool) -> Dict[str, list]:
    """Sharding G with packing and Zig-Zag partners.

    Returns blocks as tuples (first_seg, n_segs, tokens, seq, seq_block_idx,
    seq_nblocks, zz_partner, cost) -- seq is -1 for a packed block -- and segments
    as tuples (seq, start_in_seq, length, tok0), tok0 being the segment's offset in
    the packed token order of the input.
    """
    if block_size <= 0:
        raise ValueError("block size must be positive")
    if any(L < 0 for L in seqlens):
        raise ValueError("negative sequence length")
    seq_start = [0] * len(seqlens)
    acc = 0
    for i, L in enumerate(seqlens):
        seq_start[i] = acc
        acc += L

    blocks: List[tuple] = []
    segs: List[tuple] = []
    # unpacked sequences, in input order
    for i, L in enumerate(seqlens):
        if L < block_size:
            continue
        k = -(-L // block_size)
        for j in range(k):
            start = j * block_size
            ln = min(block_size, L - start)
            partner = (k - 1 - j) if (causal and k - 1 - j != j) else -1
            cost = segment_cost(start, ln, L, causal)
            blocks.append((len(segs), 1, ln, i, j, k, partner, cost))
            segs.append((i, start, ln, seq_start[i] + start))

    # short sequences: first-fit-decreasing into bins of block_size tokens
    short = [i for i, L in enumerate(seqlens) if 0 < L < block_size]
    short.sort(key=lambda i: (-seqlens[i], i))
    bins: List[List[int]] = []
    room: List[int] = []
    for i in short:
        for bi in range(len(bins)):
            if room[bi] >= seqlens[i]:
                bins[bi].append(i)
                room[bi] -= seqlens[i]
                break
        else:
            bins.append([i])
            room.append(block_size - seqlens[i])
    for members in bins:
        first = len(segs)
        tokens = 0
        cost = 0
        for i in members:
            L = seqlens[i]
            segs.append((i, 0, L, seq_start[i]))
            tokens += L
            cost += segment_cost(0, L, L, causal)
        blocks.append((first, len(members), tokens, -1, 0, 1, -1, cost))
    return {"blocks": blocks, "segs": segs, "seqlens": list(seqlens), "block_size": block_size,
            "causal": causal}


def default_cap(n_blocks: int, n_workers: int, block_size: int) -> int:
    return block_size * (-(-n_blocks // n_workers)) if n_blocks else block_size


def distribute(part: Dict[str, list], n_workers: int, token_cap: Optional[int] = None) -> Dict[str, list]:
    """Assignment M (LPT under a token cap) and the work list of (Q, KV, mask) items.

    Returns worker_of_block, load (sum of block costs per worker), tokens per
    worker, the cap used, and items as tuples
    (worker, q_block, kv_block, q_tok0, q_len, kv_tok0, kv_len, mask).
    """
    if n_workers <= 0:
        raise ValueError("need at least one worker")
    blocks, segs = part["blocks"], part["segs"]
    K = len(blocks)
    cap = token_cap if (token_cap is not None and token_cap > 0) else default_cap(K, n_workers, part["block_size"])
    order = sorted(range(K), key=lambda b: (-blocks[b][7], b))
    load = [0] * n_workers
    tokens = [0] * n_workers
    owner = [-1] * K
    for b in order:
        need = blocks[b][2]
        best = -1
        for w in range(n_workers):
            if tokens[w] + need > cap:
                continue
            if best < 0 or load[w] < load[best]:
                best = w
        if best < 0:
            raise CapacityError(f"block {b} ({need} tokens) fits no worker under cap {cap}")
        owner[b] = best
        load[best] += blocks[b][7]
        tokens[best] += need

    out = distribute_fixed(part, owner, n_workers)
    out["cap"] = cap
    return out



def coalesce(items: Sequence[tuple], degree: int) -> List[tuple]:
    """Runs of at most `degree` consecutive items of one worker sharing a query range.

    Returns runs as tuples (worker, q_block, q_tok0, q_len, item_begin, item_end,
    part_row0, stage), part_row0 being the run's first row in the partial-result buffer
    (runs laid end to end, q_len rows each) and stage 0 (no pipeline schedule).
    """
    if degree <= 0:
        raise ValueError("coalesce degree must be positive")
    runs: List[tuple] = []
    row = 0
    i = 0
    while i < len(items):
        w, qb, _, qtok, qlen = items[i][:5]
        j = i + 1
        while (j < len(items) and j - i < degree and items[j][0] == w
               and items[j][3] == qtok and items[j][4] == qlen):
            j += 1
        runs.append((w, qb, qtok, qlen, i, j, row, 0))
        row += qlen
        i = j
    return runs


def imbalance(load: Sequence[int]) -> float:
    """(max(load) - mean(load)) / max(load), the pages' imbalance ratio (Section 6.2)."""
    mx = max(load)
    if mx == 0:
        return 0.0
    return (mx - sum(load) / len(load)) / mx


def transfers(part: Dict[str, list], dist: Dict[str, list]) -> List[tuple]:
    """Edges of the data-flow bipartite graph (Section 4.2, congestion-free solver; Figure 8):
    one (kv_block, src, dst, tokens) per distinct (KV block, receiving worker) where the
    block's owner src differs from the worker dst whose Q block attends to it, in work-list
    order (a worker pulls each remote block once)."""
    owner = dist["worker_of_block"]
    seen = set()
    out = []
    for (w, qb, kb, *_rest) in dist["items"]:
        src = owner[kb]
        if src == w or (kb, w) in seen:
            continue
        seen.add((kb, w))
        out.append((kb, src, w, part["blocks"][kb][2]))
    return out


def max_degree(edges: Sequence[tuple], n_workers: int) -> int:
    """Delta: the largest number of blocks one worker sends or receives. By Lemma 1 a
    congestion-free sub-stage is a matching, by Lemma 2 the busiest worker needs Delta of
    them, and a bipartite multigraph's edges split into exactly Delta matchings."""
    if not edges:
        return 0
    send = [0] * n_workers
    recv = [0] * n_workers
    for e in edges:
        send[e[1]] += 1
        recv[e[2]] += 1
    return max(max(send), max(recv))


def stages_are_matchings(edges: Sequence[tuple], stage: Sequence[int], n_stages: int) -> bool:
    """Every edge has a stage in [0, n_stages) and no worker sends or receives two blocks in
    the same stage."""
    sent, got = set(), set()
    for e, s in zip(edges, stage):
        if not 0 <= s < n_stages:
            return False
        if (s, e[1]) in sent or (s, e[2]) in got:
            return False
        sent.add((s, e[1]))
        got.add((s, e[2]))
    return True


def solve_stages(edges: Sequence[tuple], n_workers: int) -> List[int]:
    """A split of the data-flow edges into Delta matchings (Section 4.2, congestion-free
    solver: the optimum number of sub-stages is Delta, Lemmas 1 and 2), by Koenig's
    edge-colouring argument for bipartite multigraphs: colour the edges one at a time; for
    edge (u, v) take a colour a free at sender u and a colour b free at receiver v (both
    exist, each has fewer than Delta coloured edges); if a is not free at v, swap a and b
    along the path from v that alternates b, a, b, ... edges (it cannot reach u), after
    which a is free at both ends. Colour c is sub-stage c. Returns the stage of every edge."""
    delta = max_degree(edges, n_workers)
    # colour -> edge at each endpoint; senders are ("s", w), receivers ("r", w)
    at: Dict[tuple, Dict[int, int]] = {}
    stage = [-1] * len(edges)

    def ends(i):
        return ("s", edges[i][1]), ("r", edges[i][2])

    for i in range(len(edges)):
        u, v = ends(i)
        at.setdefault(u, {})
        at.setdefault(v, {})
        a = min(c for c in range(delta) if c not in at[u])
        b = min(c for c in range(delta) if c not in at[v])
        if a in at[v]:
            # the a/b alternating path from v, starting with its a-edge
            path = []
            node, colour = v, a
            while colour in at[node]:
                e = at[node][colour]
                path.append(e)
                x, y = ends(e)
                node = y if node == x else x
                colour = b if colour == a else a
            for e in path:
                x, y = ends(e)
                del at[x][stage[e]]
                del at[y][stage[e]]
            for e in path:
                x, y = ends(e)
                stage[e] = b if stage[e] == a else a
                at[x][stage[e]] = e
                at[y][stage[e]] = e
        stage[i] = a
        at[u][a] = i
        at[v][a] = i
    return stage


def schedule(part: Dict[str, list], dist: Dict[str, list], edges: Sequence[tuple], stage: Sequence[int],
             degree: int) -> Dict[str, list]:
    """The block-level pipeline with the bottom-up coalescer (Section 4.2, Figure 7; local
    computation first, Section 4.3). A work item runs in execution stage 0 when its worker
    owns the KV block, else in stage 1 + s // degree, s being the sub-stage in which the
    block reaches the worker (`degree` consecutive sub-stages merged into one stage). Each
    worker's items are taken stage by stage, keeping work-list order inside a stage. A run
    is a maximal group of consecutive items of one worker, query range and stage; the runs
    of one query range take consecutive q_len-row slices of the partial buffer, ranges in
    order of first appearance.

    Returns {"items", "item_stage", "runs" (as `coalesce`'s tuples, stage filled),
    "n_stages", "partial_rows"}."""
    if degree <= 0:
        raise ValueError("coalesce degree must be positive")
    owner = dist["worker_of_block"]
    arrive = {(e[0], e[2]): s for e, s in zip(edges, stage)}
    items = list(dist["items"])
    st = []
    for it in items:
        w, kb = it[0], it[2]
        st.append(0 if owner[kb] == w else 1 + arrive[(kb, w)] // degree)
    order = sorted(range(len(items)), key=lambda i: (items[i][0], st[i], i))
    items = [items[i] for i in order]
    st = [st[i] for i in order]
    runs = []
    i = 0
    while i < len(items):
        w, qb, _, qtok, qlen = items[i][:5]
        j = i + 1
        while j < len(items) and items[j][0] == w and items[j][3] == qtok and items[j][4] == qlen and st[j] == st[i]:
            j += 1
        runs.append([w, qb, qtok, qlen, i, j, -1, st[i]])
        i = j
    ranges: Dict[tuple, List[int]] = {}
    for r, run in enumerate(runs):
        ranges.setdefault((run[2], run[3]), []).append(r)
    row = 0
    for rs in ranges.values():  # insertion order: first appearance
        for r in rs:
            runs[r][6] = row
            row += runs[r][3]
    return {"items": items, "item_stage": st, "runs": [tuple(r) for r in runs],
            "n_stages": 1 + max(st, default=0), "partial_rows": row}


def worker_order(part: Dict[str, list], dist: Dict[str, list], n_workers: int) -> List[int]:
    """The workers' token layout of the transparent reshuffle (Section 4.3): position i holds
    the input token of worker 0's blocks (ascending id, segments in order), then worker 1's..."""
    order: List[int] = []
    for w in range(n_workers):
        for b, blk in enumerate(part["blocks"]):
            if dist["worker_of_block"][b] != w:
                continue
            for si in range(blk[0], blk[0] + blk[1]):
                _, _, ln, tok0 = part["segs"][si]
                order.extend(range(tok0, tok0 + ln))
    return order


def partition_ring(seqlens: Sequence[int], n_workers: int, causal: bool) -> Dict[str, list]:
    """Ring attention's sharding and assignment (Section 3.4 "Balance-optimized", Figure 5a,
    with the Zig-Zag order of Figure 4): each sequence of length L is cut into 2N equal
    blocks, block j covering [j*L // 2N, (j+1)*L // 2N); empty blocks are dropped; worker w
    takes blocks w and 2N-1-w. Returns the partition (same tuples as `partition`) and the
    owner of every block."""
    two_n = 2 * n_workers
    blocks: List[tuple] = []
    segs: List[tuple] = []
    owner: List[int] = []
    tok0 = 0
    for i, L in enumerate(seqlens):
        grid = {}
        made = []
        for j in range(two_n):
            a, e = j * L // two_n, (j + 1) * L // two_n
            if e == a:
                continue
            grid[j] = len(blocks)
            made.append(j)
            blocks.append([len(segs), 1, e - a, i, len(made) - 1, 0, -1, segment_cost(a, e - a, L, causal)])
            segs.append((i, a, e - a, tok0 + a))
            owner.append(j if j < n_workers else two_n - 1 - j)
        for j in made:
            b = blocks[grid[j]]
            b[5] = len(made)
            partner = grid.get(two_n - 1 - j, -1)
            b[6] = partner if (causal and partner >= 0 and partner != grid[j]) else -1
        tok0 += L
    return {"blocks": [tuple(b) for b in blocks], "segs": segs, "seqlens": list(seqlens),
            "block_size": max([b[2] for b in blocks], default=1), "causal": causal, "owner": owner}


def distribute_fixed(part: Dict[str, list], owner: Sequence[int], n_workers: int) -> Dict[str, list]:
    """Loads, tokens and the work list of a partition whose owners are given (same work-list
    rule as `distribute`)."""
    blocks, segs = part["blocks"], part["segs"]
    load = [0] * n_workers
    tokens = [0] * n_workers
    for b, blk in enumerate(blocks):
        load[owner[b]] += blk[7]
        tokens[owner[b]] += blk[2]
    seq_blocks: Dict[int, List[int]] = {}
    for b, blk in enumerate(blocks):
        if blk[3] >= 0:
            seq_blocks.setdefault(blk[3], []).append(b)
    causal = part["causal"]
    items: List[tuple] = []
    for w in range(n_workers):
        for qb in range(len(blocks)):
            if owner[qb] != w:
                continue
            first, nseg, _, seq, j, _, _, _ = blocks[qb]
            for si in range(first, first + nseg):
                _, _, qlen, qtok = segs[si]
                if seq < 0:
                    items.append((w, qb, qb, qtok, qlen, qtok, qlen, CAUSAL_DIAG if causal else FULL))
                    continue
                kv_list = seq_blocks[seq][: j + 1] if causal else seq_blocks[seq]
                for kb in kv_list:
                    kseg = segs[blocks[kb][0]]
                    mask = CAUSAL_DIAG if (causal and kb == qb) else FULL
                    items.append((w, qb, kb, qtok, qlen, kseg[3], kseg[2], mask))
    return {"worker_of_block": list(owner), "load": load, "tokens": tokens, "cap": max(tokens, default=0),
            "items": items}
