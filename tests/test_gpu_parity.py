"""GPU parity: the CUDA path (through the C ABI) against the float64 oracle.

Small batches are compared element by element (all heads, all tokens, all outputs); the
full-size workloads, in the launch configuration the benchmark times, on sampled rows.
"""
import numpy as np
import pytest
import torch

import workloads as W
from oracle import attention as A
from oracle import plan as P
from tests import oracle_pool as OP
from tests import parity_util as U

pytestmark = pytest.mark.gpu


@pytest.fixture(autouse=True)
def _sync():
    yield
    torch.cuda.synchronize()


@pytest.mark.parametrize("w", W.small_cases(), ids=lambda w: w.name)
def test_forward_and_backward_small(fcp, w):
    r = U.run_path(fcp, w)
    ro, rl = A.attention_forward(r["q"], r["k"], r["v"], w.seqlens, w.causal)
    U.check_forward(U.np64(r["o"]), U.np64(r["lse"]), ro, rl, w.name)
    rdq, rdk, rdv = A.attention_backward(r["q"], r["k"], r["v"], r["do"], w.seqlens, w.causal)
    for name, got, ref in zip(("dq", "dk", "dv"), r["grads"], (rdq, rdk, rdv)):
        U.check_grad(name, U.np64(got), ref, w.name)


@pytest.mark.parametrize("band", [64, 192, 512])
@pytest.mark.parametrize("w", W.small_cases(), ids=lambda w: w.name)
def test_backward_in_query_bands_small(fcp, w, band):
    """The backward run as one launch per query band (dK/dV summed over the bands in float32)
    against the oracle, element by element; bands of one step, of a ragged 3 steps and of
    several key tiles."""
    r = U.run_path(fcp, w, bwd_band=band)
    n, rows = r["att"].plan.bwd_bands()
    assert rows == band and n == -(-w.total_tokens // band)
    rdq, rdk, rdv = A.attention_backward(r["q"], r["k"], r["v"], r["do"], w.seqlens, w.causal)
    for name, got, ref in zip(("dq", "dk", "dv"), r["grads"], (rdq, rdk, rdv)):
        U.check_grad(name, U.np64(got), ref, f"{w.name} band {band}")


@pytest.mark.parametrize("c", [1, 2, 16])
def test_coalesce_degree_does_not_change_the_result(fcp, c):
    w = W.Workload("mixed small", [1500, 40, 700, 2600], 512, 8, 2, 128, 3, True)
    r = U.run_path(fcp, w, coalesce=c)
    ro, rl = A.attention_forward(r["q"], r["k"], r["v"], w.seqlens, w.causal)
    U.check_forward(U.np64(r["o"]), U.np64(r["lse"]), ro, rl, f"c={c}")


def _merge_expected(w, part_o, part_lse, coalesce):
    """Oracle merge of the partial buffers, using the oracle plan's runs (bit-identical to the
    library's plan, which the CPU tests pin)."""
    part = P.partition(w.seqlens, w.block_size, w.causal)
    dist = P.distribute(part, w.n_workers, w.token_cap)
    runs = P.coalesce(dist["items"], coalesce)
    T = w.total_tokens
    po = part_o.double().cpu().numpy()
    pl = part_lse.double().cpu().numpy()
    o = np.zeros((w.hq, T, w.head_dim))
    lse = np.full((w.hq, T), -np.inf)
    by_range = {}
    for rn in runs:
        by_range.setdefault((rn[2], rn[3]), []).append(rn[6])
    for (tok0, qlen), row0s in by_range.items():
        rows = np.array(row0s)[:, None] + np.arange(qlen)[None, :]  # [S, qlen]
        mo, ml = A.lse_merge(np.moveaxis(po[:, rows], 1, 0), np.moveaxis(pl[:, rows], 1, 0))
        o[:, tok0:tok0 + qlen] = mo
        lse[:, tok0:tok0 + qlen] = ml
    return o, lse


@pytest.mark.parametrize("head_dim", [64, 128])
@pytest.mark.parametrize("neg_inf", [0.0, 0.3])
@pytest.mark.parametrize("seqlens,coalesce", [([1000, 300, 2049, 17], 2), ([2304, 40, 3], 1), ([260], 1),
                                              ([770], 1)],
                         ids=["few partials", "many partials", "tail 4x2", "tail 2x4"])
def test_merge_kernel_matches_oracle_merge(fcp, head_dim, neg_inf, seqlens, coalesce):
    """Partials of up to 9 runs per row: the second case puts 36 partials on the 4 rows one
    warp merges, which takes the kernel's general path. The tail cases end the batch inside
    a warp's 8 rows with exactly 8 partials on the valid rows (4 rows x 2, 2 rows x 4), which
    must not be taken for one partial per row."""
    w = W.Workload("merge", seqlens, 256, 4, 2, head_dim, 3, True)
    att = fcp.FcpAttention(w.seqlens, w.block_size, w.causal, w.n_workers, w.hq, w.hkv, w.head_dim,
                           coalesce=coalesce, backward=False)
    rows = att.part_o.shape[1]
    o_p, l_p = W.make_partials(1, w.hq, rows, head_dim, seed=3, device="cuda", neg_inf_frac=neg_inf)
    att.part_o.copy_(o_p[0])
    att.part_lse.copy_(l_p[0])
    o = torch.empty((w.hq, w.total_tokens, head_dim), dtype=torch.bfloat16, device="cuda")
    lse = torch.empty((w.hq, w.total_tokens), dtype=torch.float32, device="cuda")
    fcp.block_attn_merge(att.plan, att.d_plan, att.part_o, att.part_lse, o, lse)
    torch.cuda.synchronize()
    eo, el = _merge_expected(w, att.part_o, att.part_lse, coalesce)
    got = U.np64(o)
    # bf16 output rounding: |err| <= 2^-8 |x| (+ float32 accumulation)
    assert np.all(np.abs(got - eo) <= 2.0 ** -8 * np.abs(eo) + 1e-5)
    gl = U.np64(lse)
    fin = np.isfinite(el)
    assert np.array_equal(np.isfinite(gl), fin)
    assert np.abs(gl[fin] - el[fin]).max() <= 1e-5 * max(1.0, np.abs(el[fin]).max())
    assert np.all(got[:, ~fin.all(axis=0)][~np.isfinite(el[:, ~fin.all(axis=0)])] == 0)


@pytest.mark.parametrize("head_dim", [64, 128])
def test_bwd_prologue_matches_oracle(fcp, head_dim):
    w = W.Workload("prologue", [777, 64], 256, 4, 2, head_dim, 2, True)
    plan = fcp.Plan(w.seqlens, w.block_size, w.causal).distribute(2)
    g = torch.Generator(device="cuda").manual_seed(5)
    o = torch.randn((4, w.total_tokens, head_dim), generator=g, device="cuda").to(torch.bfloat16)
    do = torch.randn((4, w.total_tokens, head_dim), generator=g, device="cuda").to(torch.bfloat16)
    di = torch.empty((4, w.total_tokens), dtype=torch.float32, device="cuda")
    acc = torch.full((4, w.total_tokens, head_dim), 7.0, dtype=torch.float32, device="cuda")
    fcp.block_attn_bwd_prologue(plan, o, do, di, acc)
    torch.cuda.synchronize()
    ref = A.rowsum_do_o(do, o)
    assert np.abs(U.np64(di) - ref).max() <= 1e-5 * max(1.0, np.abs(ref).max())
    assert torch.count_nonzero(acc).item() == 0


def test_edge_cases(fcp):
    # one token, lengths at and around the block size, packed singles, both masks
    for seqlens, b, causal in (([1], 128, True), ([128, 129, 127], 128, True), ([1, 1, 1, 1], 2, False),
                               ([256], 128, False), ([3, 700], 256, True)):
        w = W.Workload("edge", seqlens, b, 4, 2, 64, 2, causal)
        r = U.run_path(fcp, w)
        ro, rl = A.attention_forward(r["q"], r["k"], r["v"], w.seqlens, w.causal)
        U.check_forward(U.np64(r["o"]), U.np64(r["lse"]), ro, rl, str(seqlens))
        rdq, rdk, rdv = A.attention_backward(r["q"], r["k"], r["v"], r["do"], w.seqlens, w.causal)
        for name, got, ref in zip(("dq", "dk", "dv"), r["grads"], (rdq, rdk, rdv)):
            U.check_grad(name, U.np64(got), ref, str(seqlens))


@pytest.mark.parametrize("hq,hkv,head_dim", [(6, 2, 64), (6, 2, 128), (5, 1, 128), (1, 1, 64)],
                         ids=["group3 d64", "group3 d128", "group5 d128", "one head"])
def test_odd_head_groups(fcp, hq, hkv, head_dim):
    """Odd group sizes leave the last head pair of a KV group with one real head (the second
    is computed and not stored); a single head has no pair at all."""
    w = W.Workload("odd groups", [900, 130, 2100], 512, hq, hkv, head_dim, 3, True, coalesce=2)
    r = U.run_path(fcp, w)
    ro, rl = A.attention_forward(r["q"], r["k"], r["v"], w.seqlens, w.causal)
    U.check_forward(U.np64(r["o"]), U.np64(r["lse"]), ro, rl, w.name)
    rdq, rdk, rdv = A.attention_backward(r["q"], r["k"], r["v"], r["do"], w.seqlens, w.causal)
    for name, got, ref in zip(("dq", "dk", "dv"), r["grads"], (rdq, rdk, rdv)):
        U.check_grad(name, U.np64(got), ref, w.name)


def test_empty_batch_is_a_no_op(fcp):
    att = fcp.FcpAttention([0, 0], 64, True, 2, 4, 2, 64)
    q = torch.empty((4, 0, 64), dtype=torch.bfloat16, device="cuda")
    k = torch.empty((2, 0, 64), dtype=torch.bfloat16, device="cuda")
    o, lse = att.forward(q, k, k)
    dq, dk, dv = att.backward(q, k, k, o, lse, q)
    torch.cuda.synchronize()
    assert o.numel() == 0 and dq.numel() == 0
    att.check_device_error()


# ------------------------------------------------------------------ full-size workloads
def test_full_mask_sampled(fcp):
    w = W.full_mask()
    r = U.run_path(fcp, w)
    U.sampled_forward(r, w, rows_per_seq=24)


_RANGE_ROWS = 4096  # query rows per oracle task


def test_causal_mixed_all_rows(fcp):
    """The causal mixed batch (lognormal lengths plus a 32768-token outlier, 65536 tokens, 4096-
    token blocks, 16 workers, coalesce 16) in the benchmark's launch configuration.

    * O and LSE of every query row of every head, and dQ of every query row of the outlier,
      against the oracle's per-row helpers, split into (sequence, KV-head group, 4096-row
      range) tasks over a spawned process pool;
    * dQ, dK and dV of every row of every other sequence against the oracle's whole-group
      gradient;
    * dK and dV of the outlier's last 48 key rows (only the query tail after them
      contributes; its early keys are covered at full accumulation length by
      test_backward_long_accumulation_all_key_rows)."""
    w = W.causal_mixed()
    r = U.run_path(fcp, w)
    G = w.hq // w.hkv
    cpu = {n: r[n].detach().cpu() for n in ("q", "k", "v", "do", "o", "lse")}
    dq_t, dk_t, dv_t = (t.detach().cpu() for t in r["grads"])
    outlier = int(np.argmax(w.seqlens))
    starts = np.concatenate([[0], np.cumsum(w.seqlens)[:-1]]).astype(int)
    f = lambda t: t.float().numpy()  # noqa: E731

    # (sequence, group, row range) jobs, the costliest (last rows of the longest sequence) first
    # so that the pool stays balanced; their arrays are cut only when the pool takes them
    jobs = sorted(((r1 * r1 - r0 * r0, s, g, r0, r1)
                   for s, L in enumerate(w.seqlens) for g in range(w.hkv)
                   for r0 in range(0, L, _RANGE_ROWS) for r1 in [min(L, r0 + _RANGE_ROWS)]), reverse=True)

    def row_args():
        for _, s, g, r0, r1 in jobs:
            a, hs, with_dq = starts[s], slice(g * G, (g + 1) * G), s == outlier
            yield (f(cpu["q"][hs, a + r0:a + r1]), f(cpu["k"][g, a:a + r1]), f(cpu["v"][g, a:a + r1]),
                   f(cpu["do"][hs, a + r0:a + r1]) if with_dq else None,
                   f(cpu["o"][hs, a + r0:a + r1]), f(cpu["lse"][hs, a + r0:a + r1]),
                   f(dq_t[hs, a + r0:a + r1]) if with_dq else None, r0, True)

    short = [(s, g) for s in range(len(w.seqlens)) if s != outlier for g in range(w.hkv)]

    def bwd_args():
        for s, g in short:
            a, L = starts[s], w.seqlens[s]
            hs = slice(g * G, (g + 1) * G)
            yield (f(cpu["q"][hs, a:a + L]), f(cpu["k"][g, a:a + L]), f(cpu["v"][g, a:a + L]),
                   f(cpu["do"][hs, a:a + L]), True)

    with OP.pool(len(jobs)) as p:
        stats = p.imap(OP.rows_task, row_args())
        grads = p.imap(OP.group_backward_task, bwd_args())
        for (s, g), (rdq, rdk, rdv) in zip(short, grads):
            a, L = starts[s], w.seqlens[s]
            hs = slice(g * G, (g + 1) * G)
            where = f"seq {s} ({L} tokens) group {g}"
            U.check_grad("dq", U.np64(dq_t[hs, a:a + L]), rdq, where)
            U.check_grad("dk", U.np64(dk_t[g, a:a + L]), rdk, where)
            U.check_grad("dv", U.np64(dv_t[g, a:a + L]), rdv, where)
        stats = list(stats)
    keys = [(s, g) for _, s, g, _, _ in jobs]
    total = {}
    for key, st in zip(keys, stats):
        agg = total.setdefault(key, {})
        for name, x in st.items():
            y = agg.setdefault(name, [0.0, 0.0, 0.0, 0, 0.0])
            y[0], y[1], y[2], y[3], y[4] = max(y[0], x[0]), y[1] + x[1], y[2] + x[2], y[3] + x[3], max(y[4], x[4])
    assert len(total) == len(w.seqlens) * w.hkv
    for (s, g), agg in sorted(total.items()):
        for name, st in agg.items():
            U.check_stats(name, st, f"seq {s} ({w.seqlens[s]} tokens) group {g}")
    # the outlier's last key rows
    a, L = starts[outlier], w.seqlens[outlier]
    kv_rows = np.arange(L - 48, L)
    for g in range(w.hkv):
        hs = slice(g * G, (g + 1) * G)
        rdk, rdv = A.attention_dkv_rows(r["q"][hs, a + L - 48:a + L], r["do"][hs, a + L - 48:a + L],
                                        r["k"][g, a:a + L], r["v"][g, a:a + L], kv_rows, True, q_offset=L - 48)
        U.check_grad("dk", U.np64(dk_t[g, a + kv_rows]), rdk, f"outlier group {g}")
        U.check_grad("dv", U.np64(dv_t[g, a + kv_rows]), rdv, f"outlier group {g}")


_LONG_ACC = {}


@pytest.mark.parametrize("b,c,band,head_dim,causal", [(4096, 16, 0, 128, True), (1024, 1, 0, 128, True),
                                                      (4096, 16, 2048, 128, True), (4096, 16, 0, 64, True),
                                                      (4096, 16, 0, 128, False)],
                         ids=["b4096 c16", "b1024 c1", "b4096 c16 bands 2048", "b4096 c16 D64", "full mask b4096 c16"])
def test_backward_long_accumulation_all_key_rows(fcp, b, c, band, head_dim, causal):
    """dK and dV of every key row, and dQ of every query row, of two KV-head groups of a
    16384-token causal sequence (64/8 heads, D = 128) against the oracle's whole-group
    gradient: at 4096-token blocks with coalesce degree 16 (the benchmark's launch
    configuration) and at 1024-token blocks with one partial per pair. The gradient of an
    early key sums over up to 16384 queries of each of the group's 8 heads: two thousand
    64-row steps of one backward CTA, over several query blocks and items. The third case runs
    the backward in query bands of 2048 rows (one launch per band, dK/dV summed over eight
    bands in float32). The fourth runs the head_dim 64 kernels (16/2 heads, both groups), whose
    dQ^T product reads a zero panel above the 64 channels. The fifth drops the causal mask:
    every key's gradient then sums over all 16384 queries (256 steps per head)."""
    L = 16384
    hq, hkv = (64, 8) if head_dim == 128 else (16, 2)
    w = W.Workload(f"{'causal' if causal else 'full'} 16k b={b}", [L], b, hq, hkv, head_dim, max(1, L // b // 2),
                   causal, token_cap=2 * b, coalesce=c)
    r = U.run_path(fcp, w, bwd_band=band)
    assert r["att"].plan.bwd_bands()[1] == band
    G = w.hq // w.hkv
    groups = (3, 7) if hkv == 8 else (0, 1)
    q, k, v, do = (r[n].detach().cpu() for n in ("q", "k", "v", "do"))
    # the inputs depend on the seed and the shapes only, so both block sizes share one oracle run
    fingerprint = (causal,) + tuple(float(t.double().sum()) for t in (q, k, v, do))
    if _LONG_ACC.get("inputs") != fingerprint:
        f = lambda t: t.float().numpy()  # noqa: E731
        with OP.pool(len(groups), gb_per_task=8.0) as p:
            ref = p.map(OP.group_backward_task,
                        [(f(q[g * G:(g + 1) * G]), f(k[g]), f(v[g]), f(do[g * G:(g + 1) * G]), causal)
                         for g in groups])
        _LONG_ACC.clear()
        _LONG_ACC.update(inputs=fingerprint, ref=ref)
    dq, dk, dv = r["grads"]
    for g, (rdq, rdk, rdv) in zip(groups, _LONG_ACC["ref"]):
        where = f"b={b} c={c} band={band} D={head_dim} causal={causal} group {g}"
        U.check_grad("dk", U.np64(dk[g]), rdk, where)
        U.check_grad("dv", U.np64(dv[g]), rdv, where)
        U.check_grad("dq", U.np64(dq[g * G:(g + 1) * G]), rdq, where)
        # the early keys (first 128-row key tile) and a middle tile alone, so that a fault there
        # is not averaged away by the rest of the sequence
        for lo in (0, w.total_tokens // 2):
            sl = slice(lo, lo + 128)
            U.check_grad("dk", U.np64(dk[g, sl]), rdk[sl], f"{where} keys {lo}..")
            U.check_grad("dv", U.np64(dv[g, sl]), rdv[sl], f"{where} keys {lo}..")


@pytest.mark.parametrize("b", [512, 4096])
def test_block_sweep_sampled(fcp, b):
    w = W.block_sweep(b)
    r = U.run_path(fcp, w)
    U.sampled_forward(r, w, rows_per_seq=64)
    U.sampled_backward(r, w, rows_per_seq=16, kv_tail=32)


def test_long_causal_sampled(fcp):
    """524288-token sequence: 256 seeded query rows per KV-head group (all 8 heads of the group),
    dQ on 32 of them, dK/dV on the last 32 key rows, plus the merge invariant: merging at
    coalesce degree 16 gives the same output as degree 64 (one partial per query block)."""
    w = W.long_causal()
    r = U.run_path(fcp, w)
    U.sampled_forward(r, w, rows_per_seq=256)
    U.sampled_backward(r, w, rows_per_seq=32, kv_tail=32)
    o16 = r["o"].clone()
    del r
    torch.cuda.empty_cache()
    r64 = U.run_path(fcp, w, coalesce=64, backward=False)
    assert (r64["o"].float() - o16.float()).abs().max().item() <= 2e-2


@pytest.mark.parametrize("causal", [True, False])
def test_ring_plan_through_the_kernels(fcp, causal):
    """The ring baseline's plan (2N blocks per sequence, tiny blocks for short sequences) runs
    through the same kernels and matches the oracle."""
    w = W.Workload("ring", [700, 37, 1500, 5], 256, 8, 2, 128, 4, causal)
    dev = torch.device("cuda")
    q, k, v = W.make_qkv(w, device=dev)
    do = W.make_dout(w, device=dev)
    att = fcp.FcpAttention.from_plan(fcp.Plan.ring(w.seqlens, w.n_workers, w.causal), w.hq, w.hkv, w.head_dim,
                                     device=dev)
    o, lse = att.forward(q, k, v)
    grads = att.backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    att.check_device_error()
    ro, rl = A.attention_forward(q, k, v, w.seqlens, w.causal)
    U.check_forward(U.np64(o), U.np64(lse), ro, rl, "ring")
    rdq, rdk, rdv = A.attention_backward(q, k, v, do, w.seqlens, w.causal)
    for name, got, ref in zip(("dq", "dk", "dv"), grads, (rdq, rdk, rdv)):
        U.check_grad(name, U.np64(got), ref, "ring")


@pytest.mark.parametrize("kind", ["sharp", "offset"])
@pytest.mark.parametrize("causal", [True, False])
def test_extreme_scores(fcp, kind, causal):
    """Scores far from the unit range. "sharp": Q and K ~ N(0, 2.5^2), so scores have a standard
    deviation of about 6 and each softmax row is nearly one-hot. "offset": Q and K share a
    constant component of 3 per channel, so every score is near +100, where exp() of the raw
    score overflows float32 and only the running-max subtraction keeps the result finite.
    V and dO stay N(0, 1). dQ and dK get derived allowances on top of the usual mean bound
    (_derived_allowances)."""
    w = W.Workload("extreme", [700, 1300, 90], 512, 8, 2, 128, 3, causal)
    dev = torch.device("cuda")
    g = torch.Generator(device=dev).manual_seed(23)
    T = w.total_tokens

    def draw(heads, std, shift=0.0):
        x = torch.randn((heads, T, w.head_dim), generator=g, device=dev) * std + shift
        return x.to(torch.bfloat16)

    if kind == "sharp":
        q, k = draw(w.hq, 2.5), draw(w.hkv, 2.5)
    else:
        q, k = draw(w.hq, 0.5, 3.0), draw(w.hkv, 0.5, 3.0)
    v, do = draw(w.hkv, 1.0), draw(w.hq, 1.0)
    att = fcp.FcpAttention(w.seqlens, w.block_size, w.causal, w.n_workers, w.hq, w.hkv, w.head_dim, device=dev)
    o, lse = att.forward(q, k, v)
    grads = att.backward(q, k, v, o, lse, do)
    torch.cuda.synchronize()
    att.check_device_error()
    assert torch.isfinite(o).all() and torch.isfinite(lse).all()
    ro, rl = A.attention_forward(q, k, v, w.seqlens, w.causal)
    U.check_forward(U.np64(o), U.np64(lse), ro, rl, f"{kind} causal={causal}")
    rdq, rdk, rdv = A.attention_backward(q, k, v, do, w.seqlens, w.causal)
    extra = _derived_allowances(q, k, v, do, o, ro, rl, w.seqlens, causal)
    for name, got, ref in zip(("dq", "dk", "dv"), grads, (rdq, rdk, rdv)):
        U.check_grad(name, U.np64(got), ref, f"{kind} causal={causal}", extra_mean=extra.get(name, 0.0))


def _derived_allowances(q, k, v, do, o, ro, rl, seqlens, causal):
    """Mean-error allowances for dQ and dK at extreme scores, derived from two roundings the
    kernels make by design, computed exactly or in expectation from the oracle's P.

    * Di from the bf16 output. The backward forms Di = rowsum(dO * O) from the O it is given
      (bf16), so Di_gpu - Di = sum_d dO_d (O_gpu - O)_d =: e_i exactly, and every dS_ij shifts
      by -P_ij e_i. That moves dQ_i by -scale e_i (P K)_i and dK_j by -scale sum_i P_ij e_i Q_i.
      In exact arithmetic sum_j dS_ij = 0, so K's common component (3 per channel in
      "offset") cancels out of dQ; the shift does not cancel and multiplies it, and with
      near one-hot rows ("sharp") dP - Di is itself small.
    * dS rounded to bf16 before the dQ MMA. Each rounding error is uniform on +-ulp(dS_ij)/2
      (ulp = 2^(floor(log2|x|) - 7) for bf16's 8-bit significand), so the resulting dQ error
      err_id = scale sum_j e_ij K_jd has standard deviation scale sqrt(sum_j ulp_ij^2/12 K_jd^2)
      and E|err| = sqrt(2/pi) times that; this term is taken at 1.5x its expectation (a CPU
      emulation of the rounding lands within 3% of the expectation).
    Returns {"dq": mean allowance, "dk": mean allowance}."""
    Q, K, V, DO, OG = (U.np64(x) for x in (q, k, v, do, o))
    hq, hkv, D = Q.shape[0], K.shape[0], Q.shape[2]
    G, scale = hq // hkv, 1.0 / np.sqrt(D)
    dq_di = np.zeros_like(Q)
    dq_round = np.zeros_like(Q)
    dk_di = np.zeros_like(K)
    a = 0
    for L in seqlens:
        keep = np.tri(L, dtype=bool) if causal else np.ones((L, L), dtype=bool)
        for h in range(hq):
            g = h // G
            qs, ks = Q[h, a:a + L], K[g, a:a + L]
            p = np.exp(np.where(keep, qs @ ks.T * scale, -np.inf) - rl[h, a:a + L, None])
            di = (DO[h, a:a + L] * ro[h, a:a + L]).sum(-1)
            e = (DO[h, a:a + L] * (OG[h, a:a + L] - ro[h, a:a + L])).sum(-1)
            dq_di[h, a:a + L] = np.abs(scale * e[:, None] * (p @ ks))
            dk_di[g, a:a + L] += scale * (p * e[:, None]).T @ qs
            ds = p * (DO[h, a:a + L] @ V[g, a:a + L].T - di[:, None])
            mag = np.abs(np.where(ds != 0, ds, 1.0))
            ulp = np.where(ds != 0, np.exp2(np.floor(np.log2(mag)) - 7), 0.0)
            dq_round[h, a:a + L] = scale * np.sqrt((ulp ** 2 / 12) @ (ks ** 2)) * np.sqrt(2 / np.pi)
        a += L
    return {"dq": float(dq_di.mean() + 1.5 * dq_round.mean()), "dk": float(np.abs(dk_di).mean())}
