"""Shared helpers of the GPU parity tests: run the CUDA path through the C ABI on a workload
and compare against the float64 oracle, in full or on sampled rows.

Tolerances. Forward (fixed by the target): O max-abs <= 2e-2 and mean-abs <= 2e-3 against
the oracle, LSE max-abs <= 1e-3. Backward (derived from bf16 arithmetic): the outputs are
bf16, whose rounding alone leaves a mean relative error of about 0.7 * 2^-9 = 1.4e-3 (the
error is uniform on +-ulp/2 and ulp/|x| runs over (2^-8, 2^-7]); the kernels also round P and dS to
bf16 before the gradient MMAs and form Di from the bf16 O. The tests require, per tensor,
max-abs <= 2e-2 * max(1, max|ref|) and mean-abs <= 5e-3 * mean|ref| + 1e-5 (the absolute
floor covers gradients that cancel to exactly zero, e.g. dQ of a one-token sequence, where
the kernel returns rounding noise of order u * |dP|). Every comparison is recorded, so a run
reports how much of each bound it used (tests/conftest.py prints the largest share).
"""
from __future__ import annotations

import os

import numpy as np
import torch

import workloads as W
from oracle import attention as A

O_MAX, O_MEAN, LSE_MAX = 2e-2, 2e-3, 1e-3
G_MAX_REL, G_MEAN_REL, G_MEAN_ABS = 2e-2, 5e-3, 1e-5

# Every comparison appends (test, where, tensor, max err, max bound, mean err, mean bound),
# so that a run can report how much of each bound the observed errors use.
RECORD: list = []


def _record(where, name, emax, bmax, emean=None, bmean=None):
    test = os.environ.get("PYTEST_CURRENT_TEST", "").split(" ")[0]
    RECORD.append((test, where, name, float(emax), float(bmax),
                   None if emean is None else float(emean), None if bmean is None else float(bmean)))


def run_path(fcp, w: W.Workload, coalesce=None, backward=None, device="cuda", pipeline=None, bwd_band=None):
    backward = w.backward if backward is None else backward
    dev = torch.device(device)
    q, k, v = W.make_qkv(w, device=dev)
    do = W.make_dout(w, device=dev) if backward else None
    att = fcp.FcpAttention(w.seqlens, w.block_size, w.causal, w.n_workers, w.hq, w.hkv, w.head_dim,
                           token_cap=w.token_cap, coalesce=coalesce or w.coalesce, device=dev, backward=backward,
                           pipeline=pipeline, bwd_band=bwd_band)
    o, lse = att.forward(q, k, v)
    grads = att.backward(q, k, v, o, lse, do) if backward else None
    torch.cuda.synchronize()
    att.check_device_error()
    return dict(att=att, q=q, k=k, v=v, do=do, o=o, lse=lse, grads=grads)


def np64(t):
    return t.detach().double().cpu().numpy()


def check_forward(o, lse, ro, rl, where=""):
    e = np.abs(o - ro)
    le = np.abs(lse - rl)
    _record(where, "o", e.max(), O_MAX, e.mean(), O_MEAN)
    _record(where, "lse", le.max(), LSE_MAX)
    assert e.max() <= O_MAX and e.mean() <= O_MEAN, f"{where} O max {e.max():.3e} mean {e.mean():.3e}"
    assert le.max() <= LSE_MAX, f"{where} LSE max {le.max():.3e}"


def grad_bounds(ref_absmax: float, ref_absmean: float):
    """(max-abs bound, mean-abs bound) of a gradient tensor with the given reference scale."""
    return G_MAX_REL * max(1.0, ref_absmax), G_MEAN_REL * ref_absmean + G_MEAN_ABS


def check_grad(name, got, ref, where="", extra_mean=0.0):
    """extra_mean: a derived allowance added to the mean bound (see test_extreme_scores)."""
    e = np.abs(got - ref)
    bmax, bmean = grad_bounds(np.abs(ref).max(), np.abs(ref).mean())
    bmean += extra_mean
    _record(where, name, e.max(), bmax, e.mean(), bmean)
    assert e.max() <= bmax, f"{where} {name} max {e.max():.3e} (bound {bmax:.3e})"
    assert e.mean() <= bmean, f"{where} {name} mean {e.mean():.3e} (bound {bmean:.3e}) vs mean|ref| " \
                              f"{np.abs(ref).mean():.3e}"


def check_stats(name, stat, where=""):
    """Bounds on the statistics [max |err|, sum |err|, sum |ref|, count, max |ref|] that the
    oracle pool returns for one tensor: the forward bounds for "o" and "lse", the gradient
    bounds otherwise."""
    emax, esum, rsum, n, rmax = stat
    emean, rmean = esum / max(1, n), rsum / max(1, n)
    if name == "o":
        bmax, bmean = O_MAX, O_MEAN
    elif name == "lse":
        bmax, bmean = LSE_MAX, None
    else:
        bmax, bmean = grad_bounds(rmax, rmean)
    _record(where, name, emax, bmax, emean if bmean is not None else None, bmean)
    assert emax <= bmax, f"{where} {name} max {emax:.3e} (bound {bmax:.3e})"
    if bmean is not None:
        assert emean <= bmean, f"{where} {name} mean {emean:.3e} (bound {bmean:.3e})"


def sample_rows(L: int, n: int, rng: np.random.Generator):
    """n distinct positions of a length-L sequence, always including the first and last."""
    if L <= n:
        return np.arange(L)
    mid = rng.choice(np.arange(1, L - 1), size=n - 2, replace=False)
    return np.sort(np.concatenate([[0, L - 1], mid]))


def sampled_forward(r, w: W.Workload, rows_per_seq: int, seed: int = 0, chunk: int = 16):
    """Check O and LSE of sampled query rows of every sequence against the oracle."""
    rng = np.random.default_rng(seed)
    G = w.hq // w.hkv
    a = 0
    for L in w.seqlens:
        if L == 0:
            continue
        rows = sample_rows(L, rows_per_seq, rng)
        for g in range(w.hkv):
            hs = slice(g * G, (g + 1) * G)
            for c0 in range(0, len(rows), chunk):
                rr = rows[c0:c0 + chunk]
                kend = int(rr.max()) + 1 if w.causal else L
                qr = r["q"][hs, a + rr]
                ro, rl = A.attention_rows(qr, r["k"][g, a:a + kend], r["v"][g, a:a + kend], rr, w.causal)
                check_forward(np64(r["o"][hs, a + rr]), np64(r["lse"][hs, a + rr]), ro, rl,
                              f"seq@{a} rows {rr[:3]}..")
        a += L


def sampled_backward(r, w: W.Workload, rows_per_seq: int, kv_tail: int, seed: int = 1, chunk: int = 16):
    """dQ on sampled query rows; dK and dV on the last kv_tail key rows of each sequence (under
    a causal mask only the query rows after them contribute, so the oracle cost stays small)."""
    rng = np.random.default_rng(seed)
    G = w.hq // w.hkv
    dq, dk, dv = r["grads"]
    a = 0
    for L in w.seqlens:
        if L == 0:
            continue
        rows = sample_rows(L, rows_per_seq, rng)
        for g in range(w.hkv):
            hs = slice(g * G, (g + 1) * G)
            for c0 in range(0, len(rows), chunk):
                rr = rows[c0:c0 + chunk]
                kend = int(rr.max()) + 1 if w.causal else L
                rdq = A.attention_dq_rows(r["q"][hs, a + rr], r["do"][hs, a + rr], r["k"][g, a:a + kend],
                                          r["v"][g, a:a + kend], rr, w.causal)
                check_grad("dq", np64(dq[hs, a + rr]), rdq, f"seq@{a}")
            if w.causal:
                kv_rows = np.arange(max(0, L - kv_tail), L)
                first = int(kv_rows.min())
                rdk, rdv = A.attention_dkv_rows(r["q"][hs, a + first:a + L], r["do"][hs, a + first:a + L],
                                                r["k"][g, a:a + L], r["v"][g, a:a + L], kv_rows, True,
                                                q_offset=first)
                check_grad("dk", np64(dk[g, a + kv_rows]), rdk, f"seq@{a}")
                check_grad("dv", np64(dv[g, a + kv_rows]), rdv, f"seq@{a}")
        a += L
