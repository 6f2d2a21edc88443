"""Plain float64 attention over packed variable-length sequences (oracle; test infrastructure).

Definition (FCP paper, Section 2.2, attention equation, as printed in the review
of the paper): for each head, O = Softmax(Q K^T / sqrt(D) (+) M, dim=-1) V, with
Q, K, V, O of shape [H, L, D].

Readings taken where the pages are silent or garbled:

* The mask is applied as -inf on masked scores before the softmax (the printed
  elementwise product with a 0/1 mask would not mask). Causal: key j is visible
  to query i iff j <= i, positions counted within the sequence. Tokens never
  attend across sequences (varlen packing, Section 4.1).
* Grouped-query heads (Section 2.3): query head h reads KV head h // (Hq / Hkv).
* LSE is the natural-log log-sum-exp of the scaled, masked scores of a row.

Everything is computed per whole sequence: no blocks, no work list, no merge.
"""
from __future__ import annotations

import math
from typing import Iterable, Optional, Sequence, Tuple

import numpy as np

_ROW_CHUNK = 1024


def _as64(x) -> np.ndarray:
    if hasattr(x, "detach"):  # a torch tensor
        x = x.detach().to("cpu")
        import torch

        x = x.to(torch.float64).numpy()
    return np.asarray(x, dtype=np.float64)


def cu_seqlens_of(seqlens: Sequence[int]) -> np.ndarray:
    cu = np.zeros(len(seqlens) + 1, dtype=np.int64)
    cu[1:] = np.cumsum(np.asarray(seqlens, dtype=np.int64))
    return cu


def _scores(qh: np.ndarray, kg: np.ndarray, rows: np.ndarray, causal: bool, scale: float) -> np.ndarray:
    """Scaled scores of query rows `rows` (positions in the sequence) against every key of the
    sequence, with the causal mask as -inf. qh: [G, n, D] queries of those rows; kg: [L, D]."""
    s = np.matmul(qh, kg.T) * scale
    if causal:
        keys = np.arange(kg.shape[0])
        s = np.where(keys[None, None, :] > rows[None, :, None], -np.inf, s)
    return s


def _softmax_rows(s: np.ndarray) -> Tuple[np.ndarray, np.ndarray]:
    """Row softmax and natural log-sum-exp; a row with no visible key gives p = 0, lse = -inf."""
    m = s.max(axis=-1, keepdims=True)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    e = np.exp(s - m_safe)
    l = e.sum(axis=-1, keepdims=True)
    with np.errstate(divide="ignore", invalid="ignore"):
        p = np.where(l > 0, e / np.where(l > 0, l, 1.0), 0.0)
        lse = np.where(l[..., 0] > 0, m_safe[..., 0] + np.log(np.where(l[..., 0] > 0, l[..., 0], 1.0)), -np.inf)
    return p, lse


def attention_forward(q, k, v, seqlens: Sequence[int], causal: bool,
                      scale: Optional[float] = None) -> Tuple[np.ndarray, np.ndarray]:
    """O [Hq,T,D] and LSE [Hq,T] (float64) of packed sequences, computed per whole sequence."""
    q, k, v = _as64(q), _as64(k), _as64(v)
    hq, T, D = q.shape
    hkv = k.shape[0]
    assert hq % hkv == 0, "query heads must be a multiple of KV heads"
    G = hq // hkv
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    cu = cu_seqlens_of(seqlens)
    assert cu[-1] == T
    o = np.zeros((hq, T, D))
    lse = np.full((hq, T), -np.inf)
    for s in range(len(seqlens)):
        a, b = int(cu[s]), int(cu[s + 1])
        for g in range(hkv):
            hs = slice(g * G, (g + 1) * G)
            kg, vg = k[g, a:b], v[g, a:b]
            for r0 in range(a, b, _ROW_CHUNK):
                r1 = min(b, r0 + _ROW_CHUNK)
                rows = np.arange(r0 - a, r1 - a)
                p, l_ = _softmax_rows(_scores(q[hs, r0:r1], kg, rows, causal, scale))
                o[hs, r0:r1] = np.matmul(p, vg)
                lse[hs, r0:r1] = l_
    return o, lse


def attention_backward(q, k, v, do, seqlens: Sequence[int], causal: bool,
                       scale: Optional[float] = None) -> Tuple[np.ndarray, np.ndarray, np.ndarray]:
    """Exact gradient (dQ, dK, dV) of sum(O * dO) for the forward above, in float64.

    With P the softmax of the scaled masked scores: dV = P^T dO, dP = dO V^T,
    dS = P * (dP - rowsum(dO * O)), dQ = scale * dS K, dK = scale * dS^T Q. KV-head
    gradients sum over the query heads of their group.
    """
    q, k, v, do = _as64(q), _as64(k), _as64(v), _as64(do)
    hq, T, D = q.shape
    hkv = k.shape[0]
    G = hq // hkv
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    cu = cu_seqlens_of(seqlens)
    dq = np.zeros_like(q)
    dk = np.zeros_like(k)
    dv = np.zeros_like(v)
    for s in range(len(seqlens)):
        a, b = int(cu[s]), int(cu[s + 1])
        for g in range(hkv):
            hs = slice(g * G, (g + 1) * G)
            kg, vg = k[g, a:b], v[g, a:b]
            for r0 in range(a, b, _ROW_CHUNK):
                r1 = min(b, r0 + _ROW_CHUNK)
                rows = np.arange(r0 - a, r1 - a)
                p, _ = _softmax_rows(_scores(q[hs, r0:r1], kg, rows, causal, scale))
                dO = do[hs, r0:r1]
                o_rows = np.matmul(p, vg)
                di = np.sum(dO * o_rows, axis=-1)
                dp = np.matmul(dO, vg.T)
                ds = p * (dp - di[..., None])
                dv[g, a:b] += np.matmul(p.transpose(0, 2, 1), dO).sum(axis=0)
                dq[hs, r0:r1] = scale * np.matmul(ds, kg)
                dk[g, a:b] += scale * np.matmul(ds.transpose(0, 2, 1), q[hs, r0:r1]).sum(axis=0)
    return dq, dk, dv


def attention_rows(q_rows, k_seq, v_seq, rows: Iterable[int], causal: bool,
                   scale: Optional[float] = None) -> Tuple[np.ndarray, np.ndarray]:
    """O and LSE for selected query rows of ONE sequence.

    q_rows: [G, n, D] queries of the n selected rows (all heads of one KV group);
    k_seq, v_seq: [L, D] the group's keys/values of the whole sequence; rows: the
    n positions within the sequence. Returns O [G, n, D], LSE [G, n].
    """
    q_rows, k_seq, v_seq = _as64(q_rows), _as64(k_seq), _as64(v_seq)
    rows = np.asarray(list(rows), dtype=np.int64)
    D = q_rows.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    p, lse = _softmax_rows(_scores(q_rows, k_seq, rows, causal, scale))
    return np.matmul(p, v_seq), lse


def attention_dq_rows(q_rows, do_rows, k_seq, v_seq, rows: Iterable[int], causal: bool,
                      scale: Optional[float] = None) -> np.ndarray:
    """dQ for selected query rows of one sequence (each row's gradient depends on that row only)."""
    q_rows, do_rows = _as64(q_rows), _as64(do_rows)
    k_seq, v_seq = _as64(k_seq), _as64(v_seq)
    rows = np.asarray(list(rows), dtype=np.int64)
    D = q_rows.shape[-1]
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    p, _ = _softmax_rows(_scores(q_rows, k_seq, rows, causal, scale))
    o_rows = np.matmul(p, v_seq)
    di = np.sum(do_rows * o_rows, axis=-1)
    dp = np.matmul(do_rows, v_seq.T)
    ds = p * (dp - di[..., None])
    return scale * np.matmul(ds, k_seq)


def attention_dkv_rows(q_seq, do_seq, k_seq, v_seq, kv_rows: Iterable[int], causal: bool,
                       scale: Optional[float] = None, q_offset: int = 0) -> Tuple[np.ndarray, np.ndarray]:
    """dK, dV [n, D] for selected key rows of one sequence, one KV group.

    q_seq, do_seq: [G, m, D] all query heads of the group for the query positions
    q_offset .. q_offset+m-1, which must run to the end of the sequence and include every
    query that sees a selected key (causal: every position >= min(kv_rows); full mask:
    all); k_seq, v_seq: [L, D] the whole sequence. Key rows near the end of a long causal
    sequence therefore need only a short tail of queries.
    """
    q_seq, do_seq = _as64(q_seq), _as64(do_seq)
    k_seq, v_seq = _as64(k_seq), _as64(v_seq)
    kv_rows = np.asarray(list(kv_rows), dtype=np.int64)
    G, m, D = q_seq.shape
    L = k_seq.shape[0]
    assert q_offset + m == L, "query rows must run to the end of the sequence"
    assert q_offset <= (int(kv_rows.min()) if causal else 0), "missing query rows that see the keys"
    scale = 1.0 / math.sqrt(D) if scale is None else scale
    dk = np.zeros((len(kv_rows), D))
    dv = np.zeros((len(kv_rows), D))
    for r0 in range(0, m, _ROW_CHUNK):
        r1 = min(m, r0 + _ROW_CHUNK)
        rows = np.arange(q_offset + r0, q_offset + r1)
        p, _ = _softmax_rows(_scores(q_seq[:, r0:r1], k_seq, rows, causal, scale))
        dO = do_seq[:, r0:r1]
        o_rows = np.matmul(p, v_seq)
        di = np.sum(dO * o_rows, axis=-1)
        psel = p[:, :, kv_rows]  # [G, n_q, n_kv]
        dp = np.matmul(dO, v_seq[kv_rows].T)
        ds = psel * (dp - di[..., None])
        dv += np.matmul(psel.transpose(0, 2, 1), dO).sum(axis=0)
        dk += scale * np.matmul(ds.transpose(0, 2, 1), q_seq[:, r0:r1]).sum(axis=0)
    return dk, dv


def lse_merge(parts_o, parts_lse) -> Tuple[np.ndarray, np.ndarray]:
    """Associative reduction of partial attention results (FCP paper, Section 2.3).

    parts_o: [S, ..., D] partial outputs, each normalised over its own key subset;
    parts_lse: [S, ...] their natural log-sum-exps. Returns the output and LSE over
    the union of the key subsets: m = max_s lse_s, w_s = exp(lse_s - m),
    O = sum_s w_s O_s / sum_s w_s, lse = m + log sum_s w_s. Parts with lse = -inf
    carry no weight; if all are -inf the result is O = 0, lse = -inf.
    """
    o = _as64(parts_o)
    lse = _as64(parts_lse)
    m = lse.max(axis=0)
    m_safe = np.where(np.isfinite(m), m, 0.0)
    w = np.exp(lse - m_safe[None])
    wsum = w.sum(axis=0)
    with np.errstate(divide="ignore", invalid="ignore"):
        out = np.where(wsum[..., None] > 0,
                       np.einsum("s...,s...d->...d", w, o) / np.where(wsum > 0, wsum, 1.0)[..., None], 0.0)
        out_lse = np.where(wsum > 0, m_safe + np.log(np.where(wsum > 0, wsum, 1.0)), -np.inf)
    return out, out_lse


def rowsum_do_o(do, o) -> np.ndarray:
    """Di = sum_d dO * O per (head, token), the softmax-gradient row term."""
    return np.sum(_as64(do) * _as64(o), axis=-1)


def attention_flops(seqlens: Sequence[int], causal: bool, hq: int, head_dim: int) -> Tuple[float, float]:
    """Forward and backward FLOPs by the convention 4 * Hq * D per unmasked score pair
    (forward) and 2.5x that (backward); pairs counted by their definition."""
    pairs = 0
    for L in seqlens:
        pairs += L * (L + 1) // 2 if causal else L * L
    fwd = 4.0 * hq * head_dim * pairs
    return fwd, 2.5 * fwd
