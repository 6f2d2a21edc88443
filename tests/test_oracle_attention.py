"""Pins of the float64 attention oracle against facts the definition and the mathematics fix.

None of these re-types the oracle's formulas: each compares it with an independent
construction (a packed-layout brute force with an explicit sequence mask, a
library routine in a special case, closed forms, finite differences, the
associativity of softmax over a split key range).
"""
import math

import numpy as np
import pytest
import torch

from oracle import attention as A


def _rand(shape, seed, scale=1.0):
    return np.random.default_rng(seed).standard_normal(shape) * scale


def _brute_force(q, k, v, seqlens, causal):
    """Attention over the whole packed token axis with an explicit visibility matrix:
    token j is visible to token i iff both lie in the same sequence and (not causal or j <= i).
    Plain loops over rows, math.exp per element."""
    hq, T, D = q.shape
    G = hq // k.shape[0]
    seq_id = np.repeat(np.arange(len(seqlens)), seqlens)
    pos = np.concatenate([np.arange(L) for L in seqlens]) if T else np.zeros(0, int)
    o = np.zeros((hq, T, D))
    lse = np.zeros((hq, T))
    for h in range(hq):
        g = h // G
        for i in range(T):
            vis = [j for j in range(T) if seq_id[j] == seq_id[i] and (not causal or pos[j] <= pos[i])]
            s = [float(np.dot(q[h, i], k[g, j])) / math.sqrt(D) for j in vis]
            mx = max(s)
            e = [math.exp(x - mx) for x in s]
            tot = sum(e)
            for w, j in zip(e, vis):
                o[h, i] += (w / tot) * v[g, j]
            lse[h, i] = mx + math.log(tot)
    return o, lse


@pytest.mark.parametrize("causal", [True, False])
@pytest.mark.parametrize("hq,hkv", [(2, 1), (4, 2), (3, 3)])
def test_forward_matches_brute_force(causal, hq, hkv):
    seqlens = [5, 1, 9, 3]
    T, D = sum(seqlens), 8
    q, k, v = _rand((hq, T, D), 1), _rand((hkv, T, D), 2), _rand((hkv, T, D), 3)
    o, lse = A.attention_forward(q, k, v, seqlens, causal)
    ob, lb = _brute_force(q, k, v, seqlens, causal)
    assert np.abs(o - ob).max() < 1e-12
    assert np.abs(lse - lb).max() < 1e-12


def test_uniform_scores_give_mean_of_v():
    """Q = 0 makes every visible score equal: full mask gives the sequence mean of V,
    causal row i the mean of V[0..i], and LSE = log(number of visible keys)."""
    seqlens = [7, 12]
    T, D = sum(seqlens), 16
    q = np.zeros((4, T, D))
    k, v = _rand((2, T, D), 4), _rand((2, T, D), 5)
    o, lse = A.attention_forward(q, k, v, seqlens, causal=False)
    a = 0
    for L in seqlens:
        for h in range(4):
            assert np.allclose(o[h, a:a + L], v[h // 2, a:a + L].mean(0)[None], atol=1e-13)
            assert np.allclose(lse[h, a:a + L], math.log(L), atol=1e-13)
        a += L
    o, lse = A.attention_forward(q, k, v, seqlens, causal=True)
    a = 0
    for L in seqlens:
        cm = np.cumsum(v[:, a:a + L], axis=1) / np.arange(1, L + 1)[None, :, None]
        for h in range(4):
            assert np.allclose(o[h, a:a + L], cm[h // 2], atol=1e-13)
            assert np.allclose(lse[h, a:a + L], np.log(np.arange(1, L + 1)), atol=1e-13)
        a += L


def test_causal_row_zero_is_v0():
    seqlens = [3, 10, 1]
    T, D = sum(seqlens), 8
    q, k, v = _rand((2, T, D), 6), _rand((1, T, D), 7), _rand((1, T, D), 8)
    o, lse = A.attention_forward(q, k, v, seqlens, causal=True)
    a = 0
    for L in seqlens:
        for h in range(2):
            assert np.allclose(o[h, a], v[0, a], atol=1e-14)
            assert abs(lse[h, a] - float(q[h, a] @ k[0, a]) / math.sqrt(D)) < 1e-13
        a += L


@pytest.mark.parametrize("causal", [False, True])
def test_single_sequence_matches_torch_sdpa(causal):
    """One sequence equals torch's scaled_dot_product_attention in float64 on the CPU (a library
    routine), with the KV heads repeated for the query heads of their group."""
    hq, hkv, L, D = 8, 2, 37, 32
    q, k, v = _rand((hq, L, D), 9), _rand((hkv, L, D), 10), _rand((hkv, L, D), 11)
    o, _ = A.attention_forward(q, k, v, [L], causal)
    tq = torch.from_numpy(q)[None]
    tk = torch.from_numpy(k).repeat_interleave(hq // hkv, dim=0)[None]
    tv = torch.from_numpy(v).repeat_interleave(hq // hkv, dim=0)[None]
    ref = torch.nn.functional.scaled_dot_product_attention(tq, tk, tv, is_causal=causal)[0].numpy()
    assert np.abs(o - ref).max() < 1e-12


def _partial(qrow, k_sub, v_sub, scale):
    """Attention of one query row over a key subset, by plain loops."""
    s = [float(np.dot(qrow, kk)) * scale for kk in k_sub]
    mx = max(s)
    e = [math.exp(x - mx) for x in s]
    tot = sum(e)
    return sum((w / tot) * vv for w, vv in zip(e, v_sub)), mx + math.log(tot)


@pytest.mark.parametrize("seed", [0, 1, 2])
def test_merge_of_any_split_equals_unsplit(seed):
    """Associativity (Section 2.3): attention over a key range, split at arbitrary points into
    parts computed separately, merged by log-sum-exp, equals the unsplit result."""
    rng = np.random.default_rng(seed)
    L, D = 40, 16
    q, k, v = rng.standard_normal((1, L, D)) * 2, rng.standard_normal((1, L, D)), rng.standard_normal((1, L, D))
    o_full, lse_full = A.attention_forward(q, k, v, [L], causal=False)
    cuts = sorted(rng.choice(np.arange(1, L), size=4, replace=False).tolist())
    bounds = [0] + cuts + [L]
    scale = 1 / math.sqrt(D)
    for i in range(L):
        po, pl = [], []
        for a, b in zip(bounds[:-1], bounds[1:]):
            oo, ll = _partial(q[0, i], k[0, a:b], v[0, a:b], scale)
            po.append(oo)
            pl.append(ll)
        om, lm = A.lse_merge(np.array(po), np.array(pl))
        assert np.abs(om - o_full[0, i]).max() < 1e-12
        assert abs(lm - lse_full[0, i]) < 1e-12


def test_merge_special_cases():
    rng = np.random.default_rng(3)
    o = rng.standard_normal((3, 5, 8))
    lse = rng.standard_normal((3, 5))
    # order of the parts does not matter
    om, lm = A.lse_merge(o, lse)
    om2, lm2 = A.lse_merge(o[::-1], lse[::-1])
    assert np.abs(om - om2).max() < 1e-13 and np.abs(lm - lm2).max() < 1e-13
    # a part with lse = -inf carries no weight
    lse_inf = lse.copy()
    lse_inf[1] = -np.inf
    om3, lm3 = A.lse_merge(o, lse_inf)
    om4, lm4 = A.lse_merge(o[[0, 2]], lse[[0, 2]])
    assert np.abs(om3 - om4).max() < 1e-13 and np.abs(lm3 - lm4).max() < 1e-13
    # equal weights average, and lse grows by log(S)
    om5, lm5 = A.lse_merge(o, np.zeros((3, 5)))
    assert np.abs(om5 - o.mean(0)).max() < 1e-13 and np.abs(lm5 - math.log(3)).max() < 1e-13
    # all parts empty
    om6, lm6 = A.lse_merge(o, np.full((3, 5), -np.inf))
    assert np.all(om6 == 0) and np.all(np.isneginf(lm6))


@pytest.mark.parametrize("causal", [True, False])
def test_backward_matches_finite_differences(causal):
    """Central differences of sum(O * dO) in float64 pin every gradient term."""
    seqlens = [4, 6]
    T, D, hq, hkv = sum(seqlens), 4, 4, 2
    q, k, v, do = _rand((hq, T, D), 12), _rand((hkv, T, D), 13), _rand((hkv, T, D), 14), _rand((hq, T, D), 15)
    dq, dk, dv = A.attention_backward(q, k, v, do, seqlens, causal)

    def loss(q_, k_, v_):
        return float(np.sum(A.attention_forward(q_, k_, v_, seqlens, causal)[0] * do))

    eps = 1e-6
    for name, x, g in (("q", q, dq), ("k", k, dk), ("v", v, dv)):
        num = np.zeros_like(x)
        it = np.nditer(x, flags=["multi_index"])
        for _ in it:
            idx = it.multi_index
            xp, xm = x.copy(), x.copy()
            xp[idx] += eps
            xm[idx] -= eps
            args_p = {"q": (xp, k, v), "k": (q, xp, v), "v": (q, k, xp)}[name]
            args_m = {"q": (xm, k, v), "k": (q, xm, v), "v": (q, k, xm)}[name]
            num[idx] = (loss(*args_p) - loss(*args_m)) / (2 * eps)
        err = np.abs(num - g).max() / max(1.0, np.abs(num).max())
        assert err < 1e-6, (name, err)


def test_row_helpers_agree_with_whole_sequence():
    """The per-row helpers used for sampled checks at full size agree with the whole-sequence oracle."""
    seqlens = [33, 70]
    T, D, hq, hkv = sum(seqlens), 16, 4, 2
    q, k, v, do = _rand((hq, T, D), 16), _rand((hkv, T, D), 17), _rand((hkv, T, D), 18), _rand((hq, T, D), 19)
    for causal in (True, False):
        o, lse = A.attention_forward(q, k, v, seqlens, causal)
        dq, dk, dv = A.attention_backward(q, k, v, do, seqlens, causal)
        a, L = 33, 70
        rows = [0, 5, 69, 40]
        for g in range(hkv):
            hs = slice(2 * g, 2 * g + 2)
            ro, rl = A.attention_rows(q[hs, a + np.array(rows)], k[g, a:a + L], v[g, a:a + L], rows, causal)
            assert np.abs(ro - o[hs][:, a + np.array(rows)]).max() < 1e-12
            assert np.abs(rl - lse[hs][:, a + np.array(rows)]).max() < 1e-12
            rdq = A.attention_dq_rows(q[hs, a + np.array(rows)], do[hs, a + np.array(rows)],
                                      k[g, a:a + L], v[g, a:a + L], rows, causal)
            assert np.abs(rdq - dq[hs][:, a + np.array(rows)]).max() < 1e-12
            kv_rows = [69, 60, 3]
            rdk, rdv = A.attention_dkv_rows(q[hs, a:a + L], do[hs, a:a + L], k[g, a:a + L], v[g, a:a + L],
                                            kv_rows, causal)
            assert np.abs(rdk - dk[g, a + np.array(kv_rows)]).max() < 1e-12
            assert np.abs(rdv - dv[g, a + np.array(kv_rows)]).max() < 1e-12
            if causal:  # only the query tail from the first selected key is needed
                tail = [69, 60, 55]
                rdk, rdv = A.attention_dkv_rows(q[hs, a + 55:a + L], do[hs, a + 55:a + L], k[g, a:a + L],
                                                v[g, a:a + L], tail, causal, q_offset=55)
                assert np.abs(rdk - dk[g, a + np.array(tail)]).max() < 1e-12
                assert np.abs(rdv - dv[g, a + np.array(tail)]).max() < 1e-12


def test_di_identity():
    """rowsum(dO * O) equals sum_j P_ij dP_ij, the identity the gradient's row term rests on."""
    L, D = 9, 8
    q, k, v, do = _rand((1, L, D), 20), _rand((1, L, D), 21), _rand((1, L, D), 22), _rand((1, L, D), 23)
    o, lse = A.attention_forward(q, k, v, [L], causal=True)
    di = A.rowsum_do_o(do, o)
    for i in range(L):
        p = [math.exp(float(q[0, i] @ k[0, j]) / math.sqrt(D) - lse[0, i]) for j in range(i + 1)]
        dp = [float(do[0, i] @ v[0, j]) for j in range(i + 1)]
        assert abs(sum(a * b for a, b in zip(p, dp)) - di[0, i]) < 1e-12


def test_flop_convention_counts_unmasked_pairs():
    for seqlens, causal in (([5, 3], True), ([5, 3], False), ([1], True)):
        pairs = 0
        for L in seqlens:
            pairs += sum(1 for i in range(L) for j in range(L) if (not causal or j <= i))
        f, b = A.attention_flops(seqlens, causal, 2, 8)
        assert f == 4 * 2 * 8 * pairs and b == 2.5 * f
