"""Pins for the oracle's vertical-line token identification (Eq. 4-5, Algorithm 1)."""
import math

import numpy as np
import torch
import pytest

from gen import decode_case
from oracle.select import (check_selection, prefix_len, proxy_sum, score_error_bound,
                           scores, select_vertical, topk_ascending, vl_count)


@pytest.mark.parametrize("P,ppm,k", [
    (896, 50_000, 45),        # L = 1024, W = 128, rho = 5%
    (32640, 50_000, 1632),    # L = 32768, W = 128
    (0, 50_000, 0),           # empty prefix selects nothing
    (1, 50_000, 1),           # max(1, .) keeps at least one key
    (20, 50_000, 1),
    (21, 50_000, 2),          # ceil(1.05)
    (10, 1_000_000, 10),      # rho = 100% takes the whole prefix
    (10, 0, 0),               # rho = 0: the pure low-bit special case
    (32640, 20_000, 653),     # ceil(652.8)
    (32640, 100_000, 3264),
])
def test_vl_count_rule(P, ppm, k):
    assert vl_count(P, ppm) == k


def test_prefix_len():
    assert prefix_len(1024, 128) == 896
    assert prefix_len(100, 128) == 0
    assert prefix_len(128, 128) == 0


def _rank_by_counting(S, k):
    """Independent top-k: j is selected iff fewer than k keys beat it, where i
    beats j when S_i > S_j, or S_i == S_j and i < j."""
    P = len(S)
    sel = []
    for j in range(P):
        beaten = sum(1 for i in range(P) if S[i] > S[j] or (S[i] == S[j] and i < j))
        if beaten < k:
            sel.append(j)
    return np.array(sel, dtype=np.int64)


@pytest.mark.parametrize("seed,L,HQ,HKV", [(0, 200, 4, 4), (1, 300, 8, 2), (2, 150, 4, 1)])
def test_topk_matches_brute_force(seed, L, HQ, HKV):
    c = decode_case(seed, 1, HQ, HKV, L, d=32, window=16, n_proxy=8, n_sinks=5)
    q = c.q_proxy.double().numpy()
    k = c.k.double().numpy()
    idx, S = select_vertical(q, k, L, 16, 50_000)
    P = L - 16
    g = HQ // HKV
    for h in range(HKV):
        # scores as a sum of per-query dot products (linearity of Algorithm 1's mean proxy)
        S_ref = np.zeros(P)
        for hq in range(h * g, (h + 1) * g):
            for t in range(q.shape[2]):
                S_ref += k[0, h, :P] @ q[0, hq, t]
        np.testing.assert_allclose(S[0, h], S_ref, rtol=1e-12, atol=1e-9)
        assert np.array_equal(idx[0, h], _rank_by_counting(S_ref, vl_count(P, 50_000)))


def test_full_ratio_selects_whole_prefix_and_zero_selects_none():
    c = decode_case(3, 1, 4, 4, 300, d=32, window=64, n_proxy=4)
    q, k = c.q_proxy.double().numpy(), c.k.double().numpy()
    idx, _ = select_vertical(q, k, 300, 64, 1_000_000)
    assert idx.shape == (1, 4, 236) and np.array_equal(idx[0, 0], np.arange(236))
    idx0, _ = select_vertical(q, k, 300, 64, 0)
    assert idx0.shape == (1, 4, 0)
    idx1, _ = select_vertical(q, k, 60, 64, 50_000)
    assert idx1.shape == (1, 4, 0)


def test_positive_scaling_of_proxies_keeps_the_set():
    c = decode_case(4, 1, 8, 2, 400, d=64, window=32, n_proxy=16, n_sinks=6)
    q, k = c.q_proxy.double().numpy(), c.k.double().numpy()
    a, _ = select_vertical(q, k, 400, 32, 50_000)
    b, _ = select_vertical(q * 8.0, k, 400, 32, 50_000)
    assert np.array_equal(a, b)


def test_ties_go_to_the_lower_position():
    S = np.array([1.0, 5.0, 3.0, 5.0, 5.0, 0.0])
    assert topk_ascending(S, 2).tolist() == [1, 3]
    assert topk_ascending(S, 3).tolist() == [1, 3, 4]
    # duplicated key rows produce equal scores: the earlier copy wins
    rng = np.random.default_rng(5)
    k = rng.standard_normal((1, 1, 50, 16))
    q = rng.standard_normal((1, 1, 4, 16))
    u = proxy_sum(q, 1)
    S0 = scores(u, k, 50)[0, 0]
    top = int(np.argmax(S0))
    k[0, 0, 49] = k[0, 0, top]          # duplicate the best key at a later position
    idx, _ = select_vertical(q, k, 50, 0, 20_000)      # k = 1
    assert idx[0, 0].tolist() == [min(top, 49)]


def test_planted_sinks_are_all_selected():
    c = decode_case(6, 1, 32, 8, 2048, window=128, n_proxy=64, sink_frac=0.02, sink_gain=8.0)
    idx, _ = select_vertical(c.q_proxy.double().numpy(), c.k.double().numpy(), 2048, 128, 50_000)
    for h in range(8):
        assert set(c.sinks[0, h].tolist()) <= set(idx[0, h].tolist())


def test_gqa_sum_equals_per_query_head_sum():
    c = decode_case(7, 2, 8, 2, 200, d=32, window=16, n_proxy=8)
    q = c.q_proxy.double().numpy()
    u = proxy_sum(q, 2)
    np.testing.assert_allclose(u[1, 1], q[1, 4:8].sum(axis=(0, 1)), rtol=1e-13)


def test_check_selection_accepts_truth_and_rejects_wrong_sets():
    c = decode_case(8, 1, 4, 4, 600, d=64, window=64, n_proxy=16, n_sinks=10)
    q, k = c.q_proxy.double().numpy(), c.k.double().numpy()
    idx, S = select_vertical(q, k, 600, 64, 50_000)
    bnd = score_error_bound(q, k, 536)
    kk = vl_count(536, 50_000)
    assert check_selection(S[0, 0], bnd[0, 0], kk, idx[0, 0])["ok"]
    worst = np.argsort(S[0, 0])[:kk]
    assert not check_selection(S[0, 0], bnd[0, 0], kk, np.sort(worst))["ok"]
    assert not check_selection(S[0, 0], bnd[0, 0], kk, idx[0, 0][:-1])["ok"]


def test_error_bound_covers_float32_evaluation():
    c = decode_case(9, 1, 32, 8, 4096, window=128, n_proxy=64, sink_frac=0.02)
    q32 = c.q_proxy.float().numpy()
    k32 = c.k.float().numpy()
    P = 4096 - 128
    u32 = q32.reshape(1, 8, 4, 64, 128).sum(axis=(2, 3), dtype=np.float32)
    S32 = np.einsum("bhd,bhpd->bhp", u32, k32[:, :, :P]).astype(np.float64)
    S = scores(proxy_sum(c.q_proxy.double().numpy(), 8), c.k.double().numpy(), P)
    bnd = score_error_bound(c.q_proxy.double().numpy(), c.k.double().numpy(), P)
    assert np.all(np.abs(S32 - S) <= bnd)


# --- Eq. 4: the softmax-mass score ------------------------------------------

def _mass_brute(q, k, L, W):
    """Pure-Python Eq. 4 on a tiny case: per (b, kvh), per proxy row of every
    query head of the group, a softmax over the L keys, summed per key."""
    B, HQ, T, d = q.shape
    HKV = k.shape[1]
    g = HQ // HKV
    P = max(0, L - W)
    out = np.zeros((B, HKV, P))
    for b in range(B):
        for kh in range(HKV):
            for h in range(kh * g, (kh + 1) * g):
                for t in range(T):
                    z = [sum(q[b, h, t, i] * k[b, kh, j, i] for i in range(d)) / math.sqrt(d) for j in range(L)]
                    m = max(z)
                    e = [math.exp(x - m) for x in z]
                    tot = sum(e)
                    for j in range(P):
                        out[b, kh, j] += e[j] / tot
    return out


def test_mass_scores_brute_force_gqa():
    from oracle.select import mass_scores
    rng = np.random.default_rng(41)
    q = rng.standard_normal((2, 4, 3, 8))
    k = rng.standard_normal((2, 2, 11, 8)) * 2
    np.testing.assert_allclose(mass_scores(q, k, 11, 4), _mass_brute(q, k, 11, 4), rtol=1e-12, atol=1e-14)


def test_mass_scores_sum_to_rows_without_window():
    """Each row's probabilities sum to one, so with W = 0 the column masses
    of a KV head sum to the number of (proxy, query head) rows."""
    from oracle.select import mass_scores
    rng = np.random.default_rng(42)
    q = rng.standard_normal((1, 6, 5, 16)) * 3
    k = rng.standard_normal((1, 2, 40, 16))
    S = mass_scores(q, k, 40, 0)
    np.testing.assert_allclose(S.sum(axis=-1), 3 * 5, rtol=1e-12)
    assert np.all(S > 0)


def test_mass_scores_shift_invariant():
    """Adding one vector to every key shifts each row's logits by a constant:
    the softmax, hence the score, is unchanged."""
    from oracle.select import mass_scores
    rng = np.random.default_rng(43)
    q = rng.standard_normal((1, 2, 4, 16))
    k = rng.standard_normal((1, 1, 30, 16))
    shifted = k + rng.standard_normal(16)[None, None, None, :] * 5
    np.testing.assert_allclose(mass_scores(q, shifted, 30, 6), mass_scores(q, k, 30, 6), rtol=1e-10)


def test_mass_planted_key_takes_the_mass():
    from oracle.select import mass_scores, select_vertical_mass
    rng = np.random.default_rng(44)
    u = rng.standard_normal(32)
    u /= np.linalg.norm(u)
    q = 0.3 * rng.standard_normal((1, 2, 8, 32)) + 3 * u     # every proxy row leans along u
    k = rng.standard_normal((1, 1, 50, 32)) * 0.1
    k[0, 0, 17] = 40 * u
    S = mass_scores(q, k, 50, 10)
    assert S[0, 0, 17] > 0.99 * 16
    idx, _ = select_vertical_mass(q, k, 50, 10, 50_000)
    assert 17 in idx[0, 0]


def test_mass_error_bound_covers_a_float32_evaluation():
    """A float32 evaluation in the bound's own recipe (float32 dot products
    of BF16-valued inputs, a scaled logit, row maximum and sum of exp2, the
    quotient and a float32 column sum) stays inside the bound."""
    from oracle.select import mass_error_bound, mass_scores
    rng = np.random.default_rng(45)
    to_bf16 = lambda x: torch.from_numpy(x).to(torch.bfloat16).double().numpy()
    q = to_bf16(rng.standard_normal((1, 4, 16, 128)))
    k = to_bf16(rng.standard_normal((1, 2, 700, 128)))
    L, W = 700, 128
    S = mass_scores(q, k, L, W)
    bnd = mass_error_bound(q, k, L, W)
    c = np.float32(1.0 / np.sqrt(128) / np.log(2.0))
    P = L - W
    for kh in range(2):
        Q = q[0, 2 * kh:2 * kh + 2].reshape(32, 128).astype(np.float32)
        K = k[0, kh, :L].astype(np.float32)
        t = (Q @ K.T).astype(np.float32) * c
        m = t.max(axis=1, keepdims=True)
        p = np.exp2(t - m).astype(np.float32)
        a = (p / p.sum(axis=1, keepdims=True, dtype=np.float32)).astype(np.float32)
        S32 = a[:, :P].sum(axis=0, dtype=np.float32)
        err = np.abs(S32.astype(np.float64) - S[0, kh])
        assert np.all(err <= bnd[0, kh]), float((err - bnd[0, kh]).max())
        assert bnd[0, kh].max() < 1e-3 * S[0, kh].max()   # tight enough to decide most keys
