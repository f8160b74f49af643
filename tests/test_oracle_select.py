"""Pins for the oracle's vertical-line token identification (Eq. 4-5, Algorithm 1)."""
import numpy as np
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
