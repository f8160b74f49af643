"""Pins for the oracle's per-query-head vertical-line sets (Algorithm 1's
B x H_Q x k output) and the per-KV-head list built from them: the union of
the group's sets, filled up to min(P, g k) by the group score."""
import numpy as np
import pytest

from gen import decode_case
from oracle.select import (head_scores, prefix_len, select_vertical, select_vertical_heads, topk_ascending,
                           union_fill, vl_count, vl_count_heads)


@pytest.mark.parametrize("seed,L,W,ppm", [(0, 300, 64, 50_000), (1, 1024, 128, 20_000), (2, 129, 128, 50_000)])
def test_mha_reduces_to_the_kv_head_reading(seed, L, W, ppm):
    # g = 1: a query head is its KV head, so both readings select the same set
    c = decode_case(seed, 2, 4, 4, L, window=W, n_proxy=16, n_sinks=4)
    q, k = c.q_proxy.double().numpy(), c.k.double().numpy()
    want, _ = select_vertical(q, k, L, W, ppm)
    ih, ik, us, _, _ = select_vertical_heads(q, k, L, W, ppm)
    assert np.array_equal(ih, want) and np.array_equal(ik, want)
    assert vl_count_heads(prefix_len(L, W), ppm, 1) == vl_count(prefix_len(L, W), ppm)


def test_head_scores_by_explicit_loops():
    c = decode_case(3, 1, 6, 2, 90, d=16, window=10, n_proxy=3, n_sinks=0)
    q, k = c.q_proxy.double().numpy(), c.k.double().numpy()
    S = head_scores(q, k, 80)
    for h in range(6):
        for j in (0, 7, 79):
            ref = sum(float(np.dot(q[0, h, t], k[0, h // 3, j])) for t in range(3))
            assert abs(S[0, h, j] - ref) <= 1e-12 * (1 + abs(ref))


def _planted(g=4, HKV=2, P=400, kk=8, s=2, T=3, d=128):
    """Query head i of KV head kh has its own proxy direction e_(kh, i).  Its
    kk planted keys (10 e_(kh, i) each) are kk - 2s of its own and the s
    positions of each of its two cyclic neighbour pairs (i - 1, i) and
    (i, i + 1), which carry both heads' directions; g s further positions
    carry 5 times the sum of the group's directions (head score 5 T, below
    every planted key of the head; group score 5 g T, above every position
    outside the union).  Returns q, keys, the head sets, and per KV head the
    union and the fill."""
    rng = np.random.default_rng(7)
    HQ, W = g * HKV, 32
    q = np.zeros((1, HQ, T, d))
    keys = 1e-3 * rng.standard_normal((1, HKV, P + W, d))
    perm = iter(rng.permutation(P).tolist())
    heads, lists = {}, {}
    for kh in range(HKV):
        e = [2 * (kh * g + i) for i in range(g)]
        for i in range(g):
            q[0, kh * g + i, :, e[i]] = 1.0
        sets = [[] for _ in range(g)]
        for i in range(g):
            for _ in range(kk - 2 * s):
                j = next(perm)
                keys[0, kh, j, e[i]] += 10.0
                sets[i].append(j)
            for _ in range(s):                     # the pair (i, i + 1)
                j = next(perm)
                keys[0, kh, j, e[i]] += 10.0
                keys[0, kh, j, e[(i + 1) % g]] += 10.0
                sets[i].append(j)
                sets[(i + 1) % g].append(j)
        fill = []
        for _ in range(g * s):
            j = next(perm)
            for i in range(g):
                keys[0, kh, j, e[i]] += 5.0
            fill.append(j)
        heads[kh] = [sorted(x) for x in sets]
        lists[kh] = (sorted(set(sum(sets, []))), sorted(fill))
    return q, keys, heads, lists, P + W, W


def test_planted_head_sets_union_and_fill():
    g, HKV, kk, s = 4, 2, 8, 2
    q, keys, heads, lists, L, W = _planted(g, HKV, 400, kk, s)
    P = L - W
    ppm = 20_000                           # k = ceil(400 * 0.02) = 8 per head
    assert vl_count(P, ppm) == kk
    ku = vl_count_heads(P, ppm, g)
    assert ku == g * kk
    ih, ik, us, _, _ = select_vertical_heads(q, keys, L, W, ppm)
    for kh in range(HKV):
        for i in range(g):
            assert ih[0, kh * g + i].tolist() == heads[kh][i]
        union, fill = lists[kh]
        assert us[0, kh] == len(union) == g * (kk - s)
        assert ik[0, kh].tolist() == sorted(union + fill)


@pytest.mark.parametrize("seed,B,HQ,HKV,L,W,ppm", [(11, 1, 8, 2, 500, 64, 20_000), (12, 2, 4, 1, 300, 32, 50_000),
                                                   (13, 1, 8, 8, 200, 16, 100_000)])
def test_definition_by_pairwise_comparison(seed, B, HQ, HKV, L, W, ppm):
    """Each head's set: no unselected position beats a selected one (score,
    then lower position); the list: contains the union, has min(P, g k)
    entries, and no position outside it beats a filled-in one by the group
    score."""
    c = decode_case(seed, B, HQ, HKV, L, window=W, n_proxy=8, n_sinks=6)
    q, k = c.q_proxy.double().numpy(), c.k.double().numpy()
    g = HQ // HKV
    P = prefix_len(L, W)
    ih, ik, us, S_heads, S_group = select_vertical_heads(q, k, L, W, ppm)
    beats = lambda S, i, j: S[i] > S[j] or (S[i] == S[j] and i < j)
    for b in range(B):
        for h in range(HQ):
            sel = set(ih[b, h].tolist())
            assert len(sel) == vl_count(P, ppm) and list(ih[b, h]) == sorted(sel)
            out = [j for j in range(P) if j not in sel]
            worst = min(sel, key=lambda j: (S_heads[b, h, j], -j))
            assert not any(beats(S_heads[b, h], j, worst) for j in out)
        for kh in range(HKV):
            union = set(ih[b, kh * g:(kh + 1) * g].ravel().tolist())
            lst = ik[b, kh].tolist()
            assert lst == sorted(set(lst)) and len(lst) == min(P, g * vl_count(P, ppm))
            assert union <= set(lst) and us[b, kh] == len(union)
            filled = set(lst) - union
            out = [j for j in range(P) if j not in set(lst)]
            if filled and out:
                worst = min(filled, key=lambda j: (S_group[b, kh, j], -j))
                assert not any(beats(S_group[b, kh], j, worst) for j in out)


def test_union_fill_small_cases():
    S = np.array([0.0, 5.0, 1.0, 5.0, 3.0, 2.0])
    assert union_fill([[2], [2]], S, 3).tolist() == [1, 2, 3]       # ties to the lower position
    assert union_fill([[0, 5], [4]], S, 3).tolist() == [0, 4, 5]     # a full union needs no fill
    assert union_fill(np.zeros((2, 0), np.int64), S, 2).tolist() == [1, 3]


def test_mse_cost_against_the_kv_head_reading(capsys):
    """Attention-output MSE (against full-precision attention) of the two
    readings on inputs whose query heads attend to different keys: each query
    head h has its own direction w_h and its own planted keys (k += 4 w_h),
    its queries q += 2 w_h.  Per query head (union filled to g k) keeps every
    head's keys in BF16; per KV head with k positions keeps a quarter of them
    (g = 4); per KV head with g k positions spends the same bytes."""
    from oracle.attention import hybrid_decode
    from oracle.metrics import exact_decode, mse
    rng = np.random.default_rng(2024)
    B, HQ, HKV, d, L, W, ppm, T = 1, 8, 2, 128, 2048, 128, 20_000, 64
    g, P = HQ // HKV, L - W
    k1 = vl_count(P, ppm)
    k = rng.standard_normal((B, HKV, L, d))
    v = rng.standard_normal((B, HKV, L, d))
    q = rng.standard_normal((B, HQ, d))
    qp = rng.standard_normal((B, HQ, T, d))
    perm = rng.permutation(P)
    for h in range(HQ):
        w = rng.standard_normal(d)
        w /= np.linalg.norm(w)
        pos = perm[h * k1:(h + 1) * k1]
        k[0, h // g, pos] += 4.0 * w
        q[0, h] += 2.0 * w
        qp[0, h] += 2.0 * w
    bf = lambda x: x.astype(np.float32).view(np.uint32).__and__(0xFFFF0000).view(np.float32).astype(np.float64)
    k, v, q, qp = bf(k), bf(v), bf(q), bf(qp)
    exact = exact_decode(q, k, v, L)
    _, idx_heads_list, us, _, _ = select_vertical_heads(qp, k, L, W, ppm)
    idx_kv, S_kv = select_vertical(qp, k, L, W, ppm)
    idx_kv_g = topk_ascending(S_kv, g * k1)                # per KV head, g k positions (same bytes)
    assert idx_kv_g.shape[-1] == g * k1 == idx_heads_list.shape[-1]
    m_heads = mse(hybrid_decode(q, k, v, L, P, idx_heads_list), exact)
    m_kv = mse(hybrid_decode(q, k, v, L, P, idx_kv), exact)
    m_kv_g = mse(hybrid_decode(q, k, v, L, P, idx_kv_g), exact)
    with capsys.disabled():
        print(f"\nMSE vs full precision: per query head (union {us.tolist()} of {g * k1}) {m_heads:.3e}, "
              f"per KV head k={k1} {m_kv:.3e}, per KV head k={g * k1} {m_kv_g:.3e}")
    assert m_heads < m_kv
