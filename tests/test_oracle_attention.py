"""Pins for the oracle's hybrid decode attention (Eq. 1-3, 8-9, Algorithm 3).

The special cases reduce to a library routine: with every position kept in
BF16 (rho = 100% or W >= L) the result is plain softmax attention, checked
against torch's float64 scaled_dot_product_attention; with rho = 0 and W = 0
it is softmax attention over the dequantised cache.
"""
import math

import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gen import decode_case
from oracle.attention import decode_alg3, effective_cache, hybrid_decode, textbook_attention
from oracle.quant import fake_quant
from oracle.select import prefix_len, select_vertical


def sdpa(q, K, V):
    """torch float64 attention for one decode query per head; GQA by repeating heads."""
    q = torch.from_numpy(np.asarray(q, np.float64))           # [B, HQ, d]
    K = torch.from_numpy(np.asarray(K, np.float64))           # [B, HKV, L, d]
    V = torch.from_numpy(np.asarray(V, np.float64))
    g = q.shape[1] // K.shape[1]
    K = K.repeat_interleave(g, dim=1)
    V = V.repeat_interleave(g, dim=1)
    return F.scaled_dot_product_attention(q[:, :, None], K, V)[:, :, 0].numpy()


def case(seed=0, B=1, HQ=8, HKV=2, L=700, W=128, **kw):
    c = decode_case(seed, B, HQ, HKV, L, window=W, n_proxy=16, sink_frac=0.03, **kw)
    return (c.q.double().numpy(), c.q_proxy.double().numpy(),
            c.k.double().numpy(), c.v.double().numpy())


def test_window_covering_context_is_exact_attention():
    q, qp, k, v = case(L=100, W=128)
    o = hybrid_decode(q, k, v, 100, prefix_len(100, 128), None)
    np.testing.assert_allclose(o, sdpa(q, k, v), rtol=1e-12, atol=1e-13)


def test_full_ratio_is_exact_attention():
    q, qp, k, v = case(L=500, W=64, B=2)
    idx, _ = select_vertical(qp, k, 500, 64, 1_000_000)
    o = hybrid_decode(q, k, v, 500, 436, idx)
    np.testing.assert_allclose(o, sdpa(q, k, v), rtol=1e-12, atol=1e-13)


def test_zero_ratio_zero_window_is_attention_on_dequantised_cache():
    q, qp, k, v = case(L=400, W=0, HQ=4, HKV=4)
    idx, _ = select_vertical(qp, k, 400, 0, 0)
    o = hybrid_decode(q, k, v, 400, 400, idx)
    np.testing.assert_allclose(o, sdpa(q, fake_quant(k), fake_quant(v)), rtol=1e-12, atol=1e-13)
    # and it really differs from the BF16 result
    assert np.abs(o - sdpa(q, k, v)).max() > 1e-3


def test_partition_roles():
    """Positions in the VL set and in [P, L) keep their BF16 rows; the rest are
    dequantised."""
    q, qp, k, v = case(L=300, W=50, HQ=2, HKV=2)
    P = 250
    idx, _ = select_vertical(qp, k, 300, 50, 100_000)
    K, V = effective_cache(k, v, 300, P, idx)
    for h in range(2):
        vl = set(idx[0, h].tolist())
        for j in range(300):
            if j >= P or j in vl:
                assert np.array_equal(K[0, h, j], k[0, h, j])
                assert np.array_equal(V[0, h, j], v[0, h, j])
            else:
                assert np.array_equal(K[0, h, j], fake_quant(k[0, h, j][None])[0])
                assert not np.array_equal(K[0, h, j], k[0, h, j])


@pytest.mark.parametrize("splits,tile", [(1, 64), (4, 64), (7, 16), (64, 3), (2000, 64)])
def test_alg3_split_merge_equals_single_pass(splits, tile):
    q, qp, k, v = case(seed=3, L=900, W=128, B=1, HQ=8, HKV=2)
    P = 772
    idx, _ = select_vertical(qp, k, 900, 128, 50_000)
    a = hybrid_decode(q, k, v, 900, P, idx)
    b = decode_alg3(q, k, v, 900, P, idx, splits=splits, tile=tile)
    np.testing.assert_allclose(b, a, rtol=1e-12, atol=1e-14)


def test_single_position_returns_its_value():
    q, qp, k, v = case(L=1, W=0, HQ=4, HKV=2)
    o = hybrid_decode(q, k, v, 1, 0, None)
    assert np.allclose(o[0, 0], v[0, 0, 0]) and np.allclose(o[0, 3], v[0, 1, 0])


def test_identical_keys_average_the_values():
    rng = np.random.default_rng(1)
    K = np.repeat(rng.standard_normal((1, 32)), 9, axis=0)
    V = rng.standard_normal((9, 32))
    o = textbook_attention(rng.standard_normal((3, 32)), K, V, 0.3)
    np.testing.assert_allclose(o, np.repeat(V.mean(0, keepdims=True), 3, 0), rtol=1e-13)


def test_position_permutation_invariance():
    rng = np.random.default_rng(2)
    K, V, q = rng.standard_normal((50, 16)), rng.standard_normal((50, 16)), rng.standard_normal((2, 16))
    perm = rng.permutation(50)
    np.testing.assert_allclose(textbook_attention(q, K, V, 0.25),
                               textbook_attention(q, K[perm], V[perm], 0.25), rtol=1e-12)


def test_scale_is_inverse_sqrt_head_dim():
    q, qp, k, v = case(L=64, W=128, HQ=2, HKV=2)
    o = hybrid_decode(q, k, v, 64, 0, None)
    o2 = hybrid_decode(q, k, v, 64, 0, None, alpha=1.0 / math.sqrt(128))
    assert np.array_equal(o, o2)
    o3 = hybrid_decode(q, k, v, 64, 0, None, alpha=1.0)
    assert np.abs(o3 - o).max() > 1e-2


@pytest.mark.parametrize("bk,bv", [(4, 4), (8, 8), (4, 8), (8, 4)])
def test_bit_widths_are_attention_on_the_dequantised_cache(bk, bv):
    """rho = 0, W = 0 with B_K / B_V bits: softmax attention (torch float64)
    over keys dequantised at B_K bits and values at B_V bits, and the two
    widths act on their own tensor only."""
    q, qp, k, v = case(seed=5, L=300, W=0, HQ=4, HKV=2)
    o = hybrid_decode(q, k, v, 300, 300, None, bits=bk, bits_v=bv)
    np.testing.assert_allclose(o, sdpa(q, fake_quant(k, bk), fake_quant(v, bv)), rtol=1e-12, atol=1e-13)
    if bk != bv:
        assert np.abs(o - hybrid_decode(q, k, v, 300, 300, None, bits=bk)).max() > 1e-6


def test_eight_bit_cache_is_closer_than_four_bit():
    """Over several seeds the 8-bit cache's output error is far below the
    4-bit one's (the grid step shrinks by 17: 255 vs 15 levels)."""
    e4, e8 = [], []
    for seed in range(4):
        q, qp, k, v = case(seed=10 + seed, L=400, W=0, HQ=4, HKV=2)
        ex = sdpa(q, k, v)
        e4.append(np.mean((hybrid_decode(q, k, v, 400, 400, None, bits=4) - ex) ** 2))
        e8.append(np.mean((hybrid_decode(q, k, v, 400, 400, None, bits=8) - ex) ** 2))
    assert np.mean(e8) < np.mean(e4) / 50


def test_alg3_split_merge_with_mixed_widths():
    q, qp, k, v = case(seed=6, L=500, W=64, B=2)
    idx, _ = select_vertical(qp, k, 500, 64, 50_000)
    ref = hybrid_decode(q, k, v, 500, 436, idx, bits=8, bits_v=4)
    np.testing.assert_allclose(decode_alg3(q, k, v, 500, 436, idx, splits=5, tile=32, bits=8, bits_v=4), ref,
                               rtol=1e-12, atol=1e-13)
