"""The C++ float64 oracle against the Python oracle (both pinned to the
paper by the other ``test_oracle_*`` files): quantiser codes, steps and
zeros identical; vertical-line sets identical; decode and prefill outputs
equal to float64 rounding (the two differ only in summation order).  Plus
direct pins of the C++ number formats."""
import numpy as np
import pytest
import torch

from gen import decode_case, prefill_case
from oracle import cpp_oracle as C
from oracle.attention import hybrid_decode
from oracle.prefill import e4m3_values, hybrid_prefill
from oracle.quant import quantize
from oracle.select import select_vertical, select_vertical_mass, vl_count
from tests.gpu_util import mixed_rows, tie_rows


def _np(t):
    return t.double().numpy()


@pytest.mark.parametrize("bits", [4, 8])
@pytest.mark.parametrize("rows", ["mixed", "ties"])
def test_quantiser_identical(bits, rows):
    x = _np(mixed_rows(3, (64, 128)) if rows == "mixed" else tie_rows(4, (64, 128), bits))
    c, s, z = quantize(x, bits)
    c2, s2, z2 = C.quantize(x, bits)
    assert np.array_equal(c, c2)
    assert np.array_equal(s.astype(np.float64), s2) and np.array_equal(z.astype(np.float64), z2)


def test_quantiser_extreme_spans_and_range_error():
    # ranges a hair above 15 * (a binary16 value): the step is the next binary16 up
    rows = np.zeros((3, 128))
    for i, (hi, tiny) in enumerate([(15.0, 2.0 ** -80), (7.5, 2.0 ** -90), (30.0, 2.0 ** -70)]):
        rows[i, 0], rows[i, 1] = -tiny, hi
    c, s, z = quantize(rows)
    c2, s2, z2 = C.quantize(rows)
    assert np.array_equal(c, c2) and np.array_equal(s.astype(np.float64), s2)
    bad = np.zeros((1, 128))
    bad[0, 5] = -70000.0
    with pytest.raises(ValueError):
        C.quantize(bad)


def test_e4m3_table_identical():
    assert [C.e4m3_value(i) for i in range(127)] == list(e4m3_values())
    assert C.e4m3_value(126) == 448.0 and C.e4m3_value(1) == 2.0 ** -9


@pytest.mark.parametrize("mass", [False, True])
@pytest.mark.parametrize("seed,B,HQ,HKV,Lc,W,ppm", [(1000, 1, 4, 4, 1024, 128, 50_000),
                                                     (1001, 2, 8, 2, 700, 64, 100_000),
                                                     (5, 1, 8, 8, 300, 0, 1_000_000)])
def test_selection_identical(mass, seed, B, HQ, HKV, Lc, W, ppm):
    c = decode_case(seed, B, HQ, HKV, Lc, window=W, n_proxy=64, n_sinks=4)
    qp, k = _np(c.q_proxy), _np(c.k)
    want, S = (select_vertical_mass if mass else select_vertical)(qp, k, Lc, W, ppm)
    got, S2 = C.select_vertical(qp, k, Lc, W, ppm, mass=mass, threads=2)
    assert np.array_equal(want, got)
    np.testing.assert_allclose(S2, S, rtol=1e-12, atol=1e-12)
    assert C.vl_count(Lc - W, ppm) == vl_count(Lc - W, ppm)


@pytest.mark.parametrize("bits", [(4, 4), (8, 8), (4, 8)])
@pytest.mark.parametrize("seed,B,HQ,HKV,Lc,W,ppm", [(1000, 1, 4, 4, 1024, 128, 50_000),
                                                     (7, 2, 8, 2, 777, 100, 20_000),
                                                     (9, 1, 8, 1, 129, 128, 50_000)])
def test_decode_identical(bits, seed, B, HQ, HKV, Lc, W, ppm):
    c = decode_case(seed, B, HQ, HKV, Lc, window=W, n_proxy=64, n_sinks=4)
    q, k, v = _np(c.q), _np(c.k), _np(c.v)
    idx, _ = select_vertical(_np(c.q_proxy), k, Lc, W, ppm)
    P = max(0, Lc - W)
    want = hybrid_decode(q, k, v, Lc, P, idx, bits=bits[0], bits_v=bits[1])
    got = C.hybrid_decode(q, k, v, Lc, P, idx, bits=bits[0], bits_v=bits[1], threads=2)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)


@pytest.mark.parametrize("band", [False, True])
@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
@pytest.mark.parametrize("seed,HQ,HKV,Lc,W,ppm", [(41, 4, 2, 300, 64, 50_000), (44, 8, 2, 777, 200, 50_000),
                                                   (46, 4, 2, 257, 0, 0)])
def test_prefill_identical(band, dtype, seed, HQ, HKV, Lc, W, ppm):
    c = prefill_case(seed, 1, HQ, HKV, Lc, window=W, sink_frac=0.02)
    q, k, v = _np(c.q), _np(c.k), _np(c.v)
    idx = None
    if W < Lc and ppm:
        idx, _ = select_vertical(q[:, :, Lc - 64:Lc], k, Lc, W, ppm)
    want, a = hybrid_prefill(q, k, v, idx, W, dtype, return_abs=True, band=band)
    got, a2 = C.hybrid_prefill(q, k, v, idx, W, dtype, band=band, threads=2)
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)
    np.testing.assert_allclose(a2, a, rtol=1e-11, atol=1e-12)


def test_prefill_sampled_blocks_and_heads():
    c = prefill_case(8, 1, 8, 2, 600, window=64, sink_frac=0.02)
    q, k, v = _np(c.q), _np(c.k), _np(c.v)
    idx, _ = select_vertical(q[:, :, -64:], k, 600, 64, 50_000)
    want, _ = hybrid_prefill(q, k, v, idx, 64, "fp8", query_blocks=[0, 4], heads=[1, 6], return_abs=True)
    got, _ = C.hybrid_prefill(q, k, v, idx, 64, "fp8", query_blocks=[0, 4], heads=[1, 6])
    np.testing.assert_allclose(got, want, rtol=1e-11, atol=1e-12)
    assert not got[:, [0, 2, 3, 4, 5, 7]].any() and not got[:, :, 128:512].any()


@pytest.mark.parametrize("seed,B,HQ,HKV,Lc,W,ppm", [(1000, 1, 8, 2, 1024, 128, 50_000),
                                                   (1001, 2, 8, 8, 700, 64, 100_000),
                                                   (1002, 1, 6, 2, 500, 32, 20_000)])
def test_select_heads_identical(seed, B, HQ, HKV, Lc, W, ppm):
    from oracle.select import select_vertical_heads
    c = decode_case(seed, B, HQ, HKV, Lc, window=W, n_proxy=16, n_sinks=6)
    qp, k = _np(c.q_proxy), _np(c.k)
    ih, ik, us, _, _ = select_vertical_heads(qp, k, Lc, W, ppm)
    ih2, ik2, us2 = C.select_vertical_heads(qp, k, Lc, W, ppm, threads=2)
    assert np.array_equal(ih, ih2) and np.array_equal(ik, ik2) and np.array_equal(us, us2)


def test_e2m1_table_identical():
    from oracle.prefill import e2m1_values
    assert C.e2m1_values() == list(e2m1_values())
