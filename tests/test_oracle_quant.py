"""Pins for the oracle's asymmetric group quantiser (Algorithm 4 Quant, Eq. 9).

Each test checks a property fixed by the definition of a uniform asymmetric
grid over [min, max] of each contiguous group of 32 head_dim elements, not
the oracle's own formula.
"""
import numpy as np
import pytest
import torch

from oracle.quant import QuantRangeError, dequantize, quantize, round_up_fp16


def bf16_rows(seed, n, d=128, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(n, d, generator=g) * scale
    # give the four groups very different ranges so a wrong grouping axis shows
    x = x * torch.tensor([0.01, 1.0, 30.0, 0.3]).repeat_interleave(d // 4)
    return x.to(torch.bfloat16).double().numpy()


def test_round_up_fp16_is_smallest_half_not_below():
    rng = np.random.default_rng(0)
    x = np.concatenate([rng.standard_normal(2000) * 10.0 ** rng.integers(-6, 4, 2000),
                        [0.0, 1.0, 65504.0, 6e-8]])
    h = round_up_fp16(x).astype(np.float64)
    assert np.all(h >= x)
    below = np.nextafter(round_up_fp16(x), np.float16(-np.inf)).astype(np.float64)
    assert np.all(below < x)


def _brute_force_codes(x, s, z, qmax):
    """For every element, the index of the exactly nearest grid point z + c*s
    (rational arithmetic over all qmax + 1 candidates), ties to the even
    index; 0 for a zero step."""
    from fractions import Fraction
    out = np.zeros(x.shape, np.int64)
    for idx in np.ndindex(x.shape):
        sf, zf, xf = Fraction(float(s[idx])), Fraction(float(z[idx])), Fraction(float(x[idx]))
        if sf == 0:
            continue
        dist = [abs(xf - (zf + c * sf)) for c in range(qmax + 1)]
        best = min(dist)
        cands = [c for c in range(qmax + 1) if dist[c] == best]
        out[idx] = cands[0] if len(cands) == 1 else [c for c in cands if c % 2 == 0][0]
    return out


@pytest.mark.parametrize("bits", [4, 8])
def test_codes_are_nearest_grid_points_brute_force(bits):
    x = bf16_rows(1, 16)
    c, s, z = quantize(x, bits)
    qmax = (1 << bits) - 1
    xs = x.reshape(16, 4, 32)
    want = _brute_force_codes(xs, np.broadcast_to(s[..., None], xs.shape), np.broadcast_to(z[..., None], xs.shape),
                              qmax)
    assert np.array_equal(c.reshape(16, 4, 32).astype(np.int64), want)
    assert c.max() <= qmax and c.dtype == np.uint8


def _tie_rows(bits):
    """Rows whose elements sit exactly on a midpoint z + (c + 1/2) s, one BF16
    step either side of it, and far from it: per group the minimum 0 and the
    maximum qmax * 2^-k fix s = 2^-k and z = 0, and the remaining elements
    are chosen on that grid."""
    qmax = (1 << bits) - 1
    rows = []
    for k in (0, 3, 6):
        step = 2.0 ** -k
        for base in range(0, qmax, max(1, qmax // 7)):
            mid = (base + 0.5) * step
            vals = [0.0, qmax * step, mid, float(np.nextafter(np.float32(mid), np.float32(np.inf))),
                    float(np.nextafter(np.float32(mid), np.float32(-np.inf))), base * step, (base + 1) * step]
            g = (vals * 5)[:32]
            rows.append(g)
    n = len(rows) // 4 * 4
    x = np.array(rows[:n], np.float64).reshape(-1, 128)
    return torch.from_numpy(x).to(torch.bfloat16).double().numpy()


@pytest.mark.parametrize("bits", [4, 8])
def test_codes_at_exact_midpoints_go_to_even(bits):
    """Planted ties and near-ties: exact midpoints take the even code; BF16
    neighbours of a midpoint take the nearer code (brute force, exact)."""
    x = _tie_rows(bits)
    qmax = (1 << bits) - 1
    c, s, z = quantize(x, bits)
    xs = x.reshape(x.shape[0], 4, 32)
    want = _brute_force_codes(xs, np.broadcast_to(s[..., None], xs.shape), np.broadcast_to(z[..., None], xs.shape),
                              qmax)
    assert np.array_equal(c.reshape(xs.shape).astype(np.int64), want)
    # some elements really are ties (the test plants them)
    u = (xs - z.astype(np.float64)[..., None]) / s.astype(np.float64)[..., None]  # exact: s is a power of two
    assert np.count_nonzero(u - np.floor(u) == 0.5) > 10


def test_error_bound_half_step_over_contiguous_groups():
    x = bf16_rows(2, 256)
    xh = dequantize(*quantize(x))
    xs = x.reshape(256, 4, 32)
    rng_ = xs.max(-1) - xs.min(-1)
    err = np.abs(x - xh).reshape(256, 4, 32).max(-1)
    mn = xs.min(-1)
    z_err = np.abs(mn - mn.astype(np.float16).astype(np.float64))
    # half a grid step (range/15/2), widened by the fp16 rounding of the step
    # (at most 2^-10 relative) and of the zero point.
    assert np.all(err <= rng_ / 30.0 * (1 + 2 ** -9) + z_err + 1e-12)


def _exact_min_step_check(x, s):
    """s is the smallest float16 with 15 s >= max - min, in exact arithmetic."""
    from fractions import Fraction
    xs = x.reshape(-1, 4, 32)
    sf = s.reshape(-1, 4)
    for i in range(xs.shape[0]):
        for q in range(4):
            rng_ = Fraction(float(xs[i, q].max())) - Fraction(float(xs[i, q].min()))
            h = sf[i, q]
            assert 15 * Fraction(float(h)) >= rng_
            if float(h) > 0:
                below = np.nextafter(h, np.float16(-np.inf))
                assert 15 * Fraction(float(below)) < rng_


def test_step_is_smallest_fp16_covering_the_range():
    x = bf16_rows(3, 128)
    c, s, z = quantize(x)
    _exact_min_step_check(x, s)
    xs = x.reshape(128, 4, 32)
    assert np.all(z.astype(np.float64) <= xs.min(-1) + np.abs(xs.min(-1)) * 2 ** -11 + 1e-30)


def test_step_is_exact_for_extreme_spans():
    """Groups whose range is a tiny amount above 15 * (a float16 value): a
    float64 quotient would round down onto that value, the exact step is the
    next float16 up."""
    rows = np.zeros((6, 128))
    for i, (hi, tiny) in enumerate([(15.0, 2.0 ** -80), (7.5, 2.0 ** -90), (30.0, 2.0 ** -70),
                                    (15.0, 0.0), (3.0, 2.0 ** -100), (1.5, 2.0 ** -60)]):
        rows[i, 0] = hi
        rows[i, 1] = -tiny          # min is a tiny negative bf16 value
    c, s, z = quantize(rows)
    _exact_min_step_check(rows, s)
    assert float(s[0, 0]) == float(np.nextafter(np.float16(1.0), np.float16(2)))
    assert float(s[3, 0]) == 1.0


def test_ties_round_half_to_even():
    # group 0: min 0, max 15 -> s = 1, z = 0; x = k + 0.5 lands on exact ties
    row = np.zeros(128)
    row[0], row[1] = 0.0, 15.0
    row[2:10] = [0.5, 1.5, 2.5, 3.5, 4.5, 5.5, 6.5, 14.5]
    c, s, z = quantize(row[None])
    assert float(s[0, 0]) == 1.0 and float(z[0, 0]) == 0.0
    assert c[0, 2:10].tolist() == [0, 2, 2, 4, 4, 6, 6, 14]


def test_constant_group_has_zero_scale_and_codes():
    row = np.full((1, 128), 0.75)
    row[0, 32:64] = np.linspace(-1, 1, 32).astype(np.float32)
    row[0, 32:64] = torch.tensor(row[0, 32:64]).to(torch.bfloat16).double().numpy()
    c, s, z = quantize(row)
    assert float(s[0, 0]) == 0.0 and np.all(c[0, :32] == 0)
    assert np.all(dequantize(c, s, z)[0, :32] == 0.75)
    assert float(s[0, 1]) > 0


def test_two_valued_group_reconstructs_min_and_max_exactly():
    row = np.zeros((1, 128))
    row[0, :32] = np.where(np.arange(32) % 3 == 0, -1.5, 6.0)   # (6+1.5)/15 = 0.5 exact
    c, s, z = quantize(row)
    xh = dequantize(c, s, z)
    assert np.array_equal(xh[0, :32], row[0, :32])


def test_power_of_two_scaling_equivariance():
    x = bf16_rows(4, 32)
    c1, s1, z1 = quantize(x)
    c2, s2, z2 = quantize(x * 4.0)
    assert np.array_equal(c1, c2)
    assert np.array_equal(s1.astype(np.float64) * 4, s2.astype(np.float64))
    assert np.array_equal(z1.astype(np.float64) * 4, z2.astype(np.float64))


def test_groups_are_independent():
    x = bf16_rows(5, 16)
    y = x.copy()
    y[:, 32:64] *= 8.0
    c1, s1, z1 = quantize(x)
    c2, s2, z2 = quantize(y)
    for gi in (0, 2, 3):
        sl = slice(32 * gi, 32 * gi + 32)
        assert np.array_equal(c1[:, sl], c2[:, sl])
        assert np.array_equal(s1[:, gi], s2[:, gi]) and np.array_equal(z1[:, gi], z2[:, gi])
    assert not np.array_equal(s1[:, 1], s2[:, 1])


def test_8bit_is_finer_than_4bit():
    x = bf16_rows(6, 64)
    e4 = np.abs(dequantize(*quantize(x, 4)) - x).mean()
    e8 = np.abs(dequantize(*quantize(x, 8)) - x).mean()
    assert e8 < e4 / 8


@pytest.mark.parametrize("bad", [-70000.0, 1.0e6, np.nan])
def test_out_of_range_is_an_error(bad):
    # -70000: the zero point (group min) overflows float16;
    # 1e6: the step (range / 15) overflows float16.
    row = np.zeros((1, 128))
    row[0, 5] = bad
    with pytest.raises(QuantRangeError):
        quantize(row)


def test_large_but_representable_group_is_fine():
    row = np.zeros((1, 128))
    row[0, 5] = 70000.0          # step 4667 and zero 0 are finite float16
    c, s, z = quantize(row)
    assert c[0, 5] == 15 and np.all(c[0, :5] == 0)


@pytest.mark.parametrize("bits", [4, 8])
def test_tie_rows_plant_exact_midpoints_and_neighbours(bits):
    """The GPU tie workload really contains exact midpoints (decided to the
    even code) and near-midpoints, and its codes agree with exact rational
    brute force."""
    from tests.gpu_util import tie_rows
    x = tie_rows(7, (6, 128), bits).double().numpy()
    qmax = (1 << bits) - 1
    c, s, z = quantize(x, bits)
    xs = x.reshape(6, 4, 32)
    sd, zd = s.astype(np.float64)[..., None], z.astype(np.float64)[..., None]
    u = (xs - zd) / sd
    assert np.count_nonzero(u - np.floor(u) == 0.5) >= 20
    want = _brute_force_codes(xs, np.broadcast_to(sd, xs.shape), np.broadcast_to(zd, xs.shape), qmax)
    assert np.array_equal(c.reshape(xs.shape).astype(np.int64), want)
    # the float32 recipe (x - z) * fl32(1/s) really differs from the exact codes somewhere
    r32 = (np.float32(1.0) / s.astype(np.float32))[..., None]
    t32 = ((xs.astype(np.float32) - z.astype(np.float32)[..., None]) * r32).astype(np.float32)
    rec = np.clip(np.rint(t32), 0, qmax)
    assert np.count_nonzero(rec != want) > 0
