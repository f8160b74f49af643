"""Pins for the oracle's hybrid prefill operator (Eq. 6-7, Algorithm 2)."""
import numpy as np
import pytest
import torch
import torch.nn.functional as F

from gen import prefill_case
from oracle.prefill import (C_B, causal_attention, hybrid_prefill, quantize_symmetric)
from oracle.select import select_vertical


def _np(c):
    return c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy()


def _sdpa_causal(q, k, v):
    g = q.shape[1] // k.shape[1]
    K = torch.from_numpy(k).repeat_interleave(g, 1)
    V = torch.from_numpy(v).repeat_interleave(g, 1)
    return F.scaled_dot_product_attention(torch.from_numpy(q), K, V, is_causal=True).numpy()


def test_causal_reference_matches_torch():
    q, k, v = _np(prefill_case(0, 1, 4, 2, 200, d=64))
    np.testing.assert_allclose(causal_attention(q, k, v), _sdpa_causal(q, k, v), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_window_covering_sequence_is_exact(dtype):
    q, k, v = _np(prefill_case(1, 1, 4, 2, 150, d=64))
    o = hybrid_prefill(q, k, v, None, window=150, dtype=dtype)
    np.testing.assert_allclose(o, _sdpa_causal(q, k, v), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_full_ratio_is_exact(dtype):
    c = prefill_case(2, 1, 4, 2, 300, d=64, window=32)
    q, k, v = _np(c)
    idx = np.broadcast_to(np.arange(268), (1, 2, 268))
    o = hybrid_prefill(q, k, v, idx, window=32, dtype=dtype)
    np.testing.assert_allclose(o, _sdpa_causal(q, k, v), rtol=1e-12, atol=1e-13)


def test_int8_codes_are_integers_with_max_at_127():
    rng = np.random.default_rng(3)
    x = rng.standard_normal((64, 128))
    xh, c, s = quantize_symmetric(x, None, "int8")
    assert np.array_equal(c, np.rint(c)) and np.abs(c).max() == 127
    assert np.abs(xh - x).max() <= s.max() / 2 + 1e-15
    # integer tile products are exact in float64: the scaled product equals the
    # product of dequantised operands
    y = rng.standard_normal((16, 128))
    yh, cy, sy = quantize_symmetric(y, None, "int8")
    np.testing.assert_allclose((cy @ c.T) * (s * sy), yh @ xh.T, rtol=1e-12, atol=1e-12)


def test_fp8_codes_are_e4m3_values_with_max_at_448():
    rng = np.random.default_rng(4)
    x = rng.standard_normal((64, 128)) * 3
    xh, c, s = quantize_symmetric(x, 0, "fp8")          # per-channel scales
    assert np.abs(c).max(axis=0).min() == 448.0
    table = set(_e4m3_values().values())
    assert all(v in table for v in np.unique(c))        # every code is an e4m3 value
    rel = np.abs(xh - x) / np.maximum(np.abs(x), 1e-3)
    assert np.median(rel) < 2 ** -4                     # 3-bit mantissa


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_hybrid_beats_uniform_low_bit(dtype):
    c = prefill_case(5, 1, 4, 2, 512, d=128, window=64, sink_frac=0.02, sink_gain=20.0, q_gain=4.0)
    q, k, v = _np(c)
    ex = causal_attention(q, k, v)
    idx, _ = select_vertical(q[:, :, -64:], k, 512, 64, 50_000)
    hyb = hybrid_prefill(q, k, v, idx, window=64, dtype=dtype)
    uni = hybrid_prefill(q, k, v, None, window=0, dtype=dtype)
    e_h = np.mean((hyb - ex) ** 2)
    e_u = np.mean((uni - ex) ** 2)
    assert e_h < e_u
    assert e_h < 1e-3


def test_causality():
    c = prefill_case(6, 1, 2, 1, 256, d=64, window=32)
    q, k, v = _np(c)
    idx, _ = select_vertical(q[:, :, -32:], k, 256, 32, 50_000)
    o1 = hybrid_prefill(q, k, v, idx, window=32)
    k2, v2 = k.copy(), v.copy()
    k2[:, :, 200:] += 5.0
    v2[:, :, 200:] -= 3.0
    o2 = hybrid_prefill(q, k2, v2, idx, window=32)
    # rows before 200 see neither the changed keys nor values ...
    # ... except through the per-tile quantisation scales of tiles that mix
    # positions < 200 and >= 200, so compare only rows whose tiles are untouched.
    assert np.array_equal(o1[:, :, :128], o2[:, :, :128])
    assert not np.array_equal(o1[:, :, 230:], o2[:, :, 230:])


def _e4m3_values():
    """All finite e4m3 (fn) values from the format's definition: 1 sign bit,
    4 exponent bits (bias 7), 3 mantissa bits, subnormals at exponent 0, the
    all-ones pattern (S.1111.111) is NaN, no infinities; max 448."""
    vals = {}
    for bits in range(256):
        s, e, m = bits >> 7, (bits >> 3) & 0xF, bits & 7
        if e == 15 and m == 7:
            continue
        mag = (m / 8.0) * 2.0 ** -6 if e == 0 else (1.0 + m / 8.0) * 2.0 ** (e - 7)
        vals[bits] = -mag if s else mag
    return vals


def test_oracle_e4m3_table_matches_the_bit_patterns():
    """The oracle's e4m3 value list (built from the format) equals the
    non-negative finite values of the 256 bit patterns, decoded here by
    hand and by torch's float8_e4m3fn type."""
    from oracle.prefill import e4m3_values
    by_hand = sorted({v for v in _e4m3_values().values() if v >= 0})
    assert list(e4m3_values()) == by_hand and len(by_hand) == 127 and by_hand[-1] == 448.0
    u8 = torch.arange(256, dtype=torch.uint8)
    dec = u8.view(torch.float8_e4m3fn).double().numpy()
    for bits, v in _e4m3_values().items():
        assert dec[bits] == v


def _exact_nearest(x, s, grid_pos, even_of):
    """Brute force over the signed grid with exact rationals: the grid value
    nearest to x / s, ties to the candidate whose ``even_of`` is true."""
    from fractions import Fraction
    q = Fraction(float(x)) / Fraction(float(s))
    cands = sorted({Fraction(g) for g in grid_pos} | {-Fraction(g) for g in grid_pos})
    best = min(abs(q - c) for c in cands)
    near = [c for c in cands if abs(q - c) == best]
    if len(near) == 1:
        return float(near[0])
    return float([c for c in near if even_of(abs(float(c)))][0])


def _tie_inputs(grid, s, rng, n_rand):
    """Values x with x / s at exact midpoints of the grid, one float64 step
    either side of them, and random ones."""
    mids = (grid[:-1] + grid[1:]) / 2
    pick = mids[rng.choice(len(mids), min(40, len(mids)), replace=False)]
    xs = np.concatenate([pick * s, np.nextafter(pick * s, np.inf), np.nextafter(pick * s, -np.inf),
                         rng.uniform(0, grid[-1] * s, n_rand)])
    return np.concatenate([xs, -xs])


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
@pytest.mark.parametrize("s_mant", [1.0, 3.0, 1.0 + 2.0 ** -23])
def test_codes_are_nearest_to_the_exact_quotient(dtype, s_mant):
    """Codes against exact rational brute force: planted exact midpoints go
    to the even code, their float64 neighbours to the nearer code."""
    from oracle.prefill import C_B, _codes, e2m1_values, e4m3_values
    grid = {"fp8": e4m3_values(), "fp4": e2m1_values()}.get(dtype, np.arange(128.0))
    s = float(np.float32(s_mant * 2.0 ** -7))
    rng = np.random.default_rng(13)
    x = _tie_inputs(grid, s, rng, 100)
    got = _codes(x, np.float64(s), dtype)
    idx = {float(v): i for i, v in enumerate(grid)}
    want = [_exact_nearest(xi, s, grid, lambda a: idx[a] % 2 == 0) for xi in x]
    np.testing.assert_array_equal(got, np.array(want))
    # beyond the top of the grid: saturate
    assert _codes(np.array([grid[-1] * s * 1.5]), np.float64(s), dtype)[0] == grid[-1]
    assert C_B[dtype] == grid[-1]


def test_int8_scale_is_one_float32_rounding():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((64, 128)).astype(np.float32).astype(np.float64)
    _, c, s = quantize_symmetric(x, None, "int8")
    from fractions import Fraction
    q = Fraction(float(np.abs(x).max())) / 127                 # the exact quotient
    f = np.float32(s.item())
    assert float(f) == s.item()                                 # a float32 number ...
    for nb in (np.nextafter(f, np.float32(np.inf)), np.nextafter(f, np.float32(-np.inf))):
        assert abs(Fraction(float(f)) - q) <= abs(Fraction(float(nb)) - q)   # ... nearest to it
    assert np.abs(c).max() == 127.0


def test_value_tiles_share_one_scale():
    """One scale per key tile for V too: a huge channel in every value row
    drives the other channels' INT8 codes to zero, so rows that attend only
    to quantised keys get exactly zero in those channels."""
    L, W = 200, 8
    rng = np.random.default_rng(13)
    q = rng.standard_normal((1, 2, L, 64))
    k = rng.standard_normal((1, 1, L, 64))
    v = rng.uniform(-1, 1, (1, 1, L, 64)).astype(np.float32).astype(np.float64)
    v[..., 0] = 1000.0
    o = hybrid_prefill(q, k, v, None, window=W, dtype="int8")
    assert np.all(o[:, :, :L - W, 1:] == 0.0)
    assert np.all(o[:, :, L - W:, 1:] != 0.0)


def test_restricted_blocks_equal_full_computation():
    c = prefill_case(7, 1, 4, 2, 300, d=64, window=32)
    q, k, v = _np(c)
    idx, _ = select_vertical(q[:, :, -32:], k, 300, 32, 50_000)
    full = hybrid_prefill(q, k, v, idx, window=32, dtype="fp8")
    part = hybrid_prefill(q, k, v, idx, window=32, dtype="fp8", query_blocks=[0, 2], heads=[1, 2])
    for h in (1, 2):
        for blk in (0, 2):
            rows = slice(128 * blk, min(300, 128 * blk + 128))
            np.testing.assert_array_equal(part[0, h, rows], full[0, h, rows])
    assert np.all(part[0, 0] == 0) and np.all(part[0, 1, 128:256] == 0)


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_abs_weighted_values(dtype):
    """``a`` is the operator applied to |V| (symmetric quantisation commutes
    with |.|), and bounds |o| by the triangle inequality."""
    c = prefill_case(8, 1, 4, 2, 260, d=64, window=32)
    q, k, v = _np(c)
    idx, _ = select_vertical(q[:, :, -32:], k, 260, 32, 50_000)
    o, a = hybrid_prefill(q, k, v, idx, window=32, dtype=dtype, return_abs=True)
    np.testing.assert_array_equal(o, hybrid_prefill(q, k, v, idx, window=32, dtype=dtype))
    np.testing.assert_allclose(a, hybrid_prefill(q, k, np.abs(v), idx, window=32, dtype=dtype),
                               rtol=1e-13, atol=1e-15)
    assert np.all(a >= np.abs(o) - 1e-15)


# --- the per-query band (``band=True``): query i sees (i - W, i] in BF16 ---

def _vl(P, n, seed, early=16):
    """[1, 2, n] ascending vertical-line positions in [0, P); the first KV
    head's set has four positions below ``early`` (inside the first window)."""
    rng = np.random.default_rng(seed)
    e = rng.choice(min(early, P), size=4, replace=False)
    rest = rng.choice(np.setdiff1d(np.arange(P), e), size=n - 4, replace=False)
    return np.stack([np.sort(np.concatenate([e, rest])), np.sort(rng.choice(P, size=n, replace=False))])[None]


def _exactly_quantisable(seed, L, d, dtype):
    """Q [1,4,L,d], K, V [1,2,L,d] whose every tile quantises without error:
    each value is a code (an integer in [-127, 127], an e4m3 or an e2m1
    value) times 2^-7 (INT8), 2^-9 (FP8) or 2^-2 (FP4), and every row holds
    the largest code, so every
    tile's scale is exactly that power of two and x / s is the code itself."""
    rng = np.random.default_rng(seed)
    if dtype == "int8":
        codes, top, unit = np.arange(-127, 128, dtype=np.float64), 127.0, 2.0 ** -7
    elif dtype == "fp4":
        e = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
        codes, top, unit = np.array(sorted(set(e) | {-x for x in e})), 6.0, 2.0 ** -2
    else:
        codes, top, unit = np.array(sorted(_e4m3_values().values())), 448.0, 2.0 ** -9

    def mat(h):
        c = rng.choice(codes, size=(1, h, L, d))
        c[..., 0] = top
        return c * unit
    return mat(4), mat(2), mat(2)


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
@pytest.mark.parametrize("band", [False, True])
def test_exactly_quantisable_inputs_give_exact_attention(dtype, band):
    """With quantisation error-free, either window reading is exact causal
    attention at every row: no key is counted twice or left out by the
    segment masks (quantised prefix, vertical lines, window or band)."""
    L, W = 300, 48
    q, k, v = _exactly_quantisable(50, L, 64, dtype)
    idx = _vl(L - W, 12, 51)
    o = hybrid_prefill(q, k, v, idx, W, dtype, band=band)
    np.testing.assert_allclose(o, causal_attention(q, k, v), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_band_rows_inside_window_are_full_precision(dtype):
    """Rows i < W have every key j <= i inside their band: exact attention,
    unlike the fixed window, which quantises them; later rows quantise the
    keys W or more positions back."""
    L, W = 300, 64
    q, k, v = _np(prefill_case(52, 1, 4, 2, L, d=64, window=W, sink_frac=0.03))
    idx = _vl(L - W, 12, 53)
    ex = causal_attention(q, k, v)
    band = hybrid_prefill(q, k, v, idx, W, dtype, band=True)
    fixed = hybrid_prefill(q, k, v, idx, W, dtype)
    np.testing.assert_allclose(band[:, :, :W], ex[:, :, :W], rtol=1e-12, atol=1e-13)
    assert np.abs(fixed[:, :, 1:W] - ex[:, :, 1:W]).max() > 1e-6
    assert np.abs(band[:, :, W + 8:] - ex[:, :, W + 8:]).max() > 1e-6


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_band_agrees_with_fixed_window_on_last_row_and_without_window(dtype):
    """The last row's band (P - 1, L - 1] is the fixed window [P, L); with
    W = 0 both readings quantise every key but the vertical lines."""
    L, W = 300, 64
    q, k, v = _np(prefill_case(54, 1, 4, 2, L, d=64, window=W, sink_frac=0.03))
    idx = _vl(L - W, 12, 55)
    band = hybrid_prefill(q, k, v, idx, W, dtype, band=True)
    fixed = hybrid_prefill(q, k, v, idx, W, dtype)
    np.testing.assert_allclose(band[:, :, L - 1], fixed[:, :, L - 1], rtol=1e-12, atol=1e-13)
    assert np.abs(band[:, :, W:L - 1] - fixed[:, :, W:L - 1]).max() > 1e-6
    q0, k0, v0 = _np(prefill_case(56, 1, 4, 2, L, d=64, window=0, sink_frac=0.03))
    idx0 = _vl(L, 12, 57)
    np.testing.assert_allclose(hybrid_prefill(q0, k0, v0, idx0, 0, dtype, band=True),
                               hybrid_prefill(q0, k0, v0, idx0, 0, dtype), rtol=1e-12, atol=1e-13)


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_band_window_covering_sequence_is_exact(dtype):
    q, k, v = _np(prefill_case(58, 1, 4, 2, 150, d=64))
    o = hybrid_prefill(q, k, v, None, window=150, dtype=dtype, band=True)
    np.testing.assert_allclose(o, _sdpa_causal(q, k, v), rtol=1e-12, atol=1e-13)


def test_band_restricted_blocks_equal_full_computation():
    q, k, v = _np(prefill_case(59, 1, 4, 2, 300, d=64, window=32))
    idx = _vl(268, 10, 60)
    full = hybrid_prefill(q, k, v, idx, window=32, dtype="int8", band=True)
    part = hybrid_prefill(q, k, v, idx, window=32, dtype="int8", query_blocks=[1], heads=[3], band=True)
    np.testing.assert_array_equal(part[0, 3, 128:256], full[0, 3, 128:256])


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_double_rounding_cases_change_the_code_visibly(dtype):
    """The prefill tie workload: each planted value's exact code differs from
    the code of its rounded float32 quotient, by more than the parity
    tolerance once multiplied out at the test's scale (so a kernel that
    rounds twice fails the GPU test)."""
    from oracle.prefill import C_B, _codes, e2m1_values, e4m3_values, nearest_grid_index
    from tests.gpu_util import double_rounding_cases
    grid = {"int8": np.arange(128.0), "fp8": e4m3_values(), "fp4": e2m1_values()}[dtype]
    cases = double_rounding_cases(dtype)
    assert len(cases) >= 8
    for A, x in cases:
        A, x = A * 32, x * 32                           # the GPU test's scale: A in [32, 64)
        s = float(np.float32(np.float32(A) / np.float32(C_B[dtype])))
        exact = _codes(np.array([x]), np.float64(s), dtype)[0] * s
        t32 = float(np.float32(np.float32(x) / np.float32(s)))
        twice = grid[nearest_grid_index(np.array([t32]), 1.0, grid)[0]] * s
        tol = 2e-3 + 1e-2 * abs(exact) + 2.0 ** -8 * abs(exact)
        assert abs(exact - twice) > tol, (A, x, exact, twice)


def test_oracle_e2m1_table_is_the_two_bit_significand_grid():
    """e2m1 has one fraction bit and a subnormal step of 1/2 at the bottom of
    a two-bit exponent: its values are the multiples n/2 (0 <= n <= 12) whose
    integer n has at most two significant bits."""
    from oracle.prefill import C_B, e2m1_values
    want = [n / 2 for n in range(13) if n == 0 or (n >> (n.bit_length() - 2 if n.bit_length() > 1 else 0))
            << (n.bit_length() - 2 if n.bit_length() > 1 else 0) == n]
    assert e2m1_values().tolist() == want == [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]
    assert C_B["fp4"] == 6.0


def test_fp4_codes_are_e2m1_values_with_max_at_6():
    rng = np.random.default_rng(5)
    x = rng.standard_normal((64, 128)) * 3
    xh, c, s = quantize_symmetric(x, 0, "fp4")          # per-channel scales
    assert np.abs(c).max(axis=0).min() == 6.0
    assert set(np.unique(np.abs(c)).tolist()) <= {0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0}
    # the nearest grid value: within half the local spacing (0.5 below 2, 1 to 4, 2 to 6)
    t = np.abs(x) / s
    half = np.where(t < 2, 0.25, np.where(t < 4, 0.5, 1.0))
    assert np.all(np.abs(np.abs(c) - np.minimum(t, 6.0)) <= half + 1e-12)
