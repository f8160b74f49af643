"""Shared helpers for the GPU parity tests."""
import os
import time

import numpy as np
import torch

# BF16 attention outputs: |gpu - oracle| <= ATOL + RTOL * |oracle| elementwise.
ATOL = 2e-3
RTOL = 1e-2


def assert_attention_close(got, want, atol=ATOL, rtol=RTOL, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    bound = atol + rtol * np.abs(want)
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                           f"max abs err {err.max():.3e}, worst excess {(err - bound).max():.3e}")
    return float(err.max())


def to_np(t: torch.Tensor) -> np.ndarray:
    return t.detach().to("cpu", torch.float64).numpy()


def mixed_rows(seed, shape):
    """BF16 rows whose 4 groups have very different ranges, plus special rows:
    constant groups, exact .5 ties, tiny (subnormal-scale) ranges."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(*shape, generator=g)
    x = x * torch.tensor([0.01, 1.0, 30.0, 0.3]).repeat_interleave(32)
    n = shape[-2]
    flat = x.view(-1, n, 128)
    for s in range(flat.shape[0]):
        if n > 3:
            flat[s, 1, :32] = 0.75                                    # constant group
            flat[s, 2, :32] = torch.arange(32) % 16 + 0.5             # ties on a unit grid
            flat[s, 2, 0], flat[s, 2, 1] = 0.0, 15.0
            flat[s, 3, 32:64] = 1e-6 * torch.randn(32, generator=g)  # subnormal-size step
    return x.to(torch.bfloat16)


# Prefill: the probabilities enter the P.V product rounded to BF16 (unit
# roundoff 2^-8), which can move an output element by at most 2^-8 times the
# softmax-weighted mean of |v| over its keys (``a`` from the oracle).
P_ROUND = 2.0 ** -8


def assert_prefill_close(got, want, a, what=""):
    got = np.asarray(got, dtype=np.float64)
    want = np.asarray(want, dtype=np.float64)
    a = np.asarray(a, dtype=np.float64)
    assert got.shape == want.shape == a.shape
    assert np.all(np.isfinite(got)), f"{what}: non-finite output"
    err = np.abs(got - want)
    bound = ATOL + RTOL * np.abs(want) + P_ROUND * a
    bad = err > bound
    assert not bad.any(), (f"{what}: {bad.sum()} of {bad.size} outside tolerance; "
                           f"max abs err {err.max():.3e}, worst excess {(err - bound).max():.3e}")
    return float(err.max())


def sample_pairs(B, HKV, n, tag):
    """n distinct (sequence, KV head) pairs for a sampled full-size parity
    check, always including the first and the last pair.  The others come
    from a seed that changes from run to run (so that, over runs, every pair
    gets checked); set HYQ_SAMPLE_SEED to replay one.  The seed is printed
    and returned, so a failure message can name it."""
    seed = int(os.environ.get("HYQ_SAMPLE_SEED", time.time_ns() % (1 << 31)))
    rng = np.random.default_rng([seed, sum(map(ord, tag))])
    pairs = [(0, 0), (B - 1, HKV - 1)]
    rest = [(b, h) for b in range(B) for h in range(HKV) if (b, h) not in pairs]
    for i in rng.choice(len(rest), size=min(max(n - 2, 0), len(rest)), replace=False):
        pairs.append(rest[int(i)])
    print(f"{tag}: HYQ_SAMPLE_SEED={seed} pairs={pairs}")
    return pairs, seed


def tie_rows(seed, shape, bits=4):
    """BF16 rows whose groups of 32 sit on grids with awkward steps (3, 5, 7,
    9, 11 or 13 times a power of two: their reciprocals are inexact in
    float32) and whose elements include exact midpoints z + (k + 1/2) s and
    their BF16 neighbours, where a float32 code decision can go to the wrong
    side.  Per group: the minimum -m s and the maximum (qmax - m) s fix the
    step s and the zero -m s exactly; the other elements are drawn from the
    half-integer multiples of s (and their BF16 neighbours) that BF16
    represents."""
    qmax = (1 << bits) - 1
    rng = np.random.default_rng(seed)
    n_groups = int(np.prod(shape[:-1])) * (shape[-1] // 32)
    out = np.zeros((n_groups, 32))
    for gi in range(n_groups):
        while True:
            mant = int(rng.choice([3, 5, 7, 9, 11, 13]))
            step = mant * 2.0 ** int(rng.integers(-12, -3))
            m = int(rng.integers(0, 8))
            units = np.arange(-2 * m, 2 * (qmax - m) + 1) / 2.0           # half-integer multiples
            vals = units * step
            exact = torch.tensor(vals).to(torch.bfloat16).double().numpy() == vals
            cand = vals[exact & (units != np.floor(units))]                # representable midpoints
            ends = np.array([-m * step, (qmax - m) * step])
            ends_ok = np.all(torch.tensor(ends).to(torch.bfloat16).double().numpy() == ends)
            if ends_ok and len(cand) >= 4:
                break
        g = [-m * step, (qmax - m) * step]
        for x in rng.choice(cand, 30):
            b = torch.tensor([x]).to(torch.bfloat16)
            pick = int(rng.integers(0, 3))
            if pick:
                # the BF16 neighbour above (pick 1) or below (pick 2)
                bits16 = b.view(torch.int16).item()
                sign = 1 if x > 0 else -1
                b = torch.tensor([bits16 + (sign if pick == 1 else -sign)], dtype=torch.int16).view(torch.bfloat16)
            g.append(b.double().item())
        out[gi] = np.array(g)[rng.permutation(32)]
    return torch.from_numpy(out.reshape(shape)).to(torch.bfloat16)


def double_rounding_cases(dtype, want=16):
    """Tile maxima A and values x (BF16, 0 < x <= A) for which rounding the
    float32 quotient fl32(x / s) to the code grid, s = RN_fp32(A / c) (c = 127
    for INT8, 448 for FP8, 6 for FP4), gives another code than rounding the
    exact quotient x / s.  Exhaustive over the 128 BF16 mantissas of A in [1, 2)
    and every positive BF16 x <= A (scaling A and x by a power of two scales s
    exactly and changes nothing); returned largest quotient first, at most
    ``want`` pairs (A, x)."""
    from oracle.prefill import e2m1_values, e4m3_values, nearest_grid_index
    c, grid = {"int8": (127.0, np.arange(128.0)), "fp8": (448.0, e4m3_values()),
               "fp4": (6.0, e2m1_values())}[dtype]
    u = torch.arange(1, 0x4000, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).double().numpy()
    u = u[np.isfinite(u) & (u > 0)]
    cases = []
    for mant in range(128):
        A = 1.0 + mant / 128.0
        s = np.float32(np.float32(A) / np.float32(c))
        x = u[u <= A]
        t32 = (x.astype(np.float32) / s).astype(np.float64)
        bad = nearest_grid_index(t32, 1.0, grid) != nearest_grid_index(x, np.float64(s), grid)
        cases += [(float(t), A, float(xx)) for t, xx in zip(t32[bad], x[bad])]
    cases.sort(reverse=True)
    return [(A, x) for _, A, x in cases[:want]]
