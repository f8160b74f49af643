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
