"""GPU parity of the hybrid prefill operator (Eq. 6-7, Algorithm 2) against
the oracle's float64 restatement, INT8, FP8 and FP4 (e2m1) main paths.

The vertical-line set fed to the GPU is the oracle's own selection from the
last min(64, L) queries, so the attention comparison does not depend on
selection parity.  Tolerance: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| + 2^-8 a,
where a = sum_j p_j |v_j| / sum_j p_j from the oracle: the last term bounds
the kernel's rounding of the probabilities to BF16 before the P.V product
(unit roundoff 2^-8), a step the oracle does not take.
"""
import numpy as np
import pytest
import torch

from gen import prefill_case
from hybrid_precision_quantized_gb300 import _lib as L
from hybrid_precision_quantized_gb300 import (hyq_prefill_attention, hyq_prefill_attention_band,
                                              hyq_read_device_error, make_config, workspace)
from oracle.prefill import hybrid_prefill
from oracle.select import select_vertical
from tests.gpu_util import assert_prefill_close, to_np

pytestmark = pytest.mark.gpu

DT = {"int8": L.PREFILL_INT8, "fp8": L.PREFILL_FP8, "fp4": L.PREFILL_FP4}


def vl_for(c, Lc, W, ppm):
    q = c.q.double().numpy()
    n_proxy = min(64, Lc)
    idx, _ = select_vertical(q[:, :, Lc - n_proxy:Lc], c.k.double().numpy(), Lc, W, ppm)
    return idx


def run_gpu(c, Lc, W, ppm, dtype, idx, ws_len=None, band=False):
    B, HQ = c.q.shape[:2]
    HKV = c.k.shape[1]
    cfg = make_config(B, HQ, HKV, capacity=max(Lc, ws_len or 0, 1), window=W, rho_ppm=ppm)
    kvl = idx.shape[-1]
    vl = torch.from_numpy(np.ascontiguousarray(idx)).to(torch.int32).cuda() if kvl else None
    ws = workspace(cfg, L.OP_PREFILL_BAND if band else L.OP_PREFILL, ws_len or Lc)
    out = torch.full((B, HQ, Lc, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    fn = hyq_prefill_attention_band if band else hyq_prefill_attention
    fn(cfg, DT[dtype], c.q.cuda(), c.k.cuda(), c.v.cuda(), Lc, vl, kvl, out, ws, err)
    torch.cuda.synchronize()
    assert hyq_read_device_error(err) == 0
    return to_np(out)


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
@pytest.mark.parametrize("seed,B,HQ,HKV,Lc,W,ppm", [
    (1, 1, 4, 2, 300, 64, 50_000),      # a few tiles, ragged tails in both lists
    (2, 1, 8, 2, 1000, 128, 50_000),
    (3, 2, 4, 4, 515, 128, 20_000),     # two sequences, MHA
    (4, 1, 16, 2, 777, 100, 50_000),    # g = 8
    (5, 1, 6, 2, 1100, 128, 100_000),   # g = 3, more vertical lines
])
def test_prefill_parity(hyq, dtype, seed, B, HQ, HKV, Lc, W, ppm):
    c = prefill_case(seed, B, HQ, HKV, Lc, window=W, sink_frac=0.02)
    idx = vl_for(c, Lc, W, ppm)
    got = run_gpu(c, Lc, W, ppm, dtype, idx)
    want, a = hybrid_prefill(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(), idx, W, dtype,
                             return_abs=True)
    assert_prefill_close(got, want, a, what=f"{dtype} L={Lc}")


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
@pytest.mark.parametrize("Lc,W,ppm,what", [
    (1, 128, 50_000, "single position"),
    (100, 128, 50_000, "sequence inside the window: all BF16"),
    (129, 128, 50_000, "P = 1"),
    (600, 0, 0, "rho = 0, W = 0: all quantised"),
    (600, 64, 1_000_000, "rho = 100%: no quantised keys"),
    (256, 64, 0, "exactly one quantised MMA tile and a window"),
    (257, 0, 0, "two query blocks, one row in the second"),
])
def test_prefill_edge_cases(hyq, dtype, Lc, W, ppm, what):
    c = prefill_case(21, 1, 4, 2, Lc, window=W, sink_frac=0.03)
    idx = vl_for(c, Lc, W, ppm) if W < Lc else np.zeros((1, 2, 0), np.int64)
    got = run_gpu(c, Lc, W, ppm, dtype, idx)
    want, a = hybrid_prefill(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(),
                             idx if idx.shape[-1] else None, W, dtype, return_abs=True)
    assert_prefill_close(got, want, a, what=what)


def test_prefill_workspace_reuse_and_larger_hint(hyq):
    """A workspace sized for a longer context serves a shorter call; two calls
    give identical bits."""
    c = prefill_case(31, 1, 8, 2, 700, window=128)
    idx = vl_for(c, 700, 128, 50_000)
    a = run_gpu(c, 700, 128, 50_000, "fp8", idx, ws_len=2048)
    b = run_gpu(c, 700, 128, 50_000, "fp8", idx)
    np.testing.assert_array_equal(a, b)


def test_prefill_bad_vertical_lines_flagged(hyq):
    c = prefill_case(32, 1, 4, 2, 400, window=64)
    cfg = make_config(1, 4, 2, capacity=400, window=64, rho_ppm=50_000)
    vl = torch.tensor([[[5, 3, 9]] * 2], dtype=torch.int32, device="cuda")   # not ascending
    ws = workspace(cfg, L.OP_PREFILL, 400)
    out = torch.empty(1, 4, 400, 128, dtype=torch.bfloat16, device="cuda")
    err = torch.zeros(1, dtype=torch.int32, device="cuda")
    hyq_prefill_attention(cfg, L.PREFILL_FP8, c.q.cuda(), c.k.cuda(), c.v.cuda(), 400, vl, 3, out, ws, err)
    torch.cuda.synchronize()
    assert hyq_read_device_error(err) & L.DEVERR_INDEX


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_prefill_llama_shaped_8k_sampled(hyq, dtype):
    """Llama-3.1-8B-shaped heads at 8K: every head of four query blocks (first,
    two middle, last) against the oracle."""
    Lc, W, ppm = 8192, 128, 50_000
    c = prefill_case(1005, 1, 32, 8, Lc, window=W, sink_frac=0.02)
    idx = vl_for(c, Lc, W, ppm)
    got = run_gpu(c, Lc, W, ppm, dtype, idx)
    blocks = [0, 17, 40, Lc // 128 - 1]
    want, a = hybrid_prefill(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(), idx, W, dtype,
                             query_blocks=blocks, return_abs=True)
    for blk in blocks:
        rows = slice(128 * blk, 128 * blk + 128)
        assert_prefill_close(got[:, :, rows], want[:, :, rows], a[:, :, rows], what=f"{dtype} block {blk}")


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_prefill_llama_shaped_32k_sampled(hyq, dtype):
    """The benchmark's prefill workload (Llama-3.1-8B-shaped heads, causal 32K,
    W 128, rho 5%): the GPU computes every head and query block; the oracle
    checks three query blocks (first, middle, last) of two heads (the first
    and the last KV group)."""
    Lc, W, ppm = 32768, 128, 50_000
    c = prefill_case(1006, 1, 32, 8, Lc, window=W, sink_frac=0.02)
    idx = vl_for(c, Lc, W, ppm)
    got = run_gpu(c, Lc, W, ppm, dtype, idx)
    blocks, heads = [0, 128, Lc // 128 - 1], [0, 31]
    want, a = hybrid_prefill(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(), idx, W, dtype,
                             query_blocks=blocks, heads=heads, return_abs=True)
    for hq in heads:
        for blk in blocks:
            rows = slice(128 * blk, 128 * blk + 128)
            assert_prefill_close(got[:, hq, rows], want[:, hq, rows], a[:, hq, rows],
                                 what=f"{dtype} head {hq} block {blk}")


# --- per-query band window (hyq_prefill_attention_band) --------------------

def oracle_band(c, idx, W, dtype, **kw):
    return hybrid_prefill(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(),
                          idx if idx.shape[-1] else None, W, dtype, return_abs=True, band=True, **kw)


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
@pytest.mark.parametrize("seed,B,HQ,HKV,Lc,W,ppm", [
    (41, 1, 4, 2, 300, 64, 50_000),     # a few tiles, ragged tails
    (42, 1, 8, 2, 1000, 128, 50_000),   # the band spans two key tiles per query block
    (43, 2, 4, 4, 515, 100, 20_000),    # W not a multiple of the tile, two sequences
    (44, 1, 16, 2, 777, 200, 50_000),   # W > one tile: up to three band tiles
    (45, 1, 6, 2, 1100, 1, 100_000),    # W = 1: the band is the query's own key
])
def test_prefill_band_parity(hyq, dtype, seed, B, HQ, HKV, Lc, W, ppm):
    c = prefill_case(seed, B, HQ, HKV, Lc, window=W, sink_frac=0.02)
    idx = vl_for(c, Lc, W, ppm)
    got = run_gpu(c, Lc, W, ppm, dtype, idx, band=True)
    want, a = oracle_band(c, idx, W, dtype)
    assert_prefill_close(got, want, a, what=f"band {dtype} L={Lc} W={W}")


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
@pytest.mark.parametrize("Lc,W,ppm,what", [
    (1, 128, 50_000, "single position"),
    (100, 128, 50_000, "sequence inside the window: all BF16"),
    (129, 128, 50_000, "P = 1"),
    (600, 0, 0, "W = 0: no band, all quantised"),
    (600, 64, 1_000_000, "rho = 100%: no quantised keys"),
    (257, 128, 50_000, "two query blocks, one row in the second"),
])
def test_prefill_band_edge_cases(hyq, dtype, Lc, W, ppm, what):
    c = prefill_case(46, 1, 4, 2, Lc, window=W, sink_frac=0.03)
    idx = vl_for(c, Lc, W, ppm) if W < Lc else np.zeros((1, 2, 0), np.int64)
    got = run_gpu(c, Lc, W, ppm, dtype, idx, band=True)
    want, a = oracle_band(c, idx, W, dtype)
    assert_prefill_close(got, want, a, what=what)


def test_prefill_band_last_row_matches_fixed_window(hyq):
    """Both GPU entry points give the same last row (its band is the fixed
    window) up to the summation order of the two kernels' tiles."""
    c = prefill_case(47, 1, 8, 2, 900, window=128)
    idx = vl_for(c, 900, 128, 50_000)
    band = run_gpu(c, 900, 128, 50_000, "fp8", idx, band=True)
    fixed = run_gpu(c, 900, 128, 50_000, "fp8", idx)
    np.testing.assert_allclose(band[:, :, -1], fixed[:, :, -1], rtol=1e-2, atol=2e-3)


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_prefill_band_llama_shaped_8k_sampled(hyq, dtype):
    """Llama-3.1-8B-shaped heads at 8K with the per-query band: every head of
    four query blocks (first, second, a middle one, last) against the oracle."""
    Lc, W, ppm = 8192, 128, 50_000
    c = prefill_case(1007, 1, 32, 8, Lc, window=W, sink_frac=0.02)
    idx = vl_for(c, Lc, W, ppm)
    got = run_gpu(c, Lc, W, ppm, dtype, idx, band=True)
    blocks = [0, 1, 40, Lc // 128 - 1]
    want, a = oracle_band(c, idx, W, dtype, query_blocks=blocks)
    for blk in blocks:
        rows = slice(128 * blk, 128 * blk + 128)
        assert_prefill_close(got[:, :, rows], want[:, :, rows], a[:, :, rows], what=f"band {dtype} block {blk}")


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_prefill_band_llama_shaped_32k_sampled(hyq, dtype):
    """The benchmark's band workload (Llama-3.1-8B-shaped heads, causal 32K,
    W 128, rho 5%, the window read per query): the GPU computes every head
    and query block; the oracle checks three query blocks (first, middle,
    last) of two heads (the first and the last KV group)."""
    Lc, W, ppm = 32768, 128, 50_000
    c = prefill_case(1006, 1, 32, 8, Lc, window=W, sink_frac=0.02)
    idx = vl_for(c, Lc, W, ppm)
    got = run_gpu(c, Lc, W, ppm, dtype, idx, band=True)
    blocks, heads = [0, 128, Lc // 128 - 1], [0, 31]
    want, a = oracle_band(c, idx, W, dtype, query_blocks=blocks, heads=heads)
    for hq in heads:
        for blk in blocks:
            rows = slice(128 * blk, 128 * blk + 128)
            assert_prefill_close(got[:, hq, rows], want[:, hq, rows], a[:, hq, rows],
                                 what=f"band {dtype} head {hq} block {blk}")


@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_prefill_codes_of_exact_quotients(hyq, dtype):
    """Values whose float32 quotient x / s lands exactly on a midpoint of the
    code grid while the exact quotient does not (found exhaustively, largest
    quotients first), one per 64-key tile: key 64t carries such a value and
    is the only key query row 64t + 1 attends to (one-hot query and key on
    dimension t, logit ~22), so that row's output is the dequantised value
    row, and a code decided by rounding twice falls outside the tolerance."""
    from types import SimpleNamespace
    from tests.gpu_util import double_rounding_cases
    cases = double_rounding_cases(dtype, want=12)
    T = len(cases)
    Lc = 64 * T + 2
    rng = np.random.default_rng(31)
    q = np.zeros((1, 1, Lc, 128))
    k = np.zeros((1, 1, Lc, 128))
    v = np.zeros((1, 1, Lc, 128))
    for t, (A, x) in enumerate(cases):
        A, x = A * 32, x * 32
        rows = slice(64 * t, 64 * t + 64)
        v[0, 0, rows] = rng.uniform(-A / 4, A / 4, (64, 128))
        v[0, 0, 64 * t + 5, 7] = A                        # the tile maximum
        v[0, 0, 64 * t, 3 + t] = x                        # the planted value
        k[0, 0, 64 * t, t] = 16.0
        q[0, 0, 64 * t + 1, t] = 16.0
    c = SimpleNamespace(q=torch.from_numpy(q).to(torch.bfloat16), k=torch.from_numpy(k).to(torch.bfloat16),
                        v=torch.from_numpy(v).to(torch.bfloat16))
    idx = np.zeros((1, 1, 0), np.int64)
    got = run_gpu(c, Lc, 0, 0, dtype, idx)
    want, a = hybrid_prefill(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(), None, 0, dtype,
                             return_abs=True)
    rows = [64 * t + 1 for t in range(T)]
    assert_prefill_close(got[:, :, rows], want[:, :, rows], a[:, :, rows], what=f"{dtype} planted quotients")


@pytest.mark.parametrize("band", [False, True])
@pytest.mark.parametrize("dtype", ["int8", "fp8", "fp4"])
def test_prefill_late_score_jumps(hyq, dtype, band):
    """Keys planted late in the row whose logits rise far above the row's
    earlier maximum: at positions 430 and 700 (quantised segment, kept out of
    the vertical-line list) and 940 (inside the BF16 window).  Over the rows
    that see them the rise spreads from below 0 to ~17, ~26 and ~45 (log2
    units; medians ~8, ~14 and ~25), so many rows' running maximum trails the
    tile maximum by 2^8 to 2^16 (terms formed against the stale maximum) and
    many by more (the maximum has to move); the result is the same softmax
    either way."""
    Lc, W, ppm = 1000, 128, 50_000
    c = prefill_case(41, 1, 4, 2, Lc, window=W, sink_frac=0.02)
    idx = vl_for(c, Lc, W, ppm)
    k = c.k.double().clone()
    for h in range(2):
        u = c.u[0, h].double()
        for pos, gain in ((430, 47.0), (700, 102.0), (940, 200.0)):
            assert pos not in set(idx[0, h].tolist())
            k[0, h, pos] = gain * u
    c.k = k.to(torch.bfloat16)
    got = run_gpu(c, Lc, W, ppm, dtype, idx, band=band)
    want, a = hybrid_prefill(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(), idx, W, dtype,
                             return_abs=True, band=band)
    assert_prefill_close(got, want, a, what=f"{dtype} late jumps band={band}")
