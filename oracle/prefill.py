"""Hybrid-precision prefill operator.

Follows *HyQuant: Hybrid-Precision Quantization for LLM Attention*,
§4.2 Eq. 6-7 and Appendix A.2, Algorithm 2:

    O = Softmax( alpha Q K^_Q^T || alpha Q K_FP^T ) (V^_Q || V_FP),  alpha = 1/sqrt(d)

where K_FP / V_FP are the vertical-line keys and the window (kept in BF16)
and K^_Q / V^_Q the rest, quantised tile by tile with symmetric scales
``s = max|x| / c_B`` (c_B = 127 for INT8, 448 for FP8 e4m3; Algorithm 2,
stage 2), and the queries with a per-query-block scale ``s^Q``.

Readings (the paper leaves these open):

* the window is the last W keys of the sequence (Algorithm 2, "last W
  keys"); vertical-line positions come from ``[0, L - W)``;
* the causal mask ``j <= i`` applies in every segment (a query block in the
  middle of the sequence must not see later keys);
* key tiles are B_N = 64 consecutive entries of the quantised-prefix
  positions taken in ascending order (the reordered layout of Algorithm 2,
  stage 1); the last tile may be short;
* K and V each use one scale per tile (Algorithm 2, stage 2 states the rule
  ``s_T = max|K_T| / c_B`` for K; Eq. 7 quantises V_Q as well and names no
  other rule, so V takes the same one); Q uses one scale per block of 128
  query rows of one head (``s^Q``, Algorithm 2 line 13);
* the stored scale is a float32 number, ``s = RN_fp32(max|x| / c_B)`` (the
  paper fixes no precision; one rounding of the exact quotient); the code of
  x is the grid value nearest to the exact quotient ``x / s``, ties to the
  even code: INT8 the integers -127..127, FP8 the e4m3 values (bias 7,
  three fraction bits, subnormals below 2^-6, largest 448; values beyond it
  take +-448), FP4 the e2m1 values 0, 0.5, 1, 1.5, 2, 3, 4, 6 and their
  negatives (c_B = 6: the paper names INT4/FP4 backends for the low-bit
  segment without further detail, and the same per-tile symmetric rule with
  the format's largest value is the plain reading).  A block of zeros gets
  ``s = 0`` and zero codes;
* ``band=True`` takes the window per query instead (a diagonal band): query
  ``i`` sees the keys ``(i - W, i]`` in BF16, the vertical lines at or
  before ``i - W`` in BF16 and the other keys at or before ``i - W`` from
  the quantised prefix; vertical lines, the quantised-prefix list, its
  tiles and its scales are those of the fixed window (for every row
  ``i - W <= L - 1 - W < P``, so no quantised key outside ``[0, P)`` is
  ever needed).  The two readings agree on the last row and whenever W = 0;
* the softmax probabilities are *not* quantised here.  A kernel that feeds a
  low-precision P to the PV product differs from this oracle by the P
  rounding step only; that difference is covered by the test tolerance
  (parity unpinned for that step).
"""
from __future__ import annotations

import math

import numpy as np
import torch

C_B = {"int8": 127.0, "fp8": 448.0, "fp4": 6.0}
KEY_TILE = 64
QUERY_BLOCK = 128


def e4m3_values() -> np.ndarray:
    """The non-negative finite e4m3 values, ascending, built from the format:
    exponent bias 7, three fraction bits, subnormals m 2^-9 (exponent field
    0), normals (1 + m/8) 2^(e-7); exponent field 15 with fraction 7 is NaN
    and there are no infinities, so the largest value is 448.  The index of
    a value is its 7-bit code, so an even index is an even code."""
    vals = [m * 2.0 ** -9 if e == 0 else (1 + m / 8) * 2.0 ** (e - 7)
            for e in range(16) for m in range(8) if not (e == 15 and m == 7)]
    return np.array(vals, dtype=np.float64)


def e2m1_values() -> np.ndarray:
    """The non-negative e2m1 (FP4) values, ascending, from the format:
    exponent bias 1, one fraction bit, subnormal m 2^-1 (exponent field 0),
    normals (1 + m/2) 2^(e-1); no infinities or NaN, so the largest is 6.
    The index of a value is its 3-bit code (even index = even code)."""
    vals = [m * 0.5 if e == 0 else (1 + m / 2) * 2.0 ** (e - 1) for e in range(4) for m in range(2)]
    return np.array(vals, dtype=np.float64)


_GRIDS = {"int8": np.arange(128, dtype=np.float64), "fp8": e4m3_values(), "fp4": e2m1_values()}


def nearest_grid_index(a, s, grid) -> np.ndarray:
    """Index into the ascending non-negative ``grid`` of the value nearest to
    the exact quotient a / s (a >= 0, s > 0), ties to the even index, values
    past the top taking the top.  A float64 quotient gives a candidate; it
    is moved across the midpoints (grid[i] + grid[i+1]) / 2, whose products
    with s are exact in float64 (at most 9 + 24 significant bits), by the
    exact sign of a minus that product."""
    mids = (grid[:-1] + grid[1:]) / 2
    n = len(mids)
    with np.errstate(divide="ignore", invalid="ignore"):
        i = np.searchsorted(mids, a / s)
    for _ in range(2):
        d = a - mids[np.minimum(i, n - 1)] * s
        i = np.where((i < n) & ((d > 0) | ((d == 0) & (i % 2 == 1))), i + 1, i)
        d = a - mids[np.maximum(i - 1, 0)] * s
        i = np.where((i > 0) & ((d < 0) | ((d == 0) & (i % 2 == 1))), i - 1, i)
    return i


def _codes(x: np.ndarray, s, dtype: str) -> np.ndarray:
    """Low-bit codes (as float64 code values) of the exact quotients x / s."""
    if dtype not in _GRIDS:
        raise ValueError(dtype)
    x = np.asarray(x, dtype=np.float64)
    s = np.broadcast_to(np.asarray(s, dtype=np.float64), x.shape)
    live = s > 0
    grid = _GRIDS[dtype]
    i = nearest_grid_index(np.abs(x), np.where(live, s, 1.0), grid)
    return np.where(live, np.sign(x) * grid[i], 0.0)


def quantize_symmetric(x, axis, dtype: str):
    """Symmetric quantisation with ``s = fl32(max|x| / c_B)`` over ``axis``
    (``None`` = one scale for the whole block).  ``x`` holds BF16 values, so
    ``max|x|`` and ``x`` are exact in float32.
    Returns (dequantised values, codes, scales), all float64."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max(axis=axis, keepdims=True).astype(np.float32)
    s = (amax / np.float32(C_B[dtype])).astype(np.float32)
    c = _codes(x, s, dtype)
    s64 = s.astype(np.float64)
    return c * s64, c, s64


def hybrid_prefill(q, k, v, vl_idx, window: int, dtype: str = "int8",
                   key_tile: int = KEY_TILE, query_block: int = QUERY_BLOCK,
                   query_blocks=None, heads=None, return_abs: bool = False, band: bool = False):
    """Eq. 7 with Algorithm 2's quantisation, causal, float64.

    q [B, HQ, L, d]; k, v [B, HKV, L, d]; vl_idx [B, HKV, k] (positions in
    [0, L - W), or None).  Returns o [B, HQ, L, d] float64.
    ``query_blocks`` / ``heads`` (optional lists) restrict which 128-row query
    blocks and query heads are computed (the others stay zero); each block's
    result does not depend on the others.
    With ``return_abs`` the function also returns ``a = sum_j p_j |v_j| /
    sum_j p_j`` (the same softmax weights applied to the magnitudes of the
    effective values): ``2^-8 a`` bounds what rounding the probabilities to
    BF16 (unit roundoff 2^-8) before the P.V product can change in ``o``.
    ``band`` selects the per-query window (module docstring).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, HQ, L, d = q.shape
    HKV = k.shape[1]
    g = HQ // HKV
    alpha = 1.0 / math.sqrt(d)
    P = max(0, L - window)
    out = np.zeros(q.shape)  # zero pages are mapped on first write
    mag = np.zeros(q.shape)
    for b in range(B):
        for kh in range(HKV):
            if heads is not None and not any(h in heads for h in range(kh * g, (kh + 1) * g)):
                continue  # no requested query head reads this KV head
            vl = (np.zeros(0, np.int64) if vl_idx is None
                  else np.asarray(vl_idx[b, kh], np.int64))
            qpos = np.setdiff1d(np.arange(P), vl)
            # Effective key/value rows for the quantised prefix, tile by tile.
            kq = np.zeros((len(qpos), d))
            vq = np.zeros((len(qpos), d))
            for t0 in range(0, len(qpos), key_tile):
                j = qpos[t0:t0 + key_tile]
                kq[t0:t0 + len(j)] = quantize_symmetric(k[b, kh, j], None, dtype)[0]
                vq[t0:t0 + len(j)] = quantize_symmetric(v[b, kh, j], None, dtype)[0]
            # Full-precision list: the vertical lines, then (fixed window) the
            # last W positions; a band's keys are taken per query block below.
            fp = vl if band else np.concatenate([vl, np.arange(P, L)])
            pos = np.concatenate([qpos, fp])
            Kall = np.concatenate([kq, k[b, kh, fp]])
            Vall = np.concatenate([vq, v[b, kh, fp]])
            nq = len(qpos)
            for h in range(kh * g, (kh + 1) * g):
                if heads is not None and h not in heads:
                    continue
                for r0 in range(0, L, query_block):
                    if query_blocks is not None and r0 // query_block not in query_blocks:
                        continue
                    rows = np.arange(r0, min(L, r0 + query_block))
                    qb = q[b, h, rows]
                    qhat = quantize_symmetric(qb, None, dtype)[0]
                    # Quantised segment uses the quantised queries, the
                    # full-precision segments the BF16 queries (Algorithm 2).
                    lg = np.concatenate([alpha * qhat @ Kall[:nq].T,
                                         alpha * qb @ Kall[nq:].T], axis=1)
                    Vx = Vall
                    if band:
                        # quantised prefix and vertical lines: j <= i - W;
                        # the band (i - W, i] in BF16 from the source rows
                        lim = rows - window
                        lg = np.where(pos[None, :] <= lim[:, None], lg, -np.inf)
                        bpos = np.arange(max(0, r0 - window + 1), rows[-1] + 1)
                        inb = (bpos[None, :] > lim[:, None]) & (bpos[None, :] <= rows[:, None])
                        lgb = np.where(inb, alpha * qb @ k[b, kh, bpos].T, -np.inf)
                        lg = np.concatenate([lg, lgb], axis=1)
                        Vx = np.concatenate([Vall, v[b, kh, bpos]])
                    else:
                        lg = np.where(pos[None, :] <= rows[:, None], lg, -np.inf)
                    m = lg.max(axis=1, keepdims=True)
                    e = np.exp(lg - m)
                    out[b, h, rows] = (e @ Vx) / e.sum(axis=1, keepdims=True)
                    if return_abs:
                        mag[b, h, rows] = (e @ np.abs(Vx)) / e.sum(axis=1, keepdims=True)
    return (out, mag) if return_abs else out


def causal_attention(q, k, v) -> np.ndarray:
    """Exact causal softmax attention in float64 (the full-precision reference)."""
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k, dtype=np.float64)
    v = np.asarray(v, dtype=np.float64)
    B, HQ, L, d = q.shape
    g = HQ // k.shape[1]
    alpha = 1.0 / math.sqrt(d)
    out = np.zeros_like(q)
    mask = np.tril(np.ones((L, L), dtype=bool))
    for b in range(B):
        for h in range(HQ):
            lg = alpha * q[b, h] @ k[b, h // g].T
            lg = np.where(mask, lg, -np.inf)
            e = np.exp(lg - lg.max(axis=1, keepdims=True))
            out[b, h] = (e @ v[b, h // g]) / e.sum(axis=1, keepdims=True)
    return out
