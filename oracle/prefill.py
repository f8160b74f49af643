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
* scales and codes are decided in float32, the kernel's precision (the
  paper fixes none): ``s = fl32(max|x| / c_B)`` and ``t = fl32(x / s)``;
  INT8 codes are ``clamp(rint(t), -127, 127)`` (ties to even), FP8 codes the
  e4m3 value nearest to ``t`` (ties to even, saturating at +-448); a block
  of zeros gets ``s = 0`` and zero codes;
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

C_B = {"int8": 127.0, "fp8": 448.0}
KEY_TILE = 64
QUERY_BLOCK = 128


def _codes(x: np.ndarray, s, dtype: str) -> np.ndarray:
    """Low-bit codes of ``fl32(x / s)`` (float32 in, float64 code values out)."""
    x = np.asarray(x, dtype=np.float32)
    s = np.asarray(s, dtype=np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        t = np.where(s > 0, x / np.where(s > 0, s, np.float32(1.0)), np.float32(0.0)).astype(np.float32)
    if dtype == "int8":
        return np.clip(np.rint(t), -127, 127).astype(np.float64)
    if dtype == "fp8":
        t = np.clip(t, np.float32(-448.0), np.float32(448.0))
        return torch.from_numpy(t).to(torch.float8_e4m3fn).to(torch.float64).numpy()
    raise ValueError(dtype)


def quantize_symmetric(x, axis, dtype: str):
    """Symmetric quantisation with ``s = fl32(max|x| / c_B)`` over ``axis``
    (``None`` = one scale for the whole block).  ``x`` holds BF16 values, so
    ``max|x|`` and ``x`` are exact in float32.
    Returns (dequantised values, codes, scales), all float64."""
    x = np.asarray(x, dtype=np.float64)
    amax = np.abs(x).max(axis=axis, keepdims=True).astype(np.float32)
    s = (amax / np.float32(C_B[dtype])).astype(np.float32)
    c = _codes(x.astype(np.float32), s, dtype)
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
