"""Error and coverage measures used by the paper's motivation and ablations.

* Attention-output MSE against full-precision attention (the input to
  o_proj): *HyQuant: Hybrid-Precision Quantization for LLM Attention*, §2.2
  (Fig. 2: uniform 4-bit vs uniform 8-bit vs 4-bit with the top 1% / 5%
  kept in full precision), Appendix B.5 (Fig. 6: uniform / window-only /
  vertical-line-only / both) and Appendix B.2 (Table 10: MSE falls as the
  window grows).
* Attention-mass coverage: §2.1, Table 1 -- the fraction of softmax(QK^T)
  mass that falls on the top-5% key positions together with a W = 128 local
  window.
"""
from __future__ import annotations

import math

import numpy as np

from .attention import hybrid_decode
from .select import prefix_len, select_vertical, vl_count


def mse(a, b) -> float:
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    return float(np.mean((a - b) ** 2))


def exact_decode(q, k_src, v_src, L: int) -> np.ndarray:
    """Full-precision decode attention over the BF16 cache (no quantisation)."""
    return hybrid_decode(q, k_src, v_src, L, 0, None)


def strategy_outputs(q, q_proxy, k_src, v_src, L: int, window: int, rho_ppm: int):
    """Decode outputs for the partitions compared in Fig. 2 and Fig. 6.

    Returns a dict name -> o [B, HQ, d]:
      exact    : BF16 cache, no quantisation
      int8     : every position 8-bit (same quantiser, 255 levels)
      int4     : every position 4-bit
      window   : last ``window`` positions BF16, rest 4-bit
      vl       : top-rho positions of the whole context BF16, rest 4-bit
      hybrid   : top-rho of the non-window prefix + window BF16, rest 4-bit
    """
    out = {"exact": exact_decode(q, k_src, v_src, L)}
    out["int8"] = hybrid_decode(q, k_src, v_src, L, L, None, bits=8)
    out["int4"] = hybrid_decode(q, k_src, v_src, L, L, None, bits=4)
    P = prefix_len(L, window)
    out["window"] = hybrid_decode(q, k_src, v_src, L, P, None, bits=4)
    idx_all, _ = select_vertical(q_proxy, k_src, L, 0, rho_ppm)
    out["vl"] = hybrid_decode(q, k_src, v_src, L, L, idx_all, bits=4)
    idx, _ = select_vertical(q_proxy, k_src, L, window, rho_ppm)
    out["hybrid"] = hybrid_decode(q, k_src, v_src, L, P, idx, bits=4)
    return out


def coverage(q, k_src, L: int, window: int, rho_ppm: int) -> float:
    """Mean attention mass on (global top-rho positions by column mass) U
    (last ``window`` positions), per query, as in Table 1.

    q [B, HQ, T, d] queries; k_src [B, HKV, L, d].  The column mass is the
    softmax probability summed over the T queries and the g heads of each
    KV head (Eq. 4).
    """
    q = np.asarray(q, dtype=np.float64)
    k = np.asarray(k_src, dtype=np.float64)[:, :, :L]
    B, HQ, T, d = q.shape
    HKV = k.shape[1]
    g = HQ // HKV
    alpha = 1.0 / math.sqrt(d)
    covs = []
    for b in range(B):
        for kh in range(HKV):
            qq = q[b, kh * g:(kh + 1) * g].reshape(g * T, d)
            lg = alpha * qq @ k[b, kh].T
            p = np.exp(lg - lg.max(axis=1, keepdims=True))
            p /= p.sum(axis=1, keepdims=True)
            col = p.sum(axis=0)
            n_top = vl_count(L, rho_ppm)
            top = np.argsort(-col, kind="stable")[:n_top]
            keep = np.zeros(L, dtype=bool)
            keep[top] = True
            keep[max(0, L - window):] = True
            covs.append(p[:, keep].sum(axis=1).mean())
    return float(np.mean(covs))
