"""Hybrid-precision decode attention.

Follows *HyQuant: Hybrid-Precision Quantization for LLM Attention*:

* §4.1 Eq. 1-3: the key positions of each (layer, KV head) split into three
  disjoint sets -- vertical-line positions K_VL chosen from the non-window
  prefix, the window K_Win, and the rest K_Q;
* §4.3 Eq. 8: the cache keeps K_VL and the window in full precision and the
  rest in low bits;
* §4.3 Eq. 9: low-bit blocks are dequantised and used directly in the
  attention sum;
* Appendix A.3, Algorithm 3: the same result computed as a split online
  softmax (FlashOS per split, ReduceSoftmax, then the full-precision
  segments), with ``alpha = 1 / sqrt(d)``.

The decode result for query head h (KV head ``h // g``) is the plain softmax
attention over every position j < L of the *effective* cache
``k~_j, v~_j`` (dequantised for j in K_Q, the BF16 row otherwise):

    o_h = sum_j exp(alpha q_h.k~_j - M) v~_j / sum_j exp(alpha q_h.k~_j - M).

Reading of the window for decode: the full-precision tail is every position
``[P, L)`` where ``P`` is the prefix length at the last re-selection (the last
W positions then, plus the up to 63 tokens appended since); the window and the
staging buffer of Algorithm 3 are one BF16 segment (segment order does not
change the softmax).
"""
from __future__ import annotations

import math

import numpy as np

from .quant import fake_quant


def textbook_attention(q, K, V, alpha: float) -> np.ndarray:
    """Softmax attention, two passes, float64.  q [n, d], K/V [L, d] -> [n, d]."""
    q = np.asarray(q, dtype=np.float64)
    K = np.asarray(K, dtype=np.float64)
    V = np.asarray(V, dtype=np.float64)
    logits = alpha * (q @ K.T)
    m = logits.max(axis=-1, keepdims=True)
    e = np.exp(logits - m)
    return (e @ V) / e.sum(axis=-1, keepdims=True)


def effective_cache(k_src, v_src, L: int, P: int, idx, bits: int = 4, bits_v: int | None = None):
    """Effective (K~, V~) of Eq. 8 for every (b, kvh): float64 [B, HKV, L, d].

    Positions in [0, P) not in ``idx[b, kvh]`` are replaced by
    DeQuant(Quant(.)) with B_K = ``bits`` for keys and B_V = ``bits_v``
    (default: ``bits``) for values (Algorithm 4 quantises K and V with their
    own bit-widths); ``idx`` (vertical-line positions) and [P, L) stay as
    given.  ``idx`` may be None (no vertical-line set).
    """
    K = np.array(np.asarray(k_src, dtype=np.float64)[:, :, :L, :])
    V = np.array(np.asarray(v_src, dtype=np.float64)[:, :, :L, :])
    B, HKV = K.shape[:2]
    if P <= 0:
        return K, V
    keep = np.zeros((B, HKV, P), dtype=bool)
    if idx is not None:
        idx = np.asarray(idx, dtype=np.int64)
        for b in range(B):
            for h in range(HKV):
                keep[b, h, idx[b, h]] = True
    Kq = fake_quant(K[:, :, :P, :], bits)
    Vq = fake_quant(V[:, :, :P, :], bits if bits_v is None else bits_v)
    K[:, :, :P, :] = np.where(keep[..., None], K[:, :, :P, :], Kq)
    V[:, :, :P, :] = np.where(keep[..., None], V[:, :, :P, :], Vq)
    return K, V


def hybrid_decode(q, k_src, v_src, L: int, P: int, idx, bits: int = 4,
                  alpha: float | None = None, bits_v: int | None = None) -> np.ndarray:
    """Hybrid decode output o [B, HQ, d] in float64 (plain definition);
    ``bits`` / ``bits_v`` are B_K / B_V (``bits_v`` defaults to ``bits``)."""
    q = np.asarray(q, dtype=np.float64)
    B, HQ, d = q.shape
    HKV = np.asarray(k_src).shape[1]
    g = HQ // HKV
    a = 1.0 / math.sqrt(d) if alpha is None else alpha
    K, V = effective_cache(k_src, v_src, L, P, idx, bits, bits_v)
    out = np.zeros((B, HQ, d))
    for b in range(B):
        for kh in range(HKV):
            hs = slice(kh * g, (kh + 1) * g)
            out[b, hs] = textbook_attention(q[b, hs], K[b, kh], V[b, kh], a)
    return out


# --- Algorithm 3 as written: split online softmax --------------------------

def flash_os(state, logits, values):
    """One online-softmax update (the FlashOS step of Algorithms 2 and 3).

    state = (m [n], l [n], acc [n, d]); logits [n, T]; values [T, d].
    m is the running max of the logits, l the running sum of exp(logit - m),
    acc the running sum of exp(logit - m) * v.
    """
    m, l, acc = state
    if logits.shape[-1] == 0:
        return m, l, acc
    m_new = np.maximum(m, logits.max(axis=-1))
    corr = np.exp(m - m_new)
    p = np.exp(logits - m_new[:, None])
    return m_new, l * corr + p.sum(axis=-1), acc * corr[:, None] + p @ values


def reduce_softmax(states):
    """Merge split partials (m_s, l_s, acc_s) by log-sum-exp rescaling."""
    ms = np.stack([s[0] for s in states])
    m = ms.max(axis=0)
    l = sum(s[1] * np.exp(s[0] - m) for s in states)
    acc = sum(s[2] * np.exp(s[0] - m)[:, None] for s in states)
    return m, l, acc


def decode_alg3(q, k_src, v_src, L: int, P: int, idx, splits: int = 4,
                tile: int = 64, bits: int = 4, bits_v: int | None = None) -> np.ndarray:
    """Algorithm 3: quantised prefix in ``splits`` chunks (each its own
    FlashOS from (-inf, 0, 0)), ReduceSoftmax, then the vertical-line and the
    full-precision tail segments tile by tile; o = acc / l."""
    q = np.asarray(q, dtype=np.float64)
    B, HQ, d = q.shape
    HKV = np.asarray(k_src).shape[1]
    g = HQ // HKV
    alpha = 1.0 / math.sqrt(d)
    K, V = effective_cache(k_src, v_src, L, P, idx, bits, bits_v)
    out = np.zeros((B, HQ, d))
    for b in range(B):
        for kh in range(HKV):
            qt = q[b, kh * g:(kh + 1) * g]                  # g x d packed GQA tile
            vl = np.zeros(0, dtype=np.int64) if idx is None else np.asarray(idx[b, kh], np.int64)
            qpos = np.setdiff1d(np.arange(max(P, 0)), vl)
            empty = (np.full(g, -np.inf), np.zeros(g), np.zeros((g, d)))
            parts = []
            for chunk in np.array_split(qpos, splits):
                st = empty
                for t0 in range(0, len(chunk), tile):
                    j = chunk[t0:t0 + tile]
                    st = flash_os(st, alpha * qt @ K[b, kh, j].T, V[b, kh, j])
                parts.append(st)
            st = reduce_softmax(parts) if len(qpos) else empty
            for seg in (vl, np.arange(max(P, 0), L)):
                for t0 in range(0, len(seg), tile):
                    j = seg[t0:t0 + tile]
                    st = flash_os(st, alpha * qt @ K[b, kh, j].T, V[b, kh, j])
            out[b, kh * g:(kh + 1) * g] = st[2] / st[1][:, None]
    return out
