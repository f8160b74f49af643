"""Vertical-line token identification (VTI).

Follows *HyQuant: Hybrid-Precision Quantization for LLM Attention*,
§4.1 Eq. 1-5 and Appendix A.1, Algorithm 1:

* ``P = max(0, L_K - W)``: the local window is excluded; an empty prefix
  selects nothing;
* the proxy queries are summed (Algorithm 1 averages the tail queries; a sum
  and a mean rank keys identically) and, for GQA, the g query heads that
  share a KV head are summed too, so the score is computed once per KV head
  without repeating K (the einsum form of Algorithm 1);
* ``S(j) = u . k_j`` for j in the prefix -- raw dot products, no softmax and
  no 1/sqrt(d) (Algorithm 1 takes TopK of ``Q_bar K_pre^T`` directly);
* ``k = min(P, max(1, ceil(P * rho)))`` (Algorithm 1); with ``rho = 0`` the
  set is empty (the pure low-bit special case);
* TopK is taken with ties broken toward the lower position, and the set is
  returned sorted ascending.

``rho`` is carried as an integer number of parts per million so that
``ceil(P * rho)`` is exact (5% = 50000 ppm).

Readings: one set per KV head (the cache of Algorithm 4 is laid out per KV
head, so a position can only leave the low-bit stream for the whole head);
the proxy set is the most recent (at most 64) queries, per §5.5.
"""
from __future__ import annotations

import numpy as np


def prefix_len(L: int, window: int) -> int:
    """``P = max(0, L - W)`` (Algorithm 1, first step)."""
    return max(0, int(L) - int(window))


def vl_count(P: int, rho_ppm: int) -> int:
    """``k = min(P, max(1, ceil(P * rho)))``; 0 for an empty prefix or rho = 0."""
    if P <= 0 or rho_ppm <= 0:
        return 0
    k = -((-P * int(rho_ppm)) // 1_000_000)   # exact integer ceil
    return min(P, max(1, k))


def proxy_sum(q_proxy, num_kv_heads: int) -> np.ndarray:
    """Sum of proxy queries over time and over the query heads of each KV head.

    q_proxy : [B, HQ, T, d]  ->  u : [B, HKV, d] (float64)
    """
    q = np.asarray(q_proxy, dtype=np.float64)
    B, HQ, T, d = q.shape
    g = HQ // num_kv_heads
    return q.reshape(B, num_kv_heads, g, T, d).sum(axis=(2, 3))


def scores(u, k_src, P: int) -> np.ndarray:
    """``S(j) = u . k_j`` for j in [0, P).  u [B,HKV,d], k_src [B,HKV,>=P,d]."""
    k = np.asarray(k_src, dtype=np.float64)[:, :, :P, :]
    return np.einsum("bhd,bhpd->bhp", np.asarray(u, dtype=np.float64), k)


def topk_ascending(S, k: int) -> np.ndarray:
    """Indices of the k largest scores per row, ties to the lower index,
    returned sorted ascending.  S [..., P] -> int64 [..., k]."""
    S = np.asarray(S)
    lead = S.shape[:-1]
    P = S.shape[-1]
    if k == 0 or P == 0:
        return np.zeros(lead + (0,), dtype=np.int64)
    flat = S.reshape(-1, P)
    out = np.zeros((flat.shape[0], k), dtype=np.int64)
    pos = np.arange(P)
    for r in range(flat.shape[0]):
        order = np.lexsort((pos, -flat[r]))   # primary: score desc, then index asc
        out[r] = np.sort(order[:k])
    return out.reshape(lead + (k,))


def select_vertical(q_proxy, k_src, L: int, window: int, rho_ppm: int):
    """Algorithm 1 end to end.  Returns (idx [B, HKV, k] ascending, S [B,HKV,P])."""
    HKV = np.asarray(k_src).shape[1]
    P = prefix_len(L, window)
    k = vl_count(P, rho_ppm)
    u = proxy_sum(q_proxy, HKV)
    S = scores(u, k_src, P)
    return topk_ascending(S, k), S


# --- Algorithm 1 per query head, kept per KV head ---------------------------
#
# Algorithm 1's output is one set per query head (B x H_Q x k): query head h
# scores the prefix with its own proxy sum against the keys of its KV head.
# The cache keeps a position in BF16 for a whole KV head (Algorithm 4 gathers
# the rows from the H_KV-head K), so the list stored per KV head is the union
# of the g query heads' sets.  Reading: to keep one list length per layer the
# union is filled up to min(P, g k) positions with the highest group scores
# (the per-KV-head score above) among the positions not yet in it, ties to the
# lower position; every query head's own set is then held in BF16.

def vl_count_heads(P: int, rho_ppm: int, g: int) -> int:
    """Length of the per-KV-head list in the per-query-head reading: min(P, g k)."""
    return min(max(0, P), g * vl_count(P, rho_ppm))


def head_scores(q_proxy, k_src, P: int) -> np.ndarray:
    """``S_h(j) = (sum_t q_{h,t}) . k_j`` per query head h, with k_j the key
    of h's KV head.  q_proxy [B, HQ, T, d], k_src [B, HKV, >=P, d] ->
    [B, HQ, P] float64."""
    q = np.asarray(q_proxy, dtype=np.float64)
    k = np.asarray(k_src, dtype=np.float64)[:, :, :P, :]
    B, HQ, T, d = q.shape
    HKV = k.shape[1]
    g = HQ // HKV
    u = q.sum(axis=2).reshape(B, HKV, g, d)                 # query head kh g + r of KV head kh
    return np.einsum("bhrd,bhpd->bhrp", u, k).reshape(B, HQ, P)


def union_fill(sets, S_group, ku: int) -> np.ndarray:
    """The ascending union of `sets` (rows of positions), completed to ku
    positions by the largest S_group among the others, ties to the lower
    position."""
    U = sorted({int(j) for row in sets for j in np.asarray(row).ravel()})
    P = len(S_group)
    chosen = np.zeros(P, dtype=bool)
    chosen[U] = True
    rest = np.flatnonzero(~chosen)
    need = ku - len(U)
    if need > 0:
        order = np.lexsort((rest, -np.asarray(S_group, dtype=np.float64)[rest]))
        chosen[rest[order[:need]]] = True
    return np.flatnonzero(chosen).astype(np.int64)


def select_vertical_heads(q_proxy, k_src, L: int, window: int, rho_ppm: int):
    """Algorithm 1 per query head.  Returns (idx_heads [B, HQ, k] ascending,
    idx_kv [B, HKV, ku] ascending, union sizes [B, HKV], S_heads [B, HQ, P],
    S_group [B, HKV, P])."""
    q = np.asarray(q_proxy, dtype=np.float64)
    B, HQ = q.shape[:2]
    HKV = np.asarray(k_src).shape[1]
    g = HQ // HKV
    P = prefix_len(L, window)
    k = vl_count(P, rho_ppm)
    ku = vl_count_heads(P, rho_ppm, g)
    S_heads = head_scores(q, k_src, P)
    idx_heads = topk_ascending(S_heads, k)
    S_group = scores(proxy_sum(q, HKV), k_src, P)
    idx_kv = np.zeros((B, HKV, ku), dtype=np.int64)
    usize = np.zeros((B, HKV), dtype=np.int64)
    for b in range(B):
        for kh in range(HKV):
            own = idx_heads[b, kh * g:(kh + 1) * g]
            usize[b, kh] = len(set(own.ravel().tolist()))
            idx_kv[b, kh] = union_fill(own, S_group[b, kh], ku)
    return idx_heads, idx_kv, usize, S_heads, S_group


# --- Eq. 4: the softmax-mass score (an alternative to Algorithm 1's) -------
#
# Eq. 4 defines the vertical-line score as the accumulated column mass
# S(j) = sum_{t in T} a_{t,j}, with a_{t,j} the attention probability of
# query t on key j.  Readings: T is the proxy buffer (the last <= 64 queries)
# and, for GQA, every query head of the KV group (as for Algorithm 1's
# score); a_{t,j} is the softmax over the L current keys of alpha q_t . k_j
# (alpha = 1/sqrt(d)), the keys present when the selection runs; Eq. 5 then
# takes the top-k of S over the non-window prefix [0, P).

def mass_scores(q_proxy, k_src, L: int, window: int, alpha=None) -> np.ndarray:
    """Eq. 4: ``S(j) = sum_t sum_h softmax_j(alpha q_{t,h} . k_j)`` for j in
    [0, P), the softmax over all L keys.  q_proxy [B, HQ, T, d], k_src
    [B, HKV, >=L, d] -> S [B, HKV, P] float64."""
    q = np.asarray(q_proxy, dtype=np.float64)
    k = np.asarray(k_src, dtype=np.float64)
    B, HQ, T, d = q.shape
    HKV = k.shape[1]
    g = HQ // HKV
    a = 1.0 / np.sqrt(d) if alpha is None else alpha
    P = prefix_len(L, window)
    S = np.zeros((B, HKV, P))
    if P == 0:
        return S
    for b in range(B):
        for kh in range(HKV):
            Q = q[b, kh * g:(kh + 1) * g].reshape(g * T, d)      # every (head, proxy) row
            z = a * (Q @ k[b, kh, :L].T)                          # rows x L logits
            e = np.exp(z - z.max(axis=1, keepdims=True))
            A = e / e.sum(axis=1, keepdims=True)                  # softmax over the L keys
            S[b, kh] = A[:, :P].sum(axis=0)                        # column mass on the prefix
    return S


def select_vertical_mass(q_proxy, k_src, L: int, window: int, rho_ppm: int):
    """Eq. 4-5 with the softmax-mass score.  Returns (idx [B, HKV, k]
    ascending, S [B, HKV, P])."""
    P = prefix_len(L, window)
    k = vl_count(P, rho_ppm)
    S = mass_scores(q_proxy, k_src, L, window)
    return topk_ascending(S, k), S


def mass_error_bound(q_proxy, k_src, L: int, window: int, chunks: int = 1024,
                     ex2_rel: float = 2.0 ** -21) -> np.ndarray:
    """A rigorous bound on |S32(j) - S(j)| for a float32 evaluation that
    computes, per row r and key j, z32 = q_r . k_j with exact products of the
    BF16 inputs accumulated in float32 (any order), t = fl(z32 * c) with
    c = fl(alpha log2 e), the row maximum m and the row sum l of
    ex2(t - m) (partial sums over at most ``chunks`` key ranges merged once
    with ex2 rescaling), a = ex2(t - m) / l, and S(j) = sum_r a (float32, any
    order); ex2 has relative error at most ``ex2_rel`` and flushes results
    below 2^-126 to zero.  An evaluation that forms the argument as
    fl(z32 * c - m) with one fused rounding, or a with one fused multiply-add
    into the column sum, rounds less and stays inside the same bound.

    With u = 2^-23 (one float32 ulp, covering truncating accumulators):
      dt_rj = c (1 + 2u) gamma_d sum_i |q_ri k_ji| + 2u c |z_rj|     (error of t)
      dm_r  = max_j dt_rj                                               (of m)
      eta_rj = dt_rj + dm_r + u |t_rj - m_r|                 (of t - m, log2 units)
    the computed numerator is 2^(t-m) 2^(+-eta) (1 +- ex2_rel), the row sum
    l within the a-weighted mean of those factors times (1 +- gamma_(L +
    chunks) (1 + ex2_rel)), the quotient within 2u; the column sum adds
    gamma_R sum_r a.  Elements whose numerator can flush (t - m - eta <
    -126) count with their whole weight.  Returned per (b, kvh, j < P).
    """
    q = np.asarray(q_proxy, dtype=np.float64)
    k = np.asarray(k_src, dtype=np.float64)
    B, HQ, T, d = q.shape
    HKV = k.shape[1]
    g = HQ // HKV
    R = g * T
    u = 2.0 ** -23
    alpha = 1.0 / np.sqrt(d)
    c = alpha / np.log(2.0)
    P = prefix_len(L, window)
    bound = np.zeros((B, HKV, P))
    if P == 0:
        return bound
    gl = _gamma(L + chunks) * (1 + ex2_rel) + ex2_rel
    for b in range(B):
        for kh in range(HKV):
            Q = q[b, kh * g:(kh + 1) * g].reshape(R, d)
            K = k[b, kh, :L]
            z = Q @ K.T
            t = c * z
            m = t.max(axis=1, keepdims=True)
            A = np.exp2(t - m)
            A /= A.sum(axis=1, keepdims=True)
            dt = c * (1 + 2 * u) * _gamma(d) * (np.abs(Q) @ np.abs(K).T) + 2 * u * c * np.abs(z)
            eta = dt + dt.max(axis=1, keepdims=True) + u * np.abs(t - m)
            up = np.exp2(eta) * (1 + ex2_rel)
            lo = np.exp2(-eta) * (1 - ex2_rel)
            den_hi = (A * up).sum(axis=1, keepdims=True) * (1 + gl)
            den_lo = (A * lo).sum(axis=1, keepdims=True) * (1 - gl)
            rel = np.maximum(up * (1 + 2 * u) / den_lo - 1.0, 1.0 - lo * (1 - 2 * u) / den_hi)
            rel = np.where(t - m - eta < -126.0, 1.0, rel)
            err = (A * rel)[:, :P].sum(axis=0) + _gamma(R) * (A * (1 + rel))[:, :P].sum(axis=0)
            bound[b, kh] = err
    return bound


# --- float32 error bounds used to check a float32 implementation -----------

def _gamma(n: int, unit: float = 2.0 ** -23) -> float:
    # unit = 2^-23 (one float32 ulp, not half) so that the bound also covers
    # accumulators that truncate instead of rounding to nearest.
    return n * unit / (1.0 - n * unit)


def score_error_bound(q_proxy, k_src, P: int) -> np.ndarray:
    """A rigorous bound on |S32(j) - S(j)| for any float32 evaluation order.

    The proxy sum u has n_u = T*g terms per component and the dot product d
    terms; with gamma_n = n u / (1 - n u) (u = 2^-23) the standard
    floating-point summation bounds give
        |S32 - S| <= gamma_d * sum_i |u32_i k_ji| + sum_i |k_ji| * gamma_nu * U_i
    where U_i = sum |q_i| over the summed queries, and |u32_i| <= |u_i| +
    gamma_nu U_i.  Returned per (b, kvh, j) in float64.
    """
    q = np.asarray(q_proxy, dtype=np.float64)
    k = np.abs(np.asarray(k_src, dtype=np.float64)[:, :, :P, :])
    B, HQ, T, d = q.shape
    HKV = k.shape[1]
    g = HQ // HKV
    n_u = T * g
    u = np.abs(q.reshape(B, HKV, g, T, d).sum(axis=(2, 3)))
    U = np.abs(q).reshape(B, HKV, g, T, d).sum(axis=(2, 3))
    gu = _gamma(n_u)
    u_hi = u + gu * U
    return (_gamma(d) * np.einsum("bhd,bhpd->bhp", u_hi, k)
            + gu * np.einsum("bhd,bhpd->bhp", U, k))


def check_selection(S, bound, k: int, got) -> dict:
    """Is ``got`` a valid top-k of scores known only to within ``bound``?

    Keys whose whole interval [S-b, S+b] lies above the (k+1)-th largest
    upper end must be selected; keys whose interval lies below the k-th
    largest lower end must not be.  Keys in between are "ambiguous": either
    outcome is valid.  Also checks size, uniqueness, order and range.
    """
    S = np.asarray(S, dtype=np.float64)
    b = np.asarray(bound, dtype=np.float64)
    got = np.asarray(got, dtype=np.int64)
    P = S.shape[0]
    res = dict(ok=True, ambiguous=0, reason="")
    if got.shape != (k,):
        return dict(ok=False, ambiguous=0, reason=f"size {got.shape} != ({k},)")
    if k == 0:
        return res
    if np.any(np.diff(got) <= 0) or got.min() < 0 or got.max() >= P:
        return dict(ok=False, ambiguous=0, reason="not strictly ascending / out of range")
    hi = S + b
    lo = S - b
    hi_sorted = np.sort(hi)[::-1]
    lo_sorted = np.sort(lo)[::-1]
    tau_hi = hi_sorted[k] if k < P else -np.inf      # (k+1)-th largest upper end
    tau_lo = lo_sorted[k - 1]                          # k-th largest lower end
    must = lo > tau_hi
    must_not = hi < tau_lo
    sel = np.zeros(P, dtype=bool)
    sel[got] = True
    res["ambiguous"] = int(P - must.sum() - must_not.sum())
    if np.any(must & ~sel):
        res.update(ok=False, reason=f"missed {np.flatnonzero(must & ~sel)[:8].tolist()}")
    elif np.any(must_not & sel):
        res.update(ok=False, reason=f"wrongly chose {np.flatnonzero(must_not & sel)[:8].tolist()}")
    return res
