"""Asymmetric low-bit group quantiser and its inverse.

Follows *HyQuant: Hybrid-Precision Quantization for LLM Attention*,
Appendix A.4, Algorithm 4 (``K^Q <- Quant_{B_K}(K[:, :, I_Q, :]; G)``, same for
V) and §4.3, Eq. 9 (``K^hat = DeQuant(K^Q)``).  The paper names the group
size G and the bit-width but fixes neither the grouping axis, the zero-point
form nor the rounding; the readings adopted here are:

* groups are G = 32 consecutive elements along head_dim, for K and for V;
* asymmetric affine form ``x ~ c * s + z`` with codes c in [0, 2^bits - 1];
* ``s`` = the smallest float16 value with ``(2^bits - 1) * s >= max - min``
  in exact arithmetic: the step of the 2^bits-level grid rounded *up* to
  float16, so that the top code still reaches the group maximum;
* ``z = RN_fp16(min)``;
* the code of x is the grid point z + c * s nearest to x, c in [0, qmax],
  with ties going to the even code (round-half-to-even of (x - z) / s,
  then clamped); a group with ``s == 0`` gets all-zero codes.  The decision
  is exact: each midpoint z + (c +- 1/2) s is a multiple of 2^-25 below
  2^25 in magnitude (s and z are float16), so it is exact in float64, and
  the sign of x - midpoint is exact in IEEE arithmetic;
* a group whose scale or zero is not a finite float16 (|x| beyond the
  float16 range, or NaN input) is an error.

Packing (two 4-bit codes per byte, low nibble = even element) and any tile
permutation are storage details of the kernel and are not modelled here:
the oracle returns one code per element.
"""
from __future__ import annotations

import numpy as np

GROUP = 32


class QuantRangeError(ValueError):
    """A group's scale or zero point does not fit a finite float16."""


def round_up_fp16(x: np.ndarray) -> np.ndarray:
    """Round float64 values toward +inf onto float16 (as float16)."""
    x = np.asarray(x, dtype=np.float64)
    h = x.astype(np.float16)                 # correctly rounded, nearest-even
    low = h.astype(np.float64) < x
    if np.any(low):
        h = h.copy()
        h[low] = np.nextafter(h[low], np.float16(np.inf))
    return h


def min_step_fp16(mx, mn, qmax: int) -> np.ndarray:
    """Smallest float16 h with qmax * h >= mx - mn, exactly (as float16).

    A float64 quotient gives a candidate that is at most one float16 step
    off; the candidate and its neighbours are then tested with the exact
    sign of qmax*h - mx + mn (a three-term float64 sum, decided with
    math.fsum where plain float64 arithmetic is not conclusive).
    """
    import math
    mx = np.asarray(mx, dtype=np.float64)
    mn = np.asarray(mn, dtype=np.float64)
    with np.errstate(over="ignore", invalid="ignore"):
        cand = round_up_fp16((mx - mn) / float(qmax))
    h = cand.astype(np.float64)
    lo = np.nextafter(cand, np.float16(-np.inf)).astype(np.float64)
    hi = np.nextafter(cand, np.float16(np.inf)).astype(np.float64)

    def covers(v):
        """Exact test qmax*v - mx + mn >= 0 (qmax*v is exact in float64)."""
        with np.errstate(over="ignore", invalid="ignore"):
            r = (qmax * v - mx) + mn
        bound = 4 * np.finfo(np.float64).eps * np.maximum.reduce(
            [np.abs(qmax * v), np.abs(mx), np.abs(mn)])
        out = r >= 0
        unsure = ~(np.abs(r) > bound) & np.isfinite(v)
        for i in zip(*np.nonzero(unsure)):
            out[i] = math.fsum([qmax * float(v[i]), -float(mx[i]), float(mn[i])]) >= 0
        return out | np.isinf(v) & (v > 0)

    res = np.where(covers(lo) & (lo >= 0), lo, np.where(covers(h), h, hi))
    return res.astype(np.float16)


def nearest_codes(x, z, s, qmax: int) -> np.ndarray:
    """Index c in [0, qmax] of the grid point z + c*s nearest to x, ties to
    the even index; 0 where s == 0.  x, z, s: float64 arrays (BF16 values,
    float16 zero and step) of one broadcast shape.

    A float64 quotient gives a candidate at most one index off; it is then
    moved across the midpoints z + (c +- 1/2) s, each exact in float64, by
    the exact sign of x minus that midpoint."""
    x, z, s = np.broadcast_arrays(np.asarray(x, np.float64), np.asarray(z, np.float64),
                                  np.asarray(s, np.float64))
    live = s > 0
    with np.errstate(divide="ignore", invalid="ignore"):
        c = np.where(live, np.clip(np.rint((x - z) / np.where(live, s, 1.0)), 0, qmax), 0.0)
    for _ in range(2):
        up = live & (c < qmax)
        d = x - (z + (c + 0.5) * s)            # exact sign: x against the midpoint above c
        c = np.where(up & ((d > 0) | ((d == 0) & (c % 2 == 1))), c + 1, c)
        dn = live & (c > 0)
        d = x - (z + (c - 0.5) * s)            # against the midpoint below c
        c = np.where(dn & ((d < 0) | ((d == 0) & (c % 2 == 1))), c - 1, c)
    return c


def quantize(x, bits: int = 4, group: int = GROUP):
    """Quantise rows of ``x`` (values exactly representable in BF16).

    Parameters
    ----------
    x : array [..., d] of float (BF16 values), d a multiple of ``group``.

    Returns
    -------
    codes : uint8 [..., d]           one code per element
    scale : float16 [..., d // group]
    zero  : float16 [..., d // group]
    """
    x = np.asarray(x, dtype=np.float64)
    d = x.shape[-1]
    if d % group:
        raise ValueError("head_dim must be a multiple of the group size")
    qmax = (1 << bits) - 1
    xg = x.reshape(x.shape[:-1] + (d // group, group))
    if np.isnan(xg).any():
        raise QuantRangeError("NaN input")
    mn = xg.min(axis=-1)
    mx = xg.max(axis=-1)
    scale = min_step_fp16(mx, mn, qmax)
    with np.errstate(over="ignore", invalid="ignore"):
        zero = mn.astype(np.float16)
    if not (np.isfinite(scale).all() and np.isfinite(zero).all()):
        raise QuantRangeError("group range exceeds the float16 metadata range")
    c = nearest_codes(xg, zero.astype(np.float64)[..., None], scale.astype(np.float64)[..., None], qmax)
    codes = c.astype(np.uint8).reshape(x.shape)
    return codes, scale, zero


def dequantize(codes, scale, zero, group: int = GROUP) -> np.ndarray:
    """``x_hat = c * s + z`` per element, in float64 (Eq. 9, DeQuant)."""
    codes = np.asarray(codes, dtype=np.float64)
    d = codes.shape[-1]
    cg = codes.reshape(codes.shape[:-1] + (d // group, group))
    s = np.asarray(scale, dtype=np.float64)[..., None]
    z = np.asarray(zero, dtype=np.float64)[..., None]
    return (cg * s + z).reshape(codes.shape)


def fake_quant(x, bits: int = 4, group: int = GROUP) -> np.ndarray:
    """``DeQuant(Quant(x))`` in float64."""
    c, s, z = quantize(x, bits, group)
    return dequantize(c, s, z, group)
