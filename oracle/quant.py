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
* the code decision is taken in float32 (the kernel's precision):
  ``r = fl32(1 / s)``, ``c = clamp(rint(fl32(fl32(x - z) * r)), 0, qmax)``
  with round-half-to-even; a group with ``s == 0`` gets all-zero codes;
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
    # Code decision in float32, one IEEE operation at a time.
    s32 = scale.astype(np.float32)[..., None]
    z32 = zero.astype(np.float32)[..., None]
    x32 = xg.astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore"):
        r32 = np.float32(1.0) / s32
        t = (x32 - z32) * r32
        c = np.clip(np.rint(t), 0, qmax)
    c = np.where(s32 == 0, 0, c)
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
