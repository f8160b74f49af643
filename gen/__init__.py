"""Seeded synthetic inputs for hybrid-precision (INT4 + BF16) attention.

This module holds random-input recipes only: no quantisation, selection or
attention arithmetic lives here.  Both the CPU oracle (``oracle/``) and the
CUDA path read the same tensors produced here, so it is the one piece of code
the two sides share.

Every generator is keyed on ``(seed, tag)`` through a fresh
``torch.Generator`` on the CPU, so a case is reproducible within one
PyTorch build.  Tensors come back as CPU ``bfloat16`` (model activations are
BF16 in the decode path of *HyQuant: Hybrid-Precision Quantization for LLM
Attention*, §4.3) plus integer metadata.

Recipes (the input shapes follow the workloads named in the paper's
experimental setup, §5.1 and Appendix B.8; the distributions are synthetic
stand-ins for model activations, since no weights or datasets are used):

* keys and values ~ N(0, 1);
* optional outlier channels: a few seed-chosen head_dim channels of K scaled
  by a constant factor;
* one unit direction ``u`` per (batch, KV head);
* planted vertical-line ("sink") keys: ``key = m * u + noise`` at positions
  drawn without replacement from the non-window prefix ``[0, L - W)``;
  ``m`` is a constant, or ``4 * |t|`` with ``t`` Student-t (nu = 3) for the
  heavy-tailed recipe;
* queries (and proxy queries) ~ N(0, 1) + ``q_gain * u`` of their KV head.
"""
from __future__ import annotations

import hashlib
from dataclasses import dataclass, field

import torch

__all__ = ["gen_for", "DecodeCase", "decode_case", "PrefillCase", "prefill_case",
           "rows_bf16"]


def gen_for(seed: int, *tags) -> torch.Generator:
    """A CPU generator seeded from a hash of ``(seed, *tags)``."""
    h = hashlib.sha256(repr((int(seed),) + tuple(tags)).encode()).digest()
    g = torch.Generator(device="cpu")
    g.manual_seed(int.from_bytes(h[:8], "little") & ((1 << 63) - 1))
    return g


def _normal(seed, tag, shape):
    return torch.randn(*shape, generator=gen_for(seed, tag), dtype=torch.float32)


def _unit_dirs(seed, B, HKV, d):
    u = _normal(seed, "u", (B, HKV, d))
    return u / u.norm(dim=-1, keepdim=True)


def rows_bf16(seed: int, shape, scale: float = 1.0, tag: str = "rows") -> torch.Tensor:
    """Plain N(0, scale^2) rows rounded to BF16."""
    return (_normal(seed, tag, shape) * scale).to(torch.bfloat16)


@dataclass
class DecodeCase:
    """One decode-attention input set (CPU tensors).

    q       bf16 [B, HQ, d]        query of the current step
    q_proxy bf16 [B, HQ, T, d]     the T most recent queries (oldest first)
    k, v    bf16 [B, HKV, L, d]    the full-precision keys / values
    sinks   int64 [B, HKV, n_sink] planted positions (sorted)
    u       f32  [B, HKV, d]       the planted unit directions
    """
    q: torch.Tensor
    q_proxy: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    sinks: torch.Tensor
    u: torch.Tensor
    meta: dict = field(default_factory=dict)


def decode_case(seed: int, B: int, HQ: int, HKV: int, L: int, d: int = 128, *,
                window: int = 128, n_proxy: int = 64, n_sinks: int | None = None,
                sink_frac: float = 0.0, sink_gain: float = 4.0,
                heavy_tail: bool = False, q_gain: float = 2.0,
                outlier_channels: int = 0, outlier_scale: float = 8.0,
                value_scale: float = 1.0) -> DecodeCase:
    """Synthetic decode inputs with planted vertical-line keys.

    ``n_sinks`` (absolute) wins over ``sink_frac`` (fraction of the
    non-window prefix).  Sinks are drawn without replacement from
    ``[0, max(0, L - window))``.
    """
    assert HQ % HKV == 0
    g = HQ // HKV
    P = max(0, L - window)
    u = _unit_dirs(seed, B, HKV, d)
    k = _normal(seed, "k", (B, HKV, L, d))
    v = _normal(seed, "v", (B, HKV, L, d)) * value_scale
    if outlier_channels > 0:
        gch = gen_for(seed, "outlier_channels")
        for b in range(B):
            for h in range(HKV):
                ch = torch.randperm(d, generator=gch)[:outlier_channels]
                k[b, h, :, ch] *= outlier_scale
    ns = n_sinks if n_sinks is not None else int(round(sink_frac * P))
    ns = max(0, min(ns, P))
    sinks = torch.zeros(B, HKV, ns, dtype=torch.int64)
    if ns > 0:
        gs = gen_for(seed, "sinks")
        for b in range(B):
            for h in range(HKV):
                pos = torch.randperm(P, generator=gs)[:ns].sort().values
                sinks[b, h] = pos
                if heavy_tail:
                    z = torch.randn(ns, generator=gs)
                    chi2 = (torch.randn(ns, 3, generator=gs) ** 2).sum(-1)
                    t = z / torch.sqrt(chi2 / 3.0)
                    m = 4.0 * t.abs()
                else:
                    m = torch.full((ns,), float(sink_gain))
                k[b, h, pos] += m[:, None] * u[b, h][None, :]
    uq = u.repeat_interleave(g, dim=1)  # [B, HQ, d]
    q = _normal(seed, "q", (B, HQ, d)) + q_gain * uq
    qp = _normal(seed, "q_proxy", (B, HQ, n_proxy, d)) + q_gain * uq[:, :, None, :]
    return DecodeCase(q=q.to(torch.bfloat16), q_proxy=qp.to(torch.bfloat16),
                      k=k.to(torch.bfloat16), v=v.to(torch.bfloat16),
                      sinks=sinks, u=u,
                      meta=dict(seed=seed, B=B, HQ=HQ, HKV=HKV, L=L, d=d,
                                window=window, n_proxy=n_proxy, n_sinks=ns))


@dataclass
class PrefillCase:
    """Causal prefill inputs: q bf16 [B, HQ, L, d]; k, v bf16 [B, HKV, L, d]."""
    q: torch.Tensor
    k: torch.Tensor
    v: torch.Tensor
    sinks: torch.Tensor
    u: torch.Tensor
    meta: dict = field(default_factory=dict)


def prefill_case(seed: int, B: int, HQ: int, HKV: int, L: int, d: int = 128, *,
                 window: int = 128, sink_frac: float = 0.02, sink_gain: float = 4.0,
                 q_gain: float = 2.0) -> PrefillCase:
    """Synthetic causal-prefill inputs with planted sink columns."""
    g = HQ // HKV
    P = max(0, L - window)
    u = _unit_dirs(seed, B, HKV, d)
    k = _normal(seed, "pk", (B, HKV, L, d))
    v = _normal(seed, "pv", (B, HKV, L, d))
    ns = max(0, min(P, int(round(sink_frac * P))))
    sinks = torch.zeros(B, HKV, ns, dtype=torch.int64)
    if ns > 0:
        gs = gen_for(seed, "psinks")
        for b in range(B):
            for h in range(HKV):
                pos = torch.randperm(P, generator=gs)[:ns].sort().values
                sinks[b, h] = pos
                k[b, h, pos] += sink_gain * u[b, h][None, :]
    uq = u.repeat_interleave(g, dim=1)
    q = _normal(seed, "pq", (B, HQ, L, d)) + q_gain * uq[:, :, None, :]
    return PrefillCase(q=q.to(torch.bfloat16), k=k.to(torch.bfloat16),
                       v=v.to(torch.bfloat16), sinks=sinks, u=u,
                       meta=dict(seed=seed, B=B, HQ=HQ, HKV=HKV, L=L, d=d,
                                 window=window, n_sinks=ns))
