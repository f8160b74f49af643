"""Byte accounting of the hybrid cache.

*HyQuant: Hybrid-Precision Quantization for LLM Attention*, §5.5 and
Appendix B.7, Table 14 (memory overhead against strict K4V4 for a
Qwen3-8B-sized layer, W = 128, rho = 5%) and the proxy-query buffer size of
§5.5 (64 x H_Q x d x 2 bytes).

Per KV head and token, for one of K or V:
  * a 4-bit row holds d/2 bytes of codes plus, per group of G, an FP16 scale
    and an FP16 zero (4 bytes): 80 bytes at d = 128, G = 32 (64 bytes when
    the metadata is left out, as Table 14's vertical-line row does);
  * a BF16 row holds 2d bytes (256 bytes at d = 128).
"""
from __future__ import annotations


def int4_row_bytes(d: int = 128, group: int = 32, with_meta: bool = True) -> int:
    return d // 2 + ((d // group) * 4 if with_meta else 0)


def bf16_row_bytes(d: int = 128) -> int:
    return 2 * d


def vl_overhead(rho: float, d: int = 128) -> float:
    """Extra non-window bytes when a fraction rho of positions is BF16
    instead of 4-bit (codes only), relative to all-4-bit."""
    q = int4_row_bytes(d, with_meta=False)
    return ((1.0 - rho) * q + rho * bf16_row_bytes(d)) / q - 1.0


def window_overhead(prefix: int, window: int = 128, d: int = 128, group: int = 32) -> float:
    """BF16 window bytes relative to a ``prefix``-token 4-bit cache with metadata."""
    return window * bf16_row_bytes(d) / (prefix * int4_row_bytes(d, group))


def proxy_buffer_bytes(num_q_heads: int, d: int = 128, n_proxy: int = 64) -> int:
    """Proxy-query buffer: n_proxy x H_Q x d half-precision values (§5.5)."""
    return n_proxy * num_q_heads * d * 2


def decode_bytes(B: int, HQ: int, HKV: int, d: int, n_q: int, n_vl: int,
                 n_tail: int, group: int = 32) -> int:
    """Algorithmic bytes one decode-attention call must move: every 4-bit row
    (K and V, codes + metadata), every BF16 row (vertical-line and tail, K and
    V), the query and the output."""
    return B * (HKV * (n_q * 2 * int4_row_bytes(d, group)
                       + (n_vl + n_tail) * 2 * bf16_row_bytes(d))
                + 2 * HQ * d * 2)
