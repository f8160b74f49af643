"""Device buffers of a layer's hybrid cache and the per-step driver.

PyTorch only allocates memory and provides the stream; every step runs in
libhyq's kernels through the thin binding in ``_lib``.
"""
from __future__ import annotations

import numpy as np
import torch

from . import _lib as L
from ._lib import HyqConfig, HyqLayout


def make_config(batch, num_q_heads, num_kv_heads, capacity, window=128, period=64,
                rho_ppm=50_000, head_dim=128, group=32, bits_k=4, bits_v=4, vl_mode=0) -> HyqConfig:
    return HyqConfig(batch=batch, num_q_heads=num_q_heads, num_kv_heads=num_kv_heads,
                     head_dim=head_dim, group=group, window=window, period=period,
                     rho_ppm=rho_ppm, capacity=capacity, bits_k=bits_k, bits_v=bits_v, vl_mode=vl_mode)


class HybridLayer:
    """One layer's hybrid cache: torch-owned device buffers + the C layout view."""

    def __init__(self, cfg: HyqConfig, device="cuda"):
        self.cfg = cfg
        sizes = L.hyq_layout_sizes(cfg)
        self.buf = {n: torch.zeros(s, dtype=torch.uint8, device=device)
                    for n, s in zip(L.LAYOUT_FIELDS, sizes)}
        self.c = HyqLayout(**{n: self.buf[n].data_ptr() for n in L.LAYOUT_FIELDS})
        self.nbytes = sum(sizes)

    # typed views -----------------------------------------------------------
    def counts(self) -> torch.Tensor:
        return self.buf["counts"].view(torch.int32)[: self.cfg.batch * L.COUNTS].view(self.cfg.batch, L.COUNTS)

    def err(self) -> torch.Tensor:
        return self.buf["err"].view(torch.int32)[:1]

    def qblocks(self) -> torch.Tensor:
        c = self.cfg
        nblk = -(-c.capacity // L.QBLOCK_ROWS)
        bb = L.qblock_bytes(c.bits_k, c.bits_v)
        n = c.batch * c.num_kv_heads * nblk * bb
        return self.buf["qblocks"][:n].view(c.batch, c.num_kv_heads, nblk, bb)

    def cap_vl(self) -> int:
        c = self.cfg
        return max(1, L.hyq_vl_count(c, max(0, c.capacity - c.window)))

    def cap_tail(self) -> int:
        return self.cfg.window + self.cfg.period

    def _bf16(self, name, rows):
        c = self.cfg
        n = c.batch * c.num_kv_heads * rows * 128
        return self.buf[name].view(torch.bfloat16)[:n].view(c.batch, c.num_kv_heads, rows, 128)

    def vl_k(self):
        return self._bf16("vl_k", self.cap_vl())

    def vl_v(self):
        return self._bf16("vl_v", self.cap_vl())

    def vl_idx(self):
        c = self.cfg
        n = c.batch * c.num_kv_heads * self.cap_vl()
        return self.buf["vl_idx"].view(torch.int32)[:n].view(c.batch, c.num_kv_heads, self.cap_vl())

    def tail_k(self):
        return self._bf16("tail_k", self.cap_tail())

    def tail_v(self):
        return self._bf16("tail_v", self.cap_tail())

    def q_ring(self):
        c = self.cfg
        n = c.batch * c.num_q_heads * c.period * 128
        return self.buf["q_ring"].view(torch.bfloat16)[:n].view(c.batch, c.num_q_heads, c.period, 128)

    def reset(self, stream=None):
        L.hyq_layout_reset(self.cfg, self.c, stream)


def workspace(cfg: HyqConfig, op: int, len_hint: int = 0, device="cuda") -> torch.Tensor:
    """Zero-filled workspace for one operation."""
    n = L.hyq_workspace_size(cfg, op, len_hint)
    if n == 0:
        raise ValueError("invalid config or operation")
    return torch.zeros(n, dtype=torch.uint8, device=device)


# --- quantised stream reader/writer (documented format of include/hyq.h) ---

TILE_BYTES = 2560   # B_K = B_V = 4


def _tile_maps8():
    """(row, element) of every byte of a 2048-byte 8-bit code region, for the K
    and the V orders, indexed by byte offset."""
    krow = np.zeros(2048, np.int64)
    kel = np.zeros(2048, np.int64)
    vrow = np.zeros(2048, np.int64)
    vel = np.zeros(2048, np.int64)
    for u in range(16):
        for lane in range(32):
            g, t = lane // 4, lane % 4
            base = 512 * (u // 4) + 16 * lane + 4 * (u % 4)
            for j in range(4):
                krow[base + j] = g + 8 * (u % 2)
                kel[base + j] = 16 * (u // 2) + 4 * t + (0, 2, 1, 3)[j]
                vrow[base + j] = 2 * t + (0, 8, 1, 9)[j]
                vel[base + j] = 32 * (u // 4) + 4 * g + 2 * ((u // 2) % 2) + u % 2
    return krow, kel, vrow, vel


def _tile_maps():
    """(row, element) of every nibble of a 1024-byte code region, for the K and
    the V fragment orders, indexed [byte_offset * 2 + (0 low | 1 high nibble)]."""
    krow = np.zeros(2048, np.int64)
    kel = np.zeros(2048, np.int64)
    vrow = np.zeros(2048, np.int64)
    vel = np.zeros(2048, np.int64)
    for u in range(8):
        for lane in range(32):
            g, t = lane // 4, lane % 4
            base = 512 * (u // 4) + 16 * lane + 4 * (u % 4)
            for n in range(8):
                a, b, c = n & 1, (n >> 1) & 1, n >> 2
                slot = 2 * (base + n // 2) + (n % 2)
                krow[slot] = g + 8 * a
                kel[slot] = 8 * (t + 4 * (u // 2)) + 4 * (u % 2) + 2 * b + c
                vrow[slot] = 2 * t + 8 * b + c
                vel[slot] = 32 * (u // 2) + 4 * g + 2 * (u % 2) + a
    return krow, kel, vrow, vel


_MAPS = {}


def _maps(bits=4):
    if bits not in _MAPS:
        _MAPS[bits] = _tile_maps() if bits == 4 else _tile_maps8()
    return _MAPS[bits]


def _regions(bits_k, bits_v):
    """(offset, bits, 0 = K | 1 = V) of the two code regions, and the K / V
    metadata offsets, of a tile."""
    ck, cv = 256 * bits_k, 256 * bits_v
    return ((0, bits_k, 0), (ck, bits_v, 1)), ck + cv, ck + cv + 256


def _meta_offsets(kv):
    """Byte offsets [16 rows, 4 groups] of the FP16 scale and zero of every
    (row, group) inside a tile's 256-byte metadata region: K (kv = 0) row r
    at 16 r, its four scales then its four zeros; V (kv = 1) rows paired
    (2i, 2i + 1): the scale pair of group q at 16 i + 4 q, the zero pair 128
    bytes further."""
    r = np.arange(16)[:, None]
    q = np.arange(4)[None, :]
    if kv == 0:
        so = 16 * r + 2 * q
        return so, so + 8
    so = 16 * (r // 2) + 4 * q + 2 * (r % 2)
    return so, so + 128


def unpack_qblocks(blocks: np.ndarray, n_rows: int, bits_k: int = 4, bits_v: int = 4):
    """Decode the first ``n_rows`` rows of a quantised stream.

    blocks : uint8 [nblk, qblock_bytes] or [ntiles * qtile_bytes] (one
    (batch, KV head) stream of B_K-bit keys and B_V-bit values)
    Returns k_codes, v_codes uint8 [n_rows, 128]; k_scale, k_zero, v_scale,
    v_zero float16 [n_rows, 4].
    """
    regions, mk, mv = _regions(bits_k, bits_v)
    tiles = np.asarray(blocks, dtype=np.uint8).reshape(-1, L.qtile_bytes(bits_k, bits_v))
    nt = tiles.shape[0]
    out = [np.zeros((nt * 16, 128), np.uint8), np.zeros((nt * 16, 128), np.uint8)]
    for off, bits, kv in regions:
        maps = _maps(bits)
        rmap, emap = maps[2 * kv], maps[2 * kv + 1]
        size = 256 * bits      # code bytes of 16 rows
        for ti in range(nt):
            raw = tiles[ti, off:off + size]
            vals = np.stack([raw & 15, raw >> 4], axis=1).reshape(-1) if bits == 4 else raw
            out[kv][ti * 16 + rmap, emap] = vals
    meta = []
    for off, kv in ((mk, 0), (mv, 1)):
        so, zo = _meta_offsets(kv)
        m = tiles[:, off:off + 256].copy().view(np.float16)        # [nt, 128] halves
        meta.append((m[:, so // 2].reshape(nt * 16, 4), m[:, zo // 2].reshape(nt * 16, 4)))
    n = n_rows
    kc, vc = out
    return (kc[:n], vc[:n], meta[0][0][:n], meta[0][1][:n], meta[1][0][:n], meta[1][1][:n])


def pack_qblocks(k_codes, v_codes, k_scale, k_zero, v_scale, v_zero, bits_k: int = 4,
                 bits_v: int = 4) -> np.ndarray:
    """Inverse of ``unpack_qblocks``: rows padded with zeros to whole 64-row
    blocks; returns uint8 [nblk, qblock_bytes(bits_k, bits_v)]."""
    regions, mk, mv = _regions(bits_k, bits_v)
    n = k_codes.shape[0]
    nblk = -(-n // 64)
    nt = 4 * nblk
    tiles = np.zeros((nt, L.qtile_bytes(bits_k, bits_v)), np.uint8)

    def pad(a, shape, dtype):
        z = np.zeros(shape, dtype)
        z[: a.shape[0]] = a
        return z

    codes = [pad(np.asarray(k_codes), (nt * 16, 128), np.uint8), pad(np.asarray(v_codes), (nt * 16, 128), np.uint8)]
    for off, bits, kv in regions:
        maps = _maps(bits)
        rmap, emap = maps[2 * kv], maps[2 * kv + 1]
        size = 256 * bits      # code bytes of 16 rows
        for ti in range(nt):
            vals = codes[kv][ti * 16 + rmap, emap]
            if bits == 4:
                nib = vals.reshape(size, 2)
                vals = nib[:, 0] | (nib[:, 1] << 4)
            tiles[ti, off:off + size] = vals
    for off, kv, sc, zr in ((mk, 0, k_scale, k_zero), (mv, 1, v_scale, v_zero)):
        so, zo = _meta_offsets(kv)
        m = np.zeros((nt, 128), np.float16)
        m[:, so // 2] = pad(np.asarray(sc, np.float16), (nt * 16, 4), np.float16).reshape(nt, 16, 4)
        m[:, zo // 2] = pad(np.asarray(zr, np.float16), (nt * 16, 4), np.float16).reshape(nt, 16, 4)
        tiles[:, off:off + 256] = m.view(np.uint8)
    return tiles.reshape(nblk, 4 * L.qtile_bytes(bits_k, bits_v))


class HybridDecoder:
    """Decode-time driver of one layer (the re-selecting mode).

    Every ``period`` steps the vertical-line set is chosen again from the
    proxy ring against the caller's BF16 keys and the layout is rebuilt
    (select + rebuild); every step appends the token and runs the fused
    decode attention.
    """

    def __init__(self, cfg: HyqConfig, k_src: torch.Tensor, v_src: torch.Tensor, device="cuda"):
        self.cfg = cfg
        self.layer = HybridLayer(cfg, device)
        self.k_src, self.v_src = k_src, v_src
        self.ws_sel = workspace(cfg, L.OP_SELECT, cfg.capacity, device)
        self.ws_dec = workspace(cfg, L.OP_DECODE, cfg.capacity, device)
        kmax = max(1, L.hyq_vl_count(cfg, max(0, cfg.capacity - cfg.window)))
        self.idx = torch.zeros(cfg.batch, cfg.num_kv_heads, kmax, dtype=torch.int32, device=device)
        self.length = 0
        self.since = 0
        self.ring_n = 0

    def freeze(self, L_ctx: int, q_tail: torch.Tensor, stream=None):
        """Prefill -> decode (Algorithm 4): choose the vertical-line set from the
        tail queries ``q_tail`` [B, HQ, T, 128] and build the layout for the
        first ``L_ctx`` positions of k_src / v_src."""
        self.layer.reset(stream)
        self.maintain(L_ctx, q_tail, q_tail.shape[2], stream)
        self.length = L_ctx
        self.since = 0

    def maintain(self, L_ctx: int, q_proxy, n_proxy: int, stream=None):
        k = L.hyq_select_vertical(self.cfg, q_proxy, n_proxy, self.k_src, L_ctx,
                                  self.idx, self.ws_sel, stream) if n_proxy > 0 else 0
        if n_proxy == 0:
            k = 0
        L.hyq_rebuild(self.cfg, self.k_src, self.v_src, L_ctx, self.idx, k, self.layer.c, stream)
        return k

    def step(self, q, k_new, v_new, out, stream=None):
        """Append this token, re-select every ``period`` steps, attend.  Steps
        without maintenance run as one fused launch (hyq_decode_step)."""
        self.length += 1
        self.since += 1
        self.ring_n = min(self.ring_n + 1, self.cfg.period)
        if self.since < self.cfg.period:
            L.hyq_decode_step(self.cfg, q, k_new, v_new, self.layer.c, out, self.ws_dec, self.k_src, self.v_src,
                              self.cfg.capacity, stream)
            return out
        L.hyq_decode_append(self.cfg, q, k_new, v_new, self.layer.c, self.k_src, self.v_src, stream)
        self.maintain(self.length, self.layer.q_ring(), self.ring_n, stream)
        self.since = 0
        L.hyq_decode_attention(self.cfg, q, self.layer.c, out, self.ws_dec, self.cfg.capacity, stream)
        return out
