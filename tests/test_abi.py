"""The C ABI without a GPU: the library loads, exports every symbol the header
declares, sizes buffers, and rejects invalid calls on the host before any
launch.  Also the block-format reader/writer used by the tests."""
import ctypes
import os
import re

import numpy as np
import pytest

import hybrid_precision_quantized_gb300 as hyq
from hybrid_precision_quantized_gb300 import _lib as L
from oracle.select import vl_count

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "hyq.h")


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(L.lib_path()):
        import __graft_entry__
        __graft_entry__.build()
    return hyq.load()


def declared_symbols():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(hyq_[a-z_]+)\s*\(", text)))


def test_header_declares_what_the_binding_binds():
    assert declared_symbols() == sorted(L.SYMBOLS)


def test_library_exports_every_declared_symbol(lib):
    for name in declared_symbols():
        assert hasattr(lib, name), name


def cfg(**kw):
    base = dict(batch=1, num_q_heads=32, num_kv_heads=8, capacity=32768)
    base.update(kw)
    return hyq.make_config(**base)


def test_config_checks(lib):
    assert hyq.hyq_config_check(cfg()) == 0
    assert hyq.hyq_config_check(cfg(head_dim=64)) == 2          # unsupported
    assert hyq.hyq_config_check(cfg(group=64)) == 2
    assert hyq.hyq_config_check(cfg(num_q_heads=72)) == 2       # g = 9 > 8
    assert hyq.hyq_config_check(cfg(num_q_heads=30)) == 1       # not a multiple
    assert hyq.hyq_config_check(cfg(rho_ppm=-1)) == 1
    assert hyq.hyq_config_check(cfg(rho_ppm=1_000_001)) == 1
    assert hyq.hyq_config_check(cfg(window=-1)) == 1
    assert hyq.hyq_config_check(cfg(capacity=0)) == 1
    assert lib.hyq_config_check(None) == 1


@pytest.mark.parametrize("ppm", [0, 20_000, 50_000, 100_000, 1_000_000, 333_333])
def test_vl_count_matches_oracle(lib, ppm):
    c = cfg(rho_ppm=ppm)
    for P in [0, 1, 19, 20, 21, 896, 4000, 32640, 131072]:
        assert hyq.hyq_vl_count(c, P) == vl_count(P, ppm)


def test_layout_sizes(lib):
    c = cfg()
    s = hyq.hyq_layout_sizes(c)
    assert len(s) == len(L.LAYOUT_FIELDS)
    assert s[0] == 8 * 512 * 10240                    # 32768 rows = 512 blocks per head
    assert s[1] == s[2] == -(-8 * 1632 * 256 // 256) * 256
    assert s[4] == 8 * (128 + 64) * 256
    assert s[6] == 32 * 64 * 256                      # proxy ring: 64 x HQ x d x 2 bytes (§5.5)
    assert all(x % 256 == 0 for x in s)


def test_workspace_sizes(lib):
    c = cfg()
    assert hyq.hyq_workspace_size(c, L.OP_DECODE, 32768) > 0
    assert hyq.hyq_workspace_size(c, L.OP_SELECT, 32768) >= 8 * 32640 * 4
    assert hyq.hyq_workspace_size(c, 99, 0) == 0
    assert hyq.hyq_workspace_size(cfg(head_dim=64), L.OP_DECODE, 0) == 0


def _null_layout():
    return L.HyqLayout()


def _no_gpu():
    import torch
    return not torch.cuda.is_available()


# Fake device addresses are only ever passed where no GPU exists, so that a
# validation gap could never turn into a launch that touches them.
@pytest.mark.skipif(not _no_gpu(), reason="fake-pointer validation runs only without a GPU")
def test_host_validation_rejects_before_launch(lib):
    c = cfg()
    lay = _null_layout()
    P = ctypes.POINTER
    # null layout pointers
    assert lib.hyq_decode_attention(ctypes.byref(c), 256, ctypes.byref(lay), 256, 0, 256, 1 << 30, None) == 1
    assert lib.hyq_rebuild(ctypes.byref(c), 256, 256, 100, 100, None, 0, ctypes.byref(lay), None) == 1
    assert lib.hyq_layout_reset(ctypes.byref(c), ctypes.byref(lay), None) == 1
    # a fake but aligned layout: argument checks that come after the layout check
    fake = L.HyqLayout(**{n: 4096 * (i + 1) for i, n in enumerate(L.LAYOUT_FIELDS)})
    assert lib.hyq_decode_attention(ctypes.byref(c), 256, ctypes.byref(fake), 256, 0, None, 0, None) == 3
    assert lib.hyq_decode_attention(ctypes.byref(c), 256, ctypes.byref(fake), 256, 0, 256, 16, None) == 3
    assert lib.hyq_decode_attention(ctypes.byref(c), 3, ctypes.byref(fake), 256, 0, 256, 1 << 30, None) == 1
    assert lib.hyq_rebuild(ctypes.byref(c), 256, 256, 100, 40000, None, 0, ctypes.byref(fake), None) == 4
    assert lib.hyq_rebuild(ctypes.byref(c), 256, 256, 99, 100, None, 0, ctypes.byref(fake), None) == 1
    assert lib.hyq_rebuild(ctypes.byref(c), 256, 256, 1000, 1000, None, 5, ctypes.byref(fake), None) == 1
    k_out = ctypes.c_int32(-1)
    # L <= W: nothing to select, k = 0, no launch
    assert lib.hyq_select_vertical(ctypes.byref(c), None, 0, 0, None, 100, 100, None,
                                   ctypes.byref(k_out), None, 0, None) == 0 and k_out.value == 0
    assert lib.hyq_select_vertical(ctypes.byref(c), 256, 64, 64, 256, 4096, 4096, 256,
                                   ctypes.byref(k_out), None, 0, None) == 3
    assert k_out.value == vl_count(4096 - 128, 50_000)
    assert lib.hyq_quantize_append(ctypes.byref(c), 256, 256, -1, ctypes.byref(fake), None) == 1
    assert lib.hyq_quantize_append(ctypes.byref(c), 256, 256, 0, ctypes.byref(fake), None) == 0
    assert lib.hyq_decode_append(ctypes.byref(c), 256, 256, 256, ctypes.byref(fake), 256, None, 10, None) == 1
    assert lib.hyq_read_device_error(None, None, None) == 1


def test_status_strings(lib):
    for s in range(7):
        assert hyq.hyq_status_string(s)


def test_block_format_round_trip():
    rng = np.random.default_rng(0)
    n = 150
    kc = rng.integers(0, 16, (n, 128), dtype=np.uint8)
    vc = rng.integers(0, 16, (n, 128), dtype=np.uint8)
    ks, kz, vs, vz = (rng.standard_normal((n, 4)).astype(np.float16) for _ in range(4))
    blocks = hyq.pack_qblocks(kc, vc, ks, kz, vs, vz)
    assert blocks.shape == (3, 10240)
    out = hyq.unpack_qblocks(blocks, n)
    for a, b in zip(out, (kc, vc, ks, kz, vs, vz)):
        assert np.array_equal(a, b)
    # every nibble slot of a tile is used exactly once by each fragment order
    from hybrid_precision_quantized_gb300.cache import _tile_maps
    krow, kel, vrow, vel = _tile_maps()
    assert len(set(zip(krow.tolist(), kel.tolist()))) == 2048
    assert len(set(zip(vrow.tolist(), vel.tolist()))) == 2048


def test_block_format_fragment_order_examples():
    """Spot values of the documented code order: the first word of lane 0
    holds K rows 0/8 elements 0,1,2,3 and V rows 0,1,8,9 of elements 0/1;
    lane 5 (g=1, t=1), u=3 holds K elements 8*(1+4)+4+.. = 44..47 of rows 1/9."""
    from hybrid_precision_quantized_gb300.cache import _tile_maps
    krow, kel, vrow, vel = _tile_maps()
    # nibble n of the word at byte 0: slot = 2*(n//2) + n%2 = n
    assert [(krow[n], kel[n]) for n in range(8)] == [(0, 0), (8, 0), (0, 2), (8, 2), (0, 1), (8, 1), (0, 3), (8, 3)]
    assert [(vrow[n], vel[n]) for n in range(8)] == [(0, 0), (0, 1), (8, 0), (8, 1), (1, 0), (1, 1), (9, 0), (9, 1)]
    base = 2 * (512 * 0 + 16 * 5 + 4 * 3)
    assert [(krow[base + n], kel[base + n]) for n in range(8)] == [
        (1, 44), (9, 44), (1, 46), (9, 46), (1, 45), (9, 45), (1, 47), (9, 47)]
    # V: element 32*(3//2) + 4*1 + 2*(3%2) + a = 38 + a
    assert [(vrow[base + n], vel[base + n]) for n in range(8)] == [
        (2, 38), (2, 39), (10, 38), (10, 39), (3, 38), (3, 39), (11, 38), (11, 39)]


@pytest.mark.parametrize("bk,bv", [(8, 8), (4, 8), (8, 4)])
def test_block_format_round_trip_wide_codes(bk, bv):
    rng = np.random.default_rng(bk * 10 + bv)
    n = 150
    kc = rng.integers(0, 1 << bk, (n, 128), dtype=np.uint8)
    vc = rng.integers(0, 1 << bv, (n, 128), dtype=np.uint8)
    ks, kz, vs, vz = (rng.standard_normal((n, 4)).astype(np.float16) for _ in range(4))
    blocks = hyq.pack_qblocks(kc, vc, ks, kz, vs, vz, bits_k=bk, bits_v=bv)
    assert blocks.shape == (3, L.qblock_bytes(bk, bv)) == (3, 4 * (256 * (bk + bv) + 512))
    out = hyq.unpack_qblocks(blocks, n, bits_k=bk, bits_v=bv)
    for a, b in zip(out, (kc, vc, ks, kz, vs, vz)):
        assert np.array_equal(a, b)


def test_eight_bit_order_follows_the_fragment_rule():
    """Every (row, element) of a 16 x 128 tile appears once in each 8-bit
    order; in a K word the AND half (bytes 0, 2) and the permuted half (bytes
    1, 3) are consecutive element pairs of one row, four consecutive elements
    in all; a V word holds one element of tokens 2t, 2t+8, 2t+1, 2t+9."""
    from hybrid_precision_quantized_gb300.cache import _tile_maps8
    krow, kel, vrow, vel = _tile_maps8()
    assert len(set(zip(krow.tolist(), kel.tolist()))) == 2048
    assert len(set(zip(vrow.tolist(), vel.tolist()))) == 2048
    for base in range(0, 2048, 4):
        w = slice(base, base + 4)
        assert len(set(krow[w].tolist())) == 1
        assert (kel[base + 2], kel[base + 1], kel[base + 3]) == (kel[base] + 1, kel[base] + 2, kel[base] + 3)
        assert kel[base] % 4 == 0
        assert len(set(vel[w].tolist())) == 1
        t = vrow[base] // 2
        assert tuple(vrow[w].tolist()) == (2 * t, 2 * t + 8, 2 * t + 1, 2 * t + 9)
    # a lane's 16 words: K keys g and g + 8, 16-element k-steps in order
    lane = 9   # g = 2, t = 1
    ku = [(krow[512 * (u // 4) + 16 * lane + 4 * (u % 4)], kel[512 * (u // 4) + 16 * lane + 4 * (u % 4)])
          for u in range(16)]
    assert ku == [(2 + 8 * (u % 2), 16 * (u // 2) + 4) for u in range(16)]


def test_code_widths_are_validated(lib):
    ok = hyq.make_config(1, 4, 2, 256, bits_k=8, bits_v=4)
    assert L.hyq_config_check(ok) == 0
    assert L.hyq_config_check(hyq.make_config(1, 4, 2, 256, bits_k=0, bits_v=0)) == 0   # 0 means 4
    for bk, bv in [(5, 4), (4, 2), (16, 8), (-4, 4)]:
        assert L.hyq_config_check(hyq.make_config(1, 4, 2, 256, bits_k=bk, bits_v=bv)) != 0


def test_stream_size_follows_the_code_widths(lib):
    sizes = {(bk, bv): L.hyq_layout_sizes(hyq.make_config(2, 8, 2, 1000, bits_k=bk, bits_v=bv))
             for bk in (4, 8) for bv in (4, 8)}
    nblk = -(-1000 // 64)
    for (bk, bv), s in sizes.items():
        assert s[0] == -(-(2 * 2 * nblk * L.qblock_bytes(bk, bv)) // 256) * 256
        assert s[1:] == sizes[(4, 4)][1:]       # BF16 buffers do not depend on the widths


def test_prefill_band_workspace_holds_the_position_images(lib):
    """The band workspace adds BF16 key and value images of all L positions
    (2 x ceil(L / 128) images of 32 KiB per KV head) and drops the window
    from the full-precision list (at most two images at W = 128)."""
    c = cfg()
    for Lc in (1000, 8192):
        fixed = hyq.hyq_workspace_size(c, L.OP_PREFILL, Lc)
        band = hyq.hyq_workspace_size(c, L.OP_PREFILL_BAND, Lc)
        bh, img, ntb = c.batch * c.num_kv_heads, 32768, -(-Lc // 128)
        assert 2 * bh * img * (ntb - 2) <= band - fixed <= 2 * bh * img * ntb + 4096


def test_decode_plan_override_is_validated_and_sizes_the_workspace(lib):
    c = cfg()
    try:
        for merge, splits in [(5, 0), (-1, 0), (2, 1), (2, 17), (3, 0), (3, 1025)]:
            with pytest.raises(hyq.HyqError):
                hyq.hyq_set_decode_plan(merge, splits)
        hyq.hyq_set_decode_plan(3, 2)
        small = hyq.hyq_workspace_size(c, L.OP_DECODE, 32768)
        hyq.hyq_set_decode_plan(3, 7)
        large = hyq.hyq_workspace_size(c, L.OP_DECODE, 32768)
        bh = c.batch * c.num_kv_heads
        assert large - small >= bh * 5 * 8 * 130 * 4      # five more partial slots per (sequence, KV head)
    finally:
        hyq.hyq_set_decode_plan(0, 0)
