"""GPU parity of the 4-bit quantiser and the cache rebuild: codes, FP16 scales
and zeros bit-exact with the oracle; vertical-line rows, tail rows and
counters exact."""
import numpy as np
import pytest
import torch

from gen import decode_case
from hybrid_precision_quantized_gb300 import (HybridLayer, hyq_quantize_append, hyq_read_device_error,
                                              hyq_rebuild, make_config, unpack_qblocks)
from hybrid_precision_quantized_gb300 import _lib as L
from oracle.quant import quantize
from oracle.select import prefix_len, select_vertical, vl_count
from tests.gpu_util import mixed_rows

pytestmark = pytest.mark.gpu


def _check_stream(layer, b, h, n_rows, k_rows, v_rows):
    bk, bv = layer.cfg.bits_k or 4, layer.cfg.bits_v or 4
    blocks = layer.qblocks()[b, h].cpu().numpy()
    kc, vc, ks, kz, vs, vz = unpack_qblocks(blocks, n_rows, bk, bv)
    for got_c, got_s, got_z, rows, bits in ((kc, ks, kz, k_rows, bk), (vc, vs, vz, v_rows, bv)):
        c, s, z = quantize(rows, bits)
        assert np.array_equal(got_c, c), f"codes differ at {np.argwhere(got_c != c)[:5].tolist()}"
        assert np.array_equal(got_s.view(np.uint16), s.view(np.uint16)), "scales differ"
        assert np.array_equal(got_z.view(np.uint16), z.view(np.uint16)), "zeros differ"
    # rows past the stream end inside the last block are zero
    if n_rows % 64:
        kc_all, vc_all, ks_all, *_ = unpack_qblocks(blocks, blocks.shape[0] * 64, bk, bv)
        assert not kc_all[n_rows:(n_rows + 63) // 64 * 64].any()


def _check_positional(layer, b, h, P, k_rows, v_rows, vl):
    """The stream of (b, h) holds positions [0, P) at row = position, every
    code, step and zero equal to the oracle quantiser's on those rows, except
    that the vertical-line positions ``vl`` carry FP16 NaN as their key steps
    (decode leaves them out)."""
    bk, bv = layer.cfg.bits_k or 4, layer.cfg.bits_v or 4
    blocks = layer.qblocks()[b, h].cpu().numpy()
    kc, vc, ks, kz, vs, vz = unpack_qblocks(blocks, P, bk, bv)
    ck, sk, zk = quantize(k_rows[:P], bk)
    cv, sv, zv = quantize(v_rows[:P], bv)
    vl = np.asarray(vl, np.int64)
    assert np.array_equal(kc, ck) and np.array_equal(vc, cv), "codes differ"
    assert np.array_equal(kz.view(np.uint16), zk.view(np.uint16)) and np.array_equal(vz.view(np.uint16),
                                                                                      zv.view(np.uint16))
    assert np.array_equal(vs.view(np.uint16), sv.view(np.uint16)), "value steps differ"
    marked = np.zeros(P, bool)
    marked[vl] = True
    assert np.all(np.isnan(ks[marked].astype(np.float64))), "a vertical-line row is not marked"
    assert np.array_equal(ks[~marked].view(np.uint16), sk[~marked].view(np.uint16)), "key steps differ"


def test_quantize_append_bit_exact_two_appends(hyq):
    B, HQ, HKV = 2, 4, 2
    cfg = make_config(B, HQ, HKV, capacity=512, window=0)
    layer = HybridLayer(cfg)
    layer.reset()
    k1, v1 = mixed_rows(1, (B, HKV, 150, 128)), mixed_rows(2, (B, HKV, 150, 128))
    k2, v2 = mixed_rows(3, (B, HKV, 37, 128)), mixed_rows(4, (B, HKV, 37, 128))
    hyq_quantize_append(cfg, k1.cuda(), v1.cuda(), 150, layer.c)
    hyq_quantize_append(cfg, k2.cuda(), v2.cuda(), 37, layer.c)   # starts inside a block
    torch.cuda.synchronize()
    cnt = layer.counts().cpu().numpy()
    assert cnt[:, L.CNT_NQ].tolist() == [187, 187] and cnt[:, L.CNT_LEN].tolist() == [187, 187]
    assert hyq_read_device_error(layer.err()) == 0
    for b in range(B):
        for h in range(HKV):
            kr = torch.cat([k1[b, h], k2[b, h]]).double().numpy()
            vr = torch.cat([v1[b, h], v2[b, h]]).double().numpy()
            _check_stream(layer, b, h, 187, kr, vr)


def test_quantize_range_error_sets_device_word(hyq):
    cfg = make_config(1, 1, 1, capacity=128, window=0)
    layer = HybridLayer(cfg)
    layer.reset()
    k = mixed_rows(5, (1, 1, 4, 128))
    k[0, 0, 2, 40] = -70000.0           # group 1 of row 2: zero point overflows FP16
    v = mixed_rows(6, (1, 1, 4, 128))
    hyq_quantize_append(cfg, k.cuda(), v.cuda(), 4, layer.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) & L.DEVERR_QUANT_RANGE
    kc, vc, ks, kz, vs, vz = unpack_qblocks(layer.qblocks()[0, 0].cpu().numpy(), 4)
    assert not kc[2, 32:64].any() and ks[2, 1] == 0 and kz[2, 1] == 0
    c, s, z = quantize(k[0, 0, [0, 1, 3]].double().numpy())
    assert np.array_equal(kc[[0, 1, 3]], c)


def test_append_past_capacity_is_dropped_and_flagged(hyq):
    cfg = make_config(1, 1, 1, capacity=64, window=0)
    layer = HybridLayer(cfg)
    layer.reset()
    k = mixed_rows(7, (1, 1, 60, 128))
    hyq_quantize_append(cfg, k.cuda(), k.cuda(), 60, layer.c)
    hyq_quantize_append(cfg, k.cuda(), k.cuda(), 10, layer.c)   # only 4 rows fit
    torch.cuda.synchronize()
    assert layer.counts()[0, L.CNT_NQ].item() == 64
    assert hyq_read_device_error(layer.err()) & L.DEVERR_COUNT


@pytest.mark.parametrize("B,HQ,HKV,Lc,W,ppm", [
    (1, 4, 4, 1024, 128, 50_000),     # tiny decode workload
    (2, 8, 2, 777, 100, 50_000),      # ragged stream, two sequences
    (1, 4, 1, 300, 128, 0),           # no vertical lines
    (1, 4, 1, 300, 64, 1_000_000),    # everything in the prefix is vertical-line
    (1, 4, 2, 100, 128, 50_000),      # context inside the window: empty stream
])
def test_rebuild_matches_partition(hyq, B, HQ, HKV, Lc, W, ppm):
    c = decode_case(11, B, HQ, HKV, Lc, window=W, n_proxy=16, sink_frac=0.03)
    cfg = make_config(B, HQ, HKV, capacity=Lc + 64, window=W, rho_ppm=ppm)
    layer = HybridLayer(cfg)
    layer.reset()
    kq, vq = c.k.cuda(), c.v.cuda()
    idx_np, _ = select_vertical(c.q_proxy.double().numpy(), c.k.double().numpy(), Lc, W, ppm)
    k = idx_np.shape[-1]
    P = prefix_len(Lc, W)
    assert k == vl_count(P, ppm)
    idx = torch.from_numpy(idx_np).to(torch.int32).cuda().contiguous()
    hyq_rebuild(cfg, kq, vq, Lc, idx, k, layer.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) == 0
    cnt = layer.counts().cpu().numpy()
    assert cnt[:, :4].tolist() == [[P, k, Lc - P, Lc]] * B
    for b in range(B):
        for h in range(HKV):
            if P:
                _check_positional(layer, b, h, P, c.k[b, h].double().numpy(), c.v[b, h].double().numpy(),
                                  idx_np[b, h])
            assert torch.equal(layer.vl_k()[b, h, :k].cpu(), c.k[b, h, idx_np[b, h]])
            assert torch.equal(layer.vl_v()[b, h, :k].cpu(), c.v[b, h, idx_np[b, h]])
            assert np.array_equal(layer.vl_idx()[b, h, :k].cpu().numpy(), idx_np[b, h])
            assert torch.equal(layer.tail_k()[b, h, :Lc - P].cpu(), c.k[b, h, P:Lc])
            assert torch.equal(layer.tail_v()[b, h, :Lc - P].cpu(), c.v[b, h, P:Lc])


def test_rebuild_flags_unsorted_index_list(hyq):
    c = decode_case(12, 1, 2, 1, 400, window=128, n_proxy=4)
    cfg = make_config(1, 2, 1, capacity=512)
    layer = HybridLayer(cfg)
    layer.reset()
    idx = torch.tensor([[[5, 3, 9]]], dtype=torch.int32).cuda()
    hyq_rebuild(cfg, c.k.cuda(), c.v.cuda(), 400, idx, 3, layer.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) & L.DEVERR_INDEX


def test_rebuild_bit_exact_on_edge_groups(hyq):
    """Rebuild of rows with widely different group ranges, constant groups,
    unit-grid ties, subnormal-size steps, and two planted groups whose code
    argument (x - z) / s reaches exactly -0.5 and 15.5 (zero point rounded
    off an FP16 subnormal), where the clamp of the code decision acts."""
    B, HQ, HKV, Lc, W = 1, 2, 2, 400, 64
    P = Lc - W
    k_rows, v_rows = mixed_rows(8, (B, HKV, Lc, 128)), mixed_rows(9, (B, HKV, Lc, 128))
    g = torch.Generator().manual_seed(10)
    for x in (k_rows, v_rows):
        x[0, :, 10, 0:32] = 1.5 * 2.0 ** -24       # z rounds up by half a step: argument -0.5
        x[0, :, 10, 1] = 15.5 * 2.0 ** -24
        x[0, :, 11, 96:128] = 2.5 * 2.0 ** -24     # z rounds down by half a step: argument 15.5
        x[0, :, 11, 97] = 17.5 * 2.0 ** -24
        x[0, :, 12:20, 32:64] = (1e-7 * torch.randn(2, 8, 32, generator=g)).to(torch.bfloat16)
    idx_np = np.stack([np.arange(3, P, 13), np.arange(5, P, 13)])[None].astype(np.int64)
    k = idx_np.shape[-1]   # 26 of 336: a 10% ratio leaves room for them
    cfg = make_config(B, HQ, HKV, capacity=Lc + 64, window=W, rho_ppm=100_000)
    layer = HybridLayer(cfg)
    layer.reset()
    idx = torch.from_numpy(idx_np).to(torch.int32).cuda().contiguous()
    hyq_rebuild(cfg, k_rows.cuda(), v_rows.cuda(), Lc, idx, k, layer.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) == 0
    for h in range(HKV):
        _check_positional(layer, 0, h, P, k_rows[0, h].double().numpy(), v_rows[0, h].double().numpy(),
                          idx_np[0, h])


@pytest.mark.parametrize("bits", [(4, 4), (8, 8), (4, 8)])
def test_codes_at_planted_midpoints_bit_exact(hyq, bits):
    """Groups on grids whose step has an inexact float32 reciprocal, with
    elements at exact midpoints (the even code) and one BF16 step either side
    (the nearer code): appended in two calls (the second starts inside a
    block, so both the word-at-a-time and the per-element code paths run)
    and rebuilt, every code, scale and zero equal to the oracle's."""
    from tests.gpu_util import tie_rows
    B, HQ, HKV, n1, n2 = 1, 2, 2, 70, 50
    cfg = make_config(B, HQ, HKV, capacity=256, window=0, bits_k=bits[0], bits_v=bits[1])
    layer = HybridLayer(cfg)
    layer.reset()
    k = tie_rows(21, (B, HKV, n1 + n2, 128), bits[0])
    v = tie_rows(22, (B, HKV, n1 + n2, 128), bits[1])
    hyq_quantize_append(cfg, k[:, :, :n1].contiguous().cuda(), v[:, :, :n1].contiguous().cuda(), n1, layer.c)
    hyq_quantize_append(cfg, k[:, :, n1:].contiguous().cuda(), v[:, :, n1:].contiguous().cuda(), n2, layer.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) == 0
    for h in range(HKV):
        _check_stream(layer, 0, h, n1 + n2, k[0, h].double().numpy(), v[0, h].double().numpy())
    # the same rows through the rebuild (W = 0, no vertical lines)
    cfg2 = make_config(B, HQ, HKV, capacity=256, window=0, rho_ppm=0, bits_k=bits[0], bits_v=bits[1])
    layer2 = HybridLayer(cfg2)
    layer2.reset()
    idx = torch.zeros(B, HKV, 1, dtype=torch.int32, device="cuda")
    hyq_rebuild(cfg2, k.cuda(), v.cuda(), n1 + n2, idx, 0, layer2.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer2.err()) == 0
    for h in range(HKV):
        _check_stream(layer2, 0, h, n1 + n2, k[0, h].double().numpy(), v[0, h].double().numpy())


def test_rebuild_incremental_equals_fresh(hyq):
    """A rebuild over a layout already built for a shorter context (the
    re-selection every 64 tokens) quantises only the new positions and moves
    the vertical-line marks; the result is bit-identical to building the new
    context on a fresh layout, with a different index set (positions leave
    and join the set)."""
    B, HQ, HKV, L1, W, ppm = 2, 8, 2, 700, 128, 50_000
    L2 = L1 + 64
    c = decode_case(13, B, HQ, HKV, L2, window=W, n_proxy=16, sink_frac=0.03)
    cfg = make_config(B, HQ, HKV, capacity=L2 + 64, window=W, rho_ppm=ppm)
    kq, vq = c.k.cuda(), c.v.cuda()
    idx1, _ = select_vertical(c.q_proxy.double().numpy(), c.k.double().numpy(), L1, W, ppm)
    q2 = c.q_proxy.double().numpy()[:, :, ::-1] * np.array([1.0, -0.5])[None, None, :, None].repeat(8, 2)
    idx2, _ = select_vertical(q2, c.k.double().numpy(), L2, W, ppm)
    assert len(np.setdiff1d(idx1[0, 0], idx2[0, 0])) > 0          # some positions leave the set
    inc, fresh = HybridLayer(cfg), HybridLayer(cfg)
    inc.reset()
    fresh.reset()
    for lay, steps in ((inc, ((L1, idx1), (L2, idx2))), (fresh, ((L2, idx2),))):
        for Lc, ix in steps:
            t = torch.from_numpy(ix).to(torch.int32).cuda().contiguous()
            hyq_rebuild(cfg, kq, vq, Lc, t, ix.shape[-1], lay.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(inc.err()) == 0 and hyq_read_device_error(fresh.err()) == 0
    P2 = L2 - W
    assert torch.equal(inc.counts(), fresh.counts())
    rows = (P2 + 15) // 16 * 16
    ib, fb = inc.qblocks().cpu().numpy(), fresh.qblocks().cpu().numpy()
    for b in range(B):
        for h in range(HKV):
            a = ib[b, h].reshape(-1)[:rows // 16 * 2560]
            f = fb[b, h].reshape(-1)[:rows // 16 * 2560]
            assert np.array_equal(a, f)
            _check_positional(inc, b, h, P2, c.k[b, h].double().numpy(), c.v[b, h].double().numpy(), idx2[b, h])
    k2 = idx2.shape[-1]
    assert torch.equal(inc.vl_k()[:, :, :k2], fresh.vl_k()[:, :, :k2])
    assert torch.equal(inc.tail_k()[:, :, :L2 - P2], fresh.tail_k()[:, :, :L2 - P2])
