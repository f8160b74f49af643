"""GPU parity of the code-width variants (B_K, B_V) in {4, 8}^2: the
quantiser's codes, FP16 scales and zeros bit-exact with the oracle at each
tensor's own width (append, rebuild, tail aging), and decode attention within
|gpu - oracle| <= 2e-3 + 1e-2 |oracle| of the oracle over the cache
dequantised at those widths (Algorithm 4 quantises K and V with B_K and B_V
bits)."""
import numpy as np
import pytest
import torch

from gen import decode_case, gen_for
from hybrid_precision_quantized_gb300 import (HybridLayer, hyq_age_tail, hyq_decode_attention, hyq_decode_step,
                                              hyq_quantize_append, hyq_read_device_error, hyq_rebuild,
                                              hyq_set_decode_plan, make_config, workspace)
from hybrid_precision_quantized_gb300 import _lib as L
from oracle.attention import hybrid_decode
from oracle.select import prefix_len, select_vertical
from tests.gpu_util import assert_attention_close, mixed_rows, to_np
from tests.test_gpu_decode import build_and_decode, layer_counts
from tests.test_gpu_quant import _check_positional, _check_stream

pytestmark = pytest.mark.gpu

WIDE = [(8, 8), (4, 8), (8, 4)]


def wide_rows(seed, shape):
    """mixed_rows plus an 8-bit tie row: group 0 of row 4 spans 0 .. 255/16
    (step exactly 1/16 at 8 bits) with every other element an odd multiple of
    1/32, i.e. exactly halfway between two 8-bit codes."""
    x = mixed_rows(seed, shape).float()
    flat = x.view(-1, shape[-2], 128)
    if shape[-2] > 4:
        flat[:, 4, :32] = (2 * torch.arange(32) % 256 + 1) / 32.0
        flat[:, 4, 0], flat[:, 4, 1] = 0.0, 255.0 / 16
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("bk,bv", WIDE)
def test_append_bit_exact_wide_codes(hyq, bk, bv):
    B, HQ, HKV = 2, 4, 2
    cfg = make_config(B, HQ, HKV, capacity=512, window=0, bits_k=bk, bits_v=bv)
    layer = HybridLayer(cfg)
    layer.reset()
    k1, v1 = wide_rows(21, (B, HKV, 150, 128)), wide_rows(22, (B, HKV, 150, 128))
    k2, v2 = wide_rows(23, (B, HKV, 37, 128)), wide_rows(24, (B, HKV, 37, 128))
    hyq_quantize_append(cfg, k1.cuda(), v1.cuda(), 150, layer.c)
    hyq_quantize_append(cfg, k2.cuda(), v2.cuda(), 37, layer.c)   # starts inside a block
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) == 0
    assert layer.counts().cpu().numpy()[:, L.CNT_NQ].tolist() == [187, 187]
    for b in range(B):
        for h in range(HKV):
            _check_stream(layer, b, h, 187, torch.cat([k1[b, h], k2[b, h]]).double().numpy(),
                          torch.cat([v1[b, h], v2[b, h]]).double().numpy())


@pytest.mark.parametrize("bk,bv", WIDE)
@pytest.mark.parametrize("B,HQ,HKV,Lc,W,ppm", [
    (2, 8, 2, 777, 100, 50_000),      # ragged stream, two sequences
    (1, 4, 1, 300, 64, 0),            # no vertical lines
])
def test_rebuild_bit_exact_wide_codes(hyq, bk, bv, B, HQ, HKV, Lc, W, ppm):
    c = decode_case(25, B, HQ, HKV, Lc, window=W, n_proxy=16, sink_frac=0.03)
    k_rows, v_rows = wide_rows(26, (B, HKV, Lc, 128)), wide_rows(27, (B, HKV, Lc, 128))
    cfg = make_config(B, HQ, HKV, capacity=Lc + 64, window=W, rho_ppm=ppm, bits_k=bk, bits_v=bv)
    layer = HybridLayer(cfg)
    layer.reset()
    idx_np, _ = select_vertical(c.q_proxy.double().numpy(), k_rows.double().numpy(), Lc, W, ppm)
    k = idx_np.shape[-1]
    P = prefix_len(Lc, W)
    idx = torch.from_numpy(idx_np).to(torch.int32).cuda().contiguous()
    hyq_rebuild(cfg, k_rows.cuda(), v_rows.cuda(), Lc, idx, k, layer.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) == 0
    for b in range(B):
        for h in range(HKV):
            _check_positional(layer, b, h, P, k_rows[b, h].double().numpy(), v_rows[b, h].double().numpy(),
                              idx_np[b, h])


@pytest.mark.parametrize("bk,bv", WIDE)
@pytest.mark.parametrize("seed,B,HQ,HKV,Lc,W,ppm", [
    (1000, 1, 4, 4, 1024, 128, 50_000),     # tiny decode workload
    (1001, 1, 32, 8, 4096, 128, 50_000),    # Llama-3.1-8B-shaped, 4K
    (5, 2, 8, 2, 777, 100, 50_000),         # two sequences, ragged stream
    (1003, 1, 64, 8, 2048, 128, 50_000),    # g = 8
    (7, 1, 6, 2, 500, 128, 50_000),         # g = 3
])
def test_decode_parity_wide_codes(hyq, bk, bv, seed, B, HQ, HKV, Lc, W, ppm):
    c = decode_case(seed, B, HQ, HKV, Lc, window=W, n_proxy=64, sink_frac=0.02, outlier_channels=3)
    got, want, _ = build_and_decode(c, Lc, W, ppm, bits=(bk, bv))
    assert_attention_close(got, want, what=f"K{bk}V{bv} L={Lc}")


@pytest.mark.parametrize("bk,bv", WIDE)
@pytest.mark.parametrize("Lc,W,ppm,what", [
    (600, 0, 0, "rho = 0, W = 0: all quantised"),
    (129, 128, 50_000, "P = 1"),
    (193, 128, 0, "one block plus one row"),
    (1, 128, 50_000, "single position"),
])
def test_decode_edge_cases_wide_codes(hyq, bk, bv, Lc, W, ppm, what):
    c = decode_case(31, 1, 8, 2, Lc, window=W, n_proxy=16, sink_frac=0.03)
    got, want, _ = build_and_decode(c, Lc, W, ppm, bits=(bk, bv))
    assert_attention_close(got, want, what=f"K{bk}V{bv} {what}")


@pytest.mark.parametrize("merge,splits", [(1, 0), (2, 4), (3, 2), (3, 19)])
def test_decode_every_merge_plan_wide_codes(hyq, merge, splits):
    """Direct, workspace merges with 2 and 19 splits, and a cluster request
    (served by the workspace merge for 8-bit codes) all match the oracle."""
    c = decode_case(32, 1, 16, 4, 3000, window=128, n_proxy=16, sink_frac=0.02)
    try:
        hyq_set_decode_plan(merge, splits)
        got, want, _ = build_and_decode(c, 3000, 128, 50_000, bits=(8, 8))
    finally:
        hyq_set_decode_plan(0, 0)
    assert_attention_close(got, want, what=f"plan {merge}/{splits}")


def test_decode_full_size_llama_32k_k8v8(hyq):
    """The benchmark's layer shape (Llama-3.1-8B-shaped heads, 32K, W 128,
    rho 5%) with 8-bit keys and values, every head against the oracle."""
    c = decode_case(1002, 1, 32, 8, 32768, window=128, n_proxy=64, sink_frac=0.02, outlier_channels=3)
    got, want, _ = build_and_decode(c, 32768, 128, 50_000, bits=(8, 8))
    assert_attention_close(got, want, what="K8V8 32K")


@pytest.mark.parametrize("bk,bv", [(8, 8), (4, 8)])
def test_fused_steps_and_tail_aging_wide_codes(hyq, bk, bv):
    """Fused decode steps, then hyq_age_tail (frozen mode): the aged rows
    join the stream bit-exact at their widths, and attention before and after
    matches the oracle."""
    B, HQ, HKV, W, ppm, T = 1, 8, 2, 128, 50_000, 64
    L0 = 700
    cap = L0 + T
    c = decode_case(33, B, HQ, HKV, cap, window=W, n_proxy=16, sink_frac=0.02)
    cfg = make_config(B, HQ, HKV, capacity=cap, window=W, rho_ppm=ppm, bits_k=bk, bits_v=bv)
    lay = HybridLayer(cfg)
    lay.reset()
    idx_np, _ = select_vertical(c.q_proxy.double().numpy(), c.k[:, :, :L0].double().numpy(), L0, W, ppm)
    k = idx_np.shape[-1]
    idx = torch.from_numpy(idx_np).to(torch.int32).cuda().contiguous()
    ks = torch.zeros(B, HKV, cap, 128, dtype=torch.bfloat16, device="cuda")
    vs = torch.zeros_like(ks)
    ks[:, :, :L0] = c.k[:, :, :L0].cuda()
    vs[:, :, :L0] = c.v[:, :, :L0].cuda()
    hyq_rebuild(cfg, ks, vs, L0, idx, k, lay.c)
    ws = workspace(cfg, L.OP_DECODE, cap)
    out = torch.empty(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    g = gen_for(33, "q-steps")
    k_np, v_np = c.k.double().numpy(), c.v.double().numpy()
    Lc = L0
    for _ in range(T):
        q = torch.randn(B, HQ, 128, generator=g).to(torch.bfloat16)
        hyq_decode_step(cfg, q.cuda(), c.k[:, :, Lc].contiguous().cuda(), c.v[:, :, Lc].contiguous().cuda(),
                        lay.c, out, ws, ks, vs, cap)
        Lc += 1
    torch.cuda.synchronize()
    P0 = L0 - W
    want = hybrid_decode(q.double().numpy(), k_np, v_np, Lc, P0, idx_np, bits=bk, bits_v=bv)
    assert_attention_close(to_np(out), want, what=f"K{bk}V{bv} after {T} fused steps")
    hyq_age_tail(cfg, lay.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(lay.err()) == 0
    P = Lc - W
    assert layer_counts(lay)[:4] == [P, k, W, Lc]
    for h in range(HKV):
        _check_positional(lay, 0, h, P, c.k[0, h].double().numpy(), c.v[0, h].double().numpy(), idx_np[0, h])
    q = torch.randn(B, HQ, 128, generator=g).to(torch.bfloat16)
    hyq_decode_attention(cfg, q.cuda(), lay.c, out, ws, cap)
    torch.cuda.synchronize()
    want = hybrid_decode(q.double().numpy(), k_np, v_np, Lc, P, idx_np, bits=bk, bits_v=bv)
    assert_attention_close(to_np(out), want, what=f"K{bk}V{bv} after aging")
