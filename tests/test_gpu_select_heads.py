"""GPU parity of Algorithm 1 per query head (hyq_config.vl_mode =
VL_PER_QUERY_HEAD): each query head's set, the stored per-KV-head list (the
union of the group's sets filled up to min(P, g k) by the group score), and a
decode over a cache built from that list.

Scores are float32 on the GPU and float64 in the oracle: every set must be a
valid top-k within the rigorous float32 bound (``check_selection``), and equal
to the oracle's wherever no key lies in the ambiguous band."""
import numpy as np
import pytest
import torch

from gen import decode_case
from hybrid_precision_quantized_gb300 import (HybridLayer, hyq_decode_attention, hyq_read_device_error,
                                              hyq_rebuild, hyq_select_vertical, hyq_select_vertical_heads,
                                              hyq_vl_count, make_config, workspace)
from hybrid_precision_quantized_gb300 import _lib as L
from oracle.attention import hybrid_decode
from oracle.select import (check_selection, prefix_len, score_error_bound, select_vertical_heads, vl_count,
                           vl_count_heads)
from tests.gpu_util import assert_attention_close, to_np

pytestmark = pytest.mark.gpu


def run_heads(c, Lc, W, ppm):
    B, HQ = c.q.shape[:2]
    HKV = c.k.shape[1]
    cfg = make_config(B, HQ, HKV, capacity=Lc, window=W, rho_ppm=ppm, vl_mode=L.VL_PER_QUERY_HEAD)
    ws = workspace(cfg, L.OP_SELECT, Lc)
    P = prefix_len(Lc, W)
    k, ku = vl_count(P, ppm), vl_count_heads(P, ppm, HQ // HKV)
    assert hyq_vl_count(cfg, P) == ku
    ih = torch.full((B, HQ, max(k, 1)), -1, dtype=torch.int32, device="cuda")
    ik = torch.full((B, HKV, max(ku, 1)), -1, dtype=torch.int32, device="cuda")
    qp, kk = c.q_proxy.cuda(), c.k.cuda()
    assert hyq_select_vertical_heads(cfg, qp, qp.shape[2], kk, Lc, ih, ik, ws) == (k, ku)
    # the per-KV-head entry point computes the same list on this config
    ik2 = torch.full_like(ik, -1)
    assert hyq_select_vertical(cfg, qp, qp.shape[2], kk, Lc, ik2, workspace(cfg, L.OP_SELECT, Lc)) == ku
    torch.cuda.synchronize()
    assert hyq_read_device_error(ws[:4].view(torch.int32)) == 0
    assert torch.equal(ik, ik2)
    return cfg, ih[..., :k].cpu().numpy(), ik[..., :ku].cpu().numpy()


def check_heads(c, Lc, W, ppm, got_h, got_kv):
    """Returns the number of ambiguous keys (0: the sets must equal the oracle's)."""
    qp, k_np = c.q_proxy.double().numpy(), c.k.double().numpy()
    B, HQ = qp.shape[:2]
    HKV = k_np.shape[1]
    g = HQ // HKV
    P = prefix_len(Lc, W)
    k, ku = vl_count(P, ppm), vl_count_heads(P, ppm, g)
    want_h, want_kv, _, S_h, S_g = select_vertical_heads(qp, k_np, Lc, W, ppm)
    # query head kh g + r scored alone against KV head kh: the bound with g = 1
    bnd_h = np.stack([score_error_bound(qp.reshape(B, HKV, g, *qp.shape[2:])[:, :, r], k_np, P)
                      for r in range(g)], axis=2).reshape(B, HQ, P)
    bnd_g = score_error_bound(qp, k_np, P)
    amb = 0
    for b in range(B):
        for h in range(HQ):
            res = check_selection(S_h[b, h], bnd_h[b, h], k, got_h[b, h])
            assert res["ok"], f"head {h}: {res['reason']}"
            amb += res["ambiguous"]
        for kh in range(HKV):
            union = np.unique(got_h[b, kh * g:(kh + 1) * g])
            S = S_g[b, kh].copy()
            bd = bnd_g[b, kh].copy()
            S[union] = np.inf                      # the union is taken first
            bd[union] = 0.0
            res = check_selection(S, bd, ku, got_kv[b, kh])
            assert res["ok"], f"KV head {kh}: {res['reason']}"
            amb += res["ambiguous"]
    if amb == 0:
        assert np.array_equal(got_h, want_h) and np.array_equal(got_kv, want_kv)
    return amb


@pytest.mark.parametrize("seed,B,HQ,HKV,Lc,W,ppm", [
    (1000, 1, 8, 2, 1024, 128, 50_000),      # g = 4
    (1001, 1, 32, 8, 4096, 128, 50_000),     # Llama-3.1-8B-shaped heads, 4K
    (1002, 2, 64, 8, 2048, 128, 20_000),     # g = 8, two sequences
    (1003, 1, 6, 2, 777, 100, 100_000),      # g = 3, ragged
    (1004, 1, 8, 8, 1500, 64, 50_000),       # MHA: the per-KV-head reading
])
def test_select_heads_parity(hyq, seed, B, HQ, HKV, Lc, W, ppm):
    c = decode_case(seed, B, HQ, HKV, Lc, window=W, n_proxy=64, sink_frac=0.02, outlier_channels=3)
    _, got_h, got_kv = run_heads(c, Lc, W, ppm)
    check_heads(c, Lc, W, ppm, got_h, got_kv)


def test_select_heads_llama_32k(hyq):
    """Llama-3.1-8B-shaped heads at 32K context (k = 1632 per query head,
    ku = 6528 per KV head)."""
    c = decode_case(1010, 1, 32, 8, 32768, window=128, n_proxy=64, sink_frac=0.02)
    _, got_h, got_kv = run_heads(c, 32768, 128, 50_000)
    assert got_h.shape == (1, 32, 1632) and got_kv.shape == (1, 8, 6528)
    check_heads(c, 32768, 128, 50_000, got_h, got_kv)


@pytest.mark.parametrize("seed,B,HQ,HKV,Lc,W,ppm", [(1020, 1, 32, 8, 3000, 128, 50_000),
                                                    (1021, 2, 8, 2, 900, 128, 100_000)])
def test_decode_over_per_head_lists(hyq, seed, B, HQ, HKV, Lc, W, ppm):
    """A cache built from the per-KV-head list (ku positions) decodes to the
    oracle's attention over the same partition."""
    c = decode_case(seed, B, HQ, HKV, Lc, window=W, n_proxy=64, sink_frac=0.02, outlier_channels=3)
    cfg, _, got_kv = run_heads(c, Lc, W, ppm)
    ku = got_kv.shape[-1]
    layer = HybridLayer(cfg)
    layer.reset()
    idx = torch.from_numpy(got_kv).to(torch.int32).cuda().contiguous()
    hyq_rebuild(cfg, c.k.cuda(), c.v.cuda(), Lc, idx, ku, layer.c)
    ws = workspace(cfg, L.OP_DECODE, 0)
    out = torch.empty(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    hyq_decode_attention(cfg, c.q.cuda(), layer.c, out, ws, 0)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) == 0
    want = hybrid_decode(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(), Lc,
                         prefix_len(Lc, W), got_kv)
    assert_attention_close(to_np(out), want, what=f"per-head lists, ku={ku}")
