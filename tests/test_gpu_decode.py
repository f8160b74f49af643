"""GPU parity of hybrid decode attention (Eq. 8-9, Algorithm 3) against the
oracle's plain float64 softmax over the effective cache.

The partition (vertical-line set) fed to the GPU is always the oracle's own
selection, so the attention comparison does not depend on selection parity.
Tolerance: |gpu - oracle| <= 2e-3 + 1e-2 |oracle| elementwise.
"""
import numpy as np
import pytest
import torch

from gen import decode_case, gen_for
from hybrid_precision_quantized_gb300 import (HybridDecoder, HybridLayer, hyq_decode_append,
                                              hyq_decode_attention, hyq_read_device_error,
                                              hyq_rebuild, make_config, workspace)
from hybrid_precision_quantized_gb300 import _lib as L
from oracle.attention import hybrid_decode
from oracle.select import check_selection, prefix_len, score_error_bound, select_vertical
from tests.gpu_util import assert_attention_close, sample_pairs, to_np

pytestmark = pytest.mark.gpu


def build_and_decode(c, Lc, W, ppm, capacity=None, len_hint=0, period=64, bits=(4, 4)):
    got, idx_np, st = decode_gpu(c, Lc, W, ppm, capacity, len_hint, period, bits)
    k_np, v_np = c.k.double().numpy(), c.v.double().numpy()
    want = hybrid_decode(c.q.double().numpy(), k_np, v_np, Lc, prefix_len(Lc, W), idx_np, bits=bits[0],
                         bits_v=bits[1])
    return got, want, st


def decode_gpu(c, Lc, W, ppm, capacity=None, len_hint=0, period=64, bits=(4, 4)):
    """Layout from the oracle's selection (B_K, B_V = ``bits``), then one GPU
    decode call."""
    B, HQ = c.q.shape[:2]
    HKV = c.k.shape[1]
    cfg = make_config(B, HQ, HKV, capacity=capacity or max(Lc, 1), window=W, rho_ppm=ppm, period=period,
                      bits_k=bits[0], bits_v=bits[1])
    layer = HybridLayer(cfg)
    layer.reset()
    qp = c.q_proxy.double().numpy()
    k_np, v_np = c.k.double().numpy(), c.v.double().numpy()
    idx_np, _ = select_vertical(qp, k_np, Lc, W, ppm)
    k = idx_np.shape[-1]
    idx = torch.from_numpy(idx_np).to(torch.int32).cuda().contiguous()
    hyq_rebuild(cfg, c.k.cuda(), c.v.cuda(), Lc, idx, k, layer.c)
    ws = workspace(cfg, L.OP_DECODE, len_hint)
    out = torch.empty(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    hyq_decode_attention(cfg, c.q.cuda(), layer.c, out, ws, len_hint)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) == 0
    return to_np(out), idx_np, (cfg, layer, ws, out)


@pytest.mark.parametrize("seed,B,HQ,HKV,Lc,W,ppm", [
    (1000, 1, 4, 4, 1024, 128, 50_000),     # tiny decode workload
    (1001, 1, 32, 8, 1024, 128, 50_000),    # Llama-3.1-8B-shaped, 1K
    (1001, 1, 32, 8, 4096, 128, 50_000),    # 4K
    (1003, 1, 64, 8, 2048, 128, 50_000),    # g = 8 (Qwen3-32B-shaped heads)
    (5, 2, 8, 2, 777, 100, 50_000),         # two sequences, ragged 4-bit stream
    (6, 1, 8, 8, 1111, 128, 20_000),        # MHA
    (7, 1, 6, 2, 500, 128, 50_000),         # g = 3
])
def test_decode_parity(hyq, seed, B, HQ, HKV, Lc, W, ppm):
    c = decode_case(seed, B, HQ, HKV, Lc, window=W, n_proxy=64, sink_frac=0.02, outlier_channels=3)
    got, want, _ = build_and_decode(c, Lc, W, ppm)
    assert_attention_close(got, want, what=f"L={Lc}")


@pytest.mark.parametrize("Lc,W,ppm,what", [
    (100, 128, 50_000, "context inside the window: no 4-bit rows"),
    (1, 128, 50_000, "single position: output is its value"),
    (600, 0, 0, "rho = 0, W = 0: pure 4-bit attention"),
    (600, 64, 1_000_000, "rho = 100%: all BF16"),
    (129, 128, 50_000, "P = 1"),
    (192, 128, 0, "exactly one 4-bit block"),
    (193, 128, 0, "one block plus one row"),
    (1000, 990, 50_000, "tail nearly the whole context"),
])
def test_decode_edge_cases(hyq, Lc, W, ppm, what):
    c = decode_case(31, 1, 8, 2, Lc, window=W, n_proxy=16, sink_frac=0.05)
    got, want, _ = build_and_decode(c, Lc, W, ppm, capacity=Lc + 64, period=64 if W < 990 else 64)
    assert_attention_close(got, want, what=what)
    if Lc == 1:
        np.testing.assert_array_equal(got[0, :4], c.v[0, 0, 0].double().numpy()[None].repeat(4, 0))


def test_decode_split_count_does_not_change_result(hyq):
    c = decode_case(41, 1, 32, 8, 3000, window=128, n_proxy=64, sink_frac=0.02)
    a, want, _ = build_and_decode(c, 3000, 128, 50_000, capacity=3000, len_hint=0)
    b, _, _ = build_and_decode(c, 3000, 128, 50_000, capacity=3000, len_hint=200)
    assert_attention_close(a, want)
    assert_attention_close(b, want)


@pytest.mark.parametrize("merge,splits", [(1, 0), (2, 2), (2, 5), (2, 16), (3, 3), (3, 19)])
def test_decode_every_merge_plan(hyq, merge, splits):
    """Direct (one block per KV head), cluster and workspace merges all give the
    oracle's result."""
    from hybrid_precision_quantized_gb300 import hyq_set_decode_plan
    c = decode_case(43, 1, 16, 4, 5000, window=128, n_proxy=64, sink_frac=0.02)
    hyq_set_decode_plan(merge, splits)
    try:
        got, want, _ = build_and_decode(c, 5000, 128, 50_000)
    finally:
        hyq_set_decode_plan(0, 0)
    assert_attention_close(got, want, what=f"plan {merge}/{splits}")


def test_decode_many_heads_direct_plan(hyq):
    """Enough (batch, KV head) pairs that the automatic plan uses one block each."""
    c = decode_case(44, 12, 16, 8, 700, window=128, n_proxy=16, sink_frac=0.02)
    got, want, _ = build_and_decode(c, 700, 128, 50_000)
    assert_attention_close(got, want, what="B=12 x 8 KV heads")


def test_decode_repeated_calls_reuse_workspace(hyq):
    c = decode_case(42, 1, 8, 2, 900, window=128, n_proxy=16, sink_frac=0.02)
    got, want, (cfg, layer, ws, out) = build_and_decode(c, 900, 128, 50_000)
    for _ in range(3):
        hyq_decode_attention(cfg, c.q.cuda(), layer.c, out, ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(to_np(out), got)   # deterministic, tickets reset


def test_decode_full_size_llama_32k(hyq):
    """Llama-3.1-8B-shaped layer at 32K context: every head against the oracle."""
    c = decode_case(1001, 1, 32, 8, 32768, window=128, n_proxy=64, sink_frac=0.02, outlier_channels=3)
    got, want, (cfg, layer, _, _) = build_and_decode(c, 32768, 128, 50_000, capacity=32768 + 64)
    cnt = layer.counts()[0].tolist()
    assert cnt[:4] == [32640, 1632, 128, 32768]
    assert_attention_close(got, want, what="32K")


@pytest.mark.parametrize("ppm,W,sink_frac",
                         [(r, w, 0.02) for r in (20_000, 50_000, 100_000) for w in (64, 128, 256)]
                         + [(50_000, 128, 0.01), (50_000, 128, 0.03)])
def test_decode_qwen32b_shaped_sweep_sampled(hyq, ppm, W, sink_frac):
    """Qwen3-32B-shaped decode: batch 4, 64/8 heads, 32K context, planted
    sinks with heavy-tailed (Student-t, 3 degrees of freedom) magnitudes, over
    the rho x W sweep.  The GPU computes every head; the oracle, which treats
    each (sequence, KV head) on its own, checks three pairs (24 query heads)
    in full: the first, the last and one drawn from a logged seed."""
    B, HQ, HKV, Lc = 4, 64, 8, 32768
    g = HQ // HKV
    c = decode_case(1004, B, HQ, HKV, Lc, window=W, n_proxy=64, sink_frac=sink_frac, heavy_tail=True)
    got, idx_np, (cfg, layer, _, _) = decode_gpu(c, Lc, W, ppm, capacity=Lc + 64)
    P = prefix_len(Lc, W)
    k = idx_np.shape[-1]
    assert layer.counts()[0].tolist()[:4] == [P, k, Lc - P, Lc]
    q, kk, vv = c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy()
    pairs, seed = sample_pairs(B, HKV, 3, f"qwen32b rho={ppm} W={W} sinks={sink_frac}")
    for b, kh in pairs:
        hs = slice(kh * g, (kh + 1) * g)
        want = hybrid_decode(q[b:b + 1, hs], kk[b:b + 1, kh:kh + 1], vv[b:b + 1, kh:kh + 1], Lc, P,
                             idx_np[b:b + 1, kh:kh + 1])
        assert_attention_close(got[b:b + 1, hs], want, what=f"rho={ppm} W={W} b={b} kvh={kh} seed={seed}")


def test_decode_pipeline_with_reselection(hyq):
    """Freeze, then 70 decode steps through HybridDecoder (append, proxy ring,
    re-selection at step 64, fused attention) against the oracle step by step."""
    B, HQ, HKV, W = 1, 8, 2, 128
    L0, steps = 700, 70
    cap = L0 + steps
    c = decode_case(51, B, HQ, HKV, cap, window=W, n_proxy=64, sink_frac=0.03)
    g = gen_for(51, "steps")
    qs = (torch.randn(steps, B, HQ, 128, generator=g) + 2.0 * c.u.repeat_interleave(HQ // HKV, 1)[None]).to(torch.bfloat16)
    k_all, v_all = c.k.clone(), c.v.clone()
    cfg = make_config(B, HQ, HKV, capacity=cap, window=W)
    k_src = torch.zeros(B, HKV, cap, 128, dtype=torch.bfloat16, device="cuda")
    v_src = torch.zeros_like(k_src)
    k_src[:, :, :L0] = k_all[:, :, :L0].cuda()
    v_src[:, :, :L0] = v_all[:, :, :L0].cuda()
    dec = HybridDecoder(cfg, k_src, v_src)
    q_tail = c.q_proxy.cuda()
    dec.freeze(L0, q_tail)
    k_np, v_np = k_all.double().numpy(), v_all.double().numpy()
    idx, _ = select_vertical(c.q_proxy.double().numpy(), k_np[:, :, :L0], L0, W, 50_000)
    P = L0 - W
    out = torch.empty(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    for s in range(steps):
        Lc = L0 + s + 1
        dec.step(qs[s].cuda(), k_all[:, :, Lc - 1].cuda().contiguous(), v_all[:, :, Lc - 1].cuda().contiguous(), out)
        if (s + 1) % 64 == 0:     # the decoder re-selected from the last 64 queries
            ring = qs[s - 63:s + 1].permute(1, 2, 0, 3).double().numpy()
            idx, S = select_vertical(ring, k_np[:, :, :Lc], Lc, W, 50_000)
            P = Lc - W
            got_idx = dec.layer.vl_idx()[:, :, :idx.shape[-1]].cpu().numpy()
            bnd = score_error_bound(ring, k_np[:, :, :Lc], P)
            for h in range(HKV):
                r = check_selection(S[0, h], bnd[0, h], idx.shape[-1], got_idx[0, h])
                assert r["ok"], r["reason"]
                if r["ambiguous"] == 0:
                    assert np.array_equal(got_idx[0, h], idx[0, h])
        if s in (0, 1, 62, 63, 64, 69):
            torch.cuda.synchronize()
            want = hybrid_decode(qs[s].double().numpy(), k_np, v_np, Lc, P, idx)
            assert_attention_close(to_np(out), want, what=f"step {s}")
    assert hyq_read_device_error(dec.layer.err()) == 0
    cnt = dec.layer.counts()[0].tolist()
    assert cnt[L.CNT_LEN] == L0 + steps and cnt[L.CNT_NTAIL] == W + steps - 64


def test_decode_append_full_tail_is_flagged(hyq):
    cfg = make_config(1, 2, 1, capacity=400, window=4, period=2)
    c = decode_case(61, 1, 2, 1, 10, window=4, n_proxy=2)
    layer = HybridLayer(cfg)
    layer.reset()
    idx = torch.zeros(1, 1, 1, dtype=torch.int32, device="cuda")
    hyq_rebuild(cfg, c.k.cuda(), c.v.cuda(), 10, idx, 0, layer.c)      # tail = 4 rows, capacity 6
    q = c.q.cuda()
    kn = c.k[:, :, 0].cuda().contiguous()
    for _ in range(3):
        hyq_decode_append(cfg, q, kn, kn, layer.c)
    torch.cuda.synchronize()
    assert layer.counts()[0, L.CNT_NTAIL].item() == 6
    assert hyq_read_device_error(layer.err()) & L.DEVERR_COUNT


def _two_layers(c, Lc, W, ppm, capacity):
    """Two identical layouts at context Lc (oracle partition) plus their inputs."""
    B, HQ = c.q.shape[:2]
    HKV = c.k.shape[1]
    cfg = make_config(B, HQ, HKV, capacity=capacity, window=W, rho_ppm=ppm)
    k_np = c.k.double().numpy()
    idx_np, _ = select_vertical(c.q_proxy.double().numpy(), k_np[:, :, :Lc], Lc, W, ppm)
    idx = torch.from_numpy(idx_np).to(torch.int32).cuda().contiguous()
    layers = []
    for _ in range(2):
        lay = HybridLayer(cfg)
        lay.reset()
        hyq_rebuild(cfg, c.k[:, :, :Lc].contiguous().cuda(), c.v[:, :, :Lc].contiguous().cuda(), Lc, idx,
                    idx_np.shape[-1], lay.c)
        layers.append(lay)
    return cfg, layers, idx_np


@pytest.mark.parametrize("plan", [(0, 0), (1, 0), (2, 4), (3, 7)])
@pytest.mark.parametrize("B,HQ,HKV", [(1, 8, 2), (2, 6, 2)])
def test_decode_step_equals_append_then_attention(hyq, plan, B, HQ, HKV):
    """The fused step leaves the same counters, tail, proxy ring and BF16 source
    rows as hyq_decode_append (bit-exact), and its output matches the oracle's
    attention over the cache with the new row, under every merge plan."""
    from hybrid_precision_quantized_gb300 import hyq_decode_step, hyq_set_decode_plan
    L0, W, ppm, steps = 900, 128, 50_000, 5
    cap = L0 + steps
    c = decode_case(71, B, HQ, HKV, cap, window=W, n_proxy=16, sink_frac=0.02)
    cfg, (la, lb), idx_np = _two_layers(c, L0, W, ppm, cap)
    srcs = []
    for _ in range(2):
        ks = torch.zeros(B, HKV, cap, 128, dtype=torch.bfloat16, device="cuda")
        vs = torch.zeros_like(ks)
        ks[:, :, :L0] = c.k[:, :, :L0].cuda()
        vs[:, :, :L0] = c.v[:, :, :L0].cuda()
        srcs.append((ks, vs))
    g = gen_for(71, "q-steps")
    qs = torch.randn(steps, B, HQ, 128, generator=g).to(torch.bfloat16)
    oa = torch.empty(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    ob = torch.empty_like(oa)
    k_np, v_np = c.k.double().numpy(), c.v.double().numpy()
    hyq_set_decode_plan(*plan)
    try:
        wsa, wsb = workspace(cfg, L.OP_DECODE, cap), workspace(cfg, L.OP_DECODE, cap)   # sized for the plan
        for s in range(steps):
            q = qs[s].cuda()
            kn = c.k[:, :, L0 + s].contiguous().cuda()
            vn = c.v[:, :, L0 + s].contiguous().cuda()
            hyq_decode_append(cfg, q, kn, vn, la.c, srcs[0][0], srcs[0][1])
            hyq_decode_attention(cfg, q, la.c, oa, wsa, cap)
            hyq_decode_step(cfg, q, kn, vn, lb.c, ob, wsb, srcs[1][0], srcs[1][1], cap)
            torch.cuda.synchronize()
            want = hybrid_decode(qs[s].double().numpy(), k_np, v_np, L0 + s + 1, L0 - W, idx_np)
            assert_attention_close(to_np(ob), want, what=f"fused step {s}, plan {plan}")
            assert_attention_close(to_np(oa), want, what=f"two calls step {s}")
    finally:
        hyq_set_decode_plan(0, 0)
    assert hyq_read_device_error(la.err()) == 0 and hyq_read_device_error(lb.err()) == 0
    assert torch.equal(la.counts(), lb.counts())
    n = la.counts()[0, L.CNT_NTAIL].item()
    assert n == W + steps
    assert torch.equal(la.tail_k()[:, :, :n], lb.tail_k()[:, :, :n])
    assert torch.equal(la.tail_v()[:, :, :n], lb.tail_v()[:, :, :n])
    assert torch.equal(la.q_ring()[:, :, :steps], lb.q_ring()[:, :, :steps])
    assert torch.equal(srcs[0][0], srcs[1][0]) and torch.equal(srcs[0][1], srcs[1][1])


def test_decode_step_full_tail_is_flagged(hyq):
    """A fused step with a full tail flags the error, leaves the layout alone
    and attends over the existing positions."""
    from hybrid_precision_quantized_gb300 import hyq_decode_step
    cfg = make_config(1, 2, 1, capacity=400, window=4, period=2)
    c = decode_case(62, 1, 2, 1, 12, window=4, n_proxy=2)
    layer = HybridLayer(cfg)
    layer.reset()
    idx = torch.zeros(1, 1, 1, dtype=torch.int32, device="cuda")
    hyq_rebuild(cfg, c.k[:, :, :10].contiguous().cuda(), c.v[:, :, :10].contiguous().cuda(), 10, idx, 0, layer.c)
    ws = workspace(cfg, L.OP_DECODE, 400)
    out = torch.empty(1, 2, 128, dtype=torch.bfloat16, device="cuda")
    q = c.q.cuda()
    for s in range(2):   # tail 4 -> 6 rows = capacity
        hyq_decode_step(cfg, q, c.k[:, :, 10 + s].contiguous().cuda(), c.v[:, :, 10 + s].contiguous().cuda(),
                        layer.c, out, ws)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) == 0
    before = layer.counts().clone()
    hyq_decode_step(cfg, q, c.k[:, :, 11].contiguous().cuda(), c.v[:, :, 11].contiguous().cuda(), layer.c, out, ws)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) & L.DEVERR_COUNT
    assert torch.equal(layer.counts(), before)
    want = hybrid_decode(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(), 12, 6, np.zeros((1, 1, 0), np.int64))
    assert_attention_close(to_np(out), want, what="full tail")


@pytest.mark.parametrize("fused", [False, True])
def test_decode_overlap_across_layers(hyq, fused):
    """With programmatic dependent launch on, calls alternating over two layers
    (the kernel before each call belongs to the other layer) give the same bits
    as with it off, fused step or attention alone, in a CUDA graph too."""
    from hybrid_precision_quantized_gb300 import hyq_decode_step, hyq_set_decode_overlap
    L0, W, ppm, steps = 1500, 128, 50_000, 4
    cap = L0 + steps
    cases = [decode_case(81 + i, 1, 8, 2, cap, window=W, n_proxy=16, sink_frac=0.02) for i in range(2)]
    g = gen_for(81, "q-steps")
    qs = torch.randn(steps, 2, 1, 8, 128, generator=g).to(torch.bfloat16).cuda()

    def run(overlap, graph):
        layers, outs = [], torch.zeros(steps, 2, 1, 8, 128, dtype=torch.bfloat16, device="cuda")
        cfg = None
        for c in cases:
            cfg, (la, _), _ = _two_layers(c, L0, W, ppm, cap)
            layers.append(la)
        ws = workspace(cfg, L.OP_DECODE, cap)
        kn = [[c.k[:, :, L0 + s].contiguous().cuda() for s in range(steps)] for c in cases]
        vn = [[c.v[:, :, L0 + s].contiguous().cuda() for s in range(steps)] for c in cases]

        def body():
            for s in range(steps):
                for i in range(2):
                    if fused:
                        hyq_decode_step(cfg, qs[s, i], kn[i][s], vn[i][s], layers[i].c, outs[s, i], ws, None, None, cap)
                    else:
                        hyq_decode_attention(cfg, qs[s, i], layers[i].c, outs[s, i], ws, cap)
        hyq_set_decode_overlap(overlap)
        try:
            if graph:
                st = torch.cuda.Stream()
                st.wait_stream(torch.cuda.current_stream())
                gr = torch.cuda.CUDAGraph()
                with torch.cuda.graph(gr, stream=st):
                    body()
                gr.replay()
            else:
                body()
            torch.cuda.synchronize()
        finally:
            hyq_set_decode_overlap(False)
        for la in layers:
            assert hyq_read_device_error(la.err()) == 0
        return outs.cpu(), [la.counts().cpu() for la in layers]

    ref, cref = run(False, False)
    for graph in (False, True):
        got, cgot = run(True, graph)
        assert torch.equal(got, ref), f"overlap changed the result (graph={graph})"
        assert all(torch.equal(a, b) for a, b in zip(cgot, cref))


@pytest.mark.parametrize("plan", [(0, 0), (1, 0), (3, 7)])
def test_decode_step_prefetch_changes_nothing(hyq, plan):
    """hyq_decode_step_prefetch (L2 prefetch of the next call's share) gives the
    same bits, counters, tail and proxy ring as hyq_decode_step, with the next
    layout another layer, the same layer, or none."""
    from hybrid_precision_quantized_gb300 import hyq_decode_step, hyq_decode_step_prefetch, hyq_set_decode_plan
    L0, W, ppm, steps = 1500, 128, 50_000, 3
    cap = L0 + steps
    cases = [decode_case(91 + i, 1, 8, 2, cap, window=W, n_proxy=16, sink_frac=0.02) for i in range(2)]
    g = gen_for(91, "q-steps")
    qs = torch.randn(steps, 2, 1, 8, 128, generator=g).to(torch.bfloat16).cuda()
    kn = [[c.k[:, :, L0 + s].contiguous().cuda() for s in range(steps)] for c in cases]
    vn = [[c.v[:, :, L0 + s].contiguous().cuda() for s in range(steps)] for c in cases]

    def run(mode):
        hyq_set_decode_plan(*plan)
        try:
            layers, cfg = [], None
            for c in cases:
                cfg, (la, _), _ = _two_layers(c, L0, W, ppm, cap)
                layers.append(la)
            ws = workspace(cfg, L.OP_DECODE, cap)
            outs = torch.zeros(steps, 2, 1, 8, 128, dtype=torch.bfloat16, device="cuda")
            for s in range(steps):
                for i in range(2):
                    lay = layers[i].c
                    if mode == "plain":
                        hyq_decode_step(cfg, qs[s, i], kn[i][s], vn[i][s], lay, outs[s, i], ws, None, None, cap)
                    else:
                        nxt = {"other": layers[1 - i].c, "self": lay, "none": None}[mode]
                        hyq_decode_step_prefetch(cfg, qs[s, i], kn[i][s], vn[i][s], lay, nxt, outs[s, i], ws,
                                                 None, None, cap)
            torch.cuda.synchronize()
        finally:
            hyq_set_decode_plan(0, 0)
        for la in layers:
            assert hyq_read_device_error(la.err()) == 0
        return (outs.cpu(), [la.counts().cpu() for la in layers], [la.tail_k().cpu() for la in layers],
                [la.q_ring().cpu() for la in layers])

    ref = run("plain")
    for mode in ("other", "self", "none"):
        got = run(mode)
        assert torch.equal(got[0], ref[0]), mode
        for a, b in zip(got[1:], ref[1:]):
            assert all(torch.equal(x, y) for x, y in zip(a, b)), mode


def test_frozen_mode_age_tail(hyq):
    """Frozen mode (Algorithm 4 as written): the vertical-line set chosen at
    freeze stays; every 64 tokens hyq_age_tail moves the tail rows older than
    the window into the 4-bit stream.  After each aging the counters, the tail
    rows and every stream row (codes, scales, zeros: bit-exact with the
    oracle quantiser) equal the partition at the new length with the frozen
    index set, and the attention matches the oracle over that partition."""
    from hybrid_precision_quantized_gb300 import hyq_age_tail, hyq_decode_step
    from tests.test_gpu_quant import _check_positional
    B, HQ, HKV, W, ppm, T = 2, 8, 2, 128, 50_000, 64
    L0, periods = 900, 2
    cap = L0 + periods * T
    c = decode_case(95, B, HQ, HKV, cap, window=W, n_proxy=16, sink_frac=0.02)
    cfg, (lay, _), idx_np = _two_layers(c, L0, W, ppm, cap)
    k = idx_np.shape[-1]
    ks = torch.zeros(B, HKV, cap, 128, dtype=torch.bfloat16, device="cuda")
    vs = torch.zeros_like(ks)
    ks[:, :, :L0] = c.k[:, :, :L0].cuda()
    vs[:, :, :L0] = c.v[:, :, :L0].cuda()
    ws = workspace(cfg, L.OP_DECODE, cap)
    g = gen_for(95, "q-steps")
    k_np, v_np = c.k.double().numpy(), c.v.double().numpy()
    out = torch.empty(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    Lc = L0
    for _ in range(periods):
        for _ in range(T):
            q = torch.randn(B, HQ, 128, generator=g).to(torch.bfloat16)
            hyq_decode_step(cfg, q.cuda(), c.k[:, :, Lc].contiguous().cuda(), c.v[:, :, Lc].contiguous().cuda(),
                            lay.c, out, ws, ks, vs, cap)
            Lc += 1
        torch.cuda.synchronize()
        assert layer_counts(lay)[:3] == [L0 - W + (Lc - L0 - T), k, W + T]
        # the last step's attention over the 4-bit stream of the last aging
        P_before = Lc - 1 - (W + T - 1)
        want = hybrid_decode(q.double().numpy(), k_np, v_np, Lc, P_before, idx_np)
        assert_attention_close(to_np(out), want, what=f"before aging, L={Lc}")
        hyq_age_tail(cfg, lay.c)
        torch.cuda.synchronize()
        assert hyq_read_device_error(lay.err()) == 0
        P = Lc - W
        assert layer_counts(lay)[:4] == [P, k, W, Lc]
        for b in range(B):
            for h in range(HKV):
                _check_positional(lay, b, h, P, c.k[b, h].double().numpy(), c.v[b, h].double().numpy(),
                                  idx_np[b, h])
                assert torch.equal(lay.tail_k()[b, h, :W].cpu(), c.k[b, h, P:Lc])
                assert torch.equal(lay.tail_v()[b, h, :W].cpu(), c.v[b, h, P:Lc])
        q = torch.randn(B, HQ, 128, generator=g).to(torch.bfloat16)
        hyq_decode_attention(cfg, q.cuda(), lay.c, out, ws, cap)
        torch.cuda.synchronize()
        want = hybrid_decode(q.double().numpy(), k_np, v_np, Lc, P, idx_np)
        assert_attention_close(to_np(out), want, what=f"after aging, L={Lc}")


def test_age_tail_without_room_is_flagged(hyq):
    """A stream without room for the aged rows leaves the layout unchanged and
    sets HYQ_DEVERR_COUNT."""
    from hybrid_precision_quantized_gb300 import hyq_age_tail, hyq_decode_step
    B, HQ, HKV, W, ppm, L0 = 1, 4, 1, 64, 0, 600
    cap = L0 + 64
    c = decode_case(96, B, HQ, HKV, cap, window=W, n_proxy=8)
    cfg, (lay, _), _ = _two_layers(c, L0, W, ppm, cap)
    ws = workspace(cfg, L.OP_DECODE, cap)
    out = torch.empty(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    for t in range(64):
        hyq_decode_step(cfg, c.q.cuda(), c.k[:, :, L0 + t].contiguous().cuda(),
                        c.v[:, :, L0 + t].contiguous().cuda(), lay.c, out, ws, None, None, cap)
    torch.cuda.synchronize()
    assert layer_counts(lay)[:3] == [L0 - W, 0, W + 64]
    stream_rows = -(-cap // 64) * 64           # the 4-bit stream's capacity in rows
    lay.counts()[0, L.CNT_NQ] = stream_rows - 10   # as if the stream were nearly full
    before = layer_counts(lay)
    hyq_age_tail(cfg, lay.c)
    torch.cuda.synchronize()
    assert hyq_read_device_error(lay.err()) & L.DEVERR_COUNT
    assert layer_counts(lay) == before


def layer_counts(lay):
    return lay.counts()[0].tolist()


def test_decode_qwen8b_shaped_batch16_32k_sampled(hyq):
    """Qwen3-8B-shaped batched decode at full size: batch 16, 32/8 heads, 32K
    context, W 128, rho 5%, the launch configuration the benchmark times
    (automatic plan).  Each sequence is its own seeded case; the oracle picks
    each sequence's vertical lines, the GPU decodes all 16 x 32 heads, and
    three (sequence, KV head) pairs are checked in full: the first, the last
    and one drawn from a logged seed."""
    B, HQ, HKV, Lc, W, ppm = 16, 32, 8, 32768, 128, 50_000
    g = HQ // HKV
    P = prefix_len(Lc, W)
    cases = [decode_case(1300 + b, 1, HQ, HKV, Lc, window=W, n_proxy=64, sink_frac=0.02, outlier_channels=3)
             for b in range(B)]
    idx_np = np.concatenate([select_vertical(c.q_proxy.double().numpy(), c.k.double().numpy(), Lc, W, ppm)[0]
                             for c in cases])
    cfg = make_config(B, HQ, HKV, capacity=Lc, window=W, rho_ppm=ppm)
    layer = HybridLayer(cfg)
    layer.reset()
    kd = torch.cat([c.k for c in cases]).cuda()
    vd = torch.cat([c.v for c in cases]).cuda()
    idx = torch.from_numpy(idx_np).to(torch.int32).cuda().contiguous()
    hyq_rebuild(cfg, kd, vd, Lc, idx, idx_np.shape[-1], layer.c)
    del kd, vd
    q = torch.cat([c.q for c in cases])
    out = torch.empty(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    ws = workspace(cfg, L.OP_DECODE, Lc)
    hyq_decode_attention(cfg, q.cuda(), layer.c, out, ws, Lc)
    torch.cuda.synchronize()
    assert hyq_read_device_error(layer.err()) == 0
    got = to_np(out)
    pairs, seed = sample_pairs(B, HKV, 3, "qwen8b batch16")
    for b, kh in pairs:
        c = cases[b]
        hs = slice(kh * g, (kh + 1) * g)
        want = hybrid_decode(c.q.double().numpy()[:, hs], c.k.double().numpy()[:, kh:kh + 1],
                             c.v.double().numpy()[:, kh:kh + 1], Lc, P, idx_np[b:b + 1, kh:kh + 1])
        assert_attention_close(got[b:b + 1, hs], want, what=f"b={b} kvh={kh} seed={seed}")
