"""Decode attention for callers that cannot allocate device memory.

Some callers have no way to give the library a workspace: plugins and
embedding runtimes that pass an attention op only its inputs and outputs, and
hot loops that must not call cudaMalloc (it synchronises the device and can
fail under memory pressure).  hyq_decode_attention_noalloc serves them from a
fixed library-owned device array.  These tests call it through the C ABI and
check it, twice in a row (the array is shared and keeps the previous call's
contents), against the workspace entry point -- the same kernel with the same
split plan, so the outputs must be identical bit for bit -- and against the
oracle's float64 hybrid attention within the decode tolerance.
"""
import numpy as np
import pytest
import torch

from gen import decode_case
from hybrid_precision_quantized_gb300 import (HybridLayer, HyqError, hyq_decode_attention,
                                              hyq_decode_attention_noalloc, hyq_read_device_error,
                                              hyq_rebuild, hyq_workspace_size, make_config, workspace)
from hybrid_precision_quantized_gb300 import _lib as L
from oracle.attention import hybrid_decode
from oracle.select import prefix_len, select_vertical
from tests.gpu_util import assert_attention_close, to_np

pytestmark = pytest.mark.gpu


def _layer(seed, B, HQ, HKV, Lc):
    c = decode_case(seed, B, HQ, HKV, Lc, window=128, n_proxy=64, sink_frac=0.02, outlier_channels=3)
    cfg = make_config(B, HQ, HKV, capacity=Lc, window=128)
    layer = HybridLayer(cfg)
    layer.reset()
    idx_np, _ = select_vertical(c.q_proxy.double().numpy(), c.k.double().numpy(), Lc, 128, 50_000)
    idx = torch.from_numpy(idx_np).to(torch.int32).cuda().contiguous()
    hyq_rebuild(cfg, c.k.cuda(), c.v.cuda(), Lc, idx, idx_np.shape[-1], layer.c)
    return c, cfg, layer, idx_np


@pytest.mark.parametrize("seed,B,HQ,HKV,Lc", [(1001, 1, 32, 8, 4096), (77, 2, 8, 2, 1500)])
def test_noalloc_matches_workspace_entry_point_twice(hyq, seed, B, HQ, HKV, Lc):
    c, cfg, layer, idx_np = _layer(seed, B, HQ, HKV, Lc)
    q = c.q.cuda()
    ref = torch.empty(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    hyq_decode_attention(cfg, q, layer.c, ref, workspace(cfg, L.OP_DECODE, Lc), Lc)
    want = hybrid_decode(c.q.double().numpy(), c.k.double().numpy(), c.v.double().numpy(), Lc,
                         prefix_len(Lc, 128), idx_np)
    for call in range(2):
        out = torch.full((B, HQ, 128), float("nan"), dtype=torch.bfloat16, device="cuda")
        hyq_decode_attention_noalloc(cfg, q, layer.c, out, Lc)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), f"no-alloc call {call} differs from the workspace entry point"
        assert_attention_close(to_np(out), want, what=f"no-alloc call {call} against the oracle")
    assert hyq_read_device_error(layer.err()) == 0


def test_noalloc_rejects_shapes_beyond_its_scratch(hyq):
    B, HQ, HKV, Lc = 512, 8, 8, 256     # 4096 (batch, KV head) pairs: partials exceed 4 MiB
    cfg = make_config(B, HQ, HKV, capacity=Lc, window=128)
    assert hyq_workspace_size(cfg, L.OP_DECODE, Lc) > L.NOALLOC_SCRATCH_BYTES
    layer = HybridLayer(cfg)
    layer.reset()
    q = torch.zeros(B, HQ, 128, dtype=torch.bfloat16, device="cuda")
    out = torch.zeros_like(q)
    with pytest.raises(HyqError) as e:
        hyq_decode_attention_noalloc(cfg, q, layer.c, out, Lc)
    assert e.value.status == 3            # HYQ_ERR_WORKSPACE, nothing launched
    torch.cuda.synchronize()
    assert not out.any()
