"""Multi-layer decode runner: one decode period (``period`` tokens) over many
layers, captured as CUDA graphs so that host overhead does not gate the
kernels.

For every token t of the period but the last, one graph holds the fused
decode step (append + attention, hyq_decode_step) of every layer; with
``prefetch_next`` each step also warms L2 with the next layer's share
(hyq_decode_step_prefetch; the layer after the last is the first).  In
``mode="frozen"`` (Algorithm 4 as written) the last token's maintenance is
hyq_age_tail (the tail rows older than the window go to the 4-bit stream,
the vertical-line set chosen at freeze stays) instead of re-selection and
rebuild; the reset then also restores the tail rows the aging shifted.
With ``score="mass"`` re-selection uses the softmax-mass score of Eq. 4
(hyq_select_vertical_mass) instead of Algorithm 1's summed logits.  At the
last token two graphs are captured: the appends of all layers with the
re-selection and rebuild of every layer, then the decode attention of all
layers (maintenance sits between the append and the attention).  A reset graph restores the
layer counters to the start of the period, so a period can be replayed any
number of times on the same synthetic inputs (the work of every replay is
identical: the same positions are re-appended and the same layout rebuilt).
"""
from __future__ import annotations

import torch

from . import _lib as L
from .cache import HybridLayer, workspace


class PeriodRunner:
    """Decode ``period`` tokens through ``n_layers`` independent layers.

    k_srcs / v_srcs : per-layer BF16 caches [B, HKV, ld, 128] (device)
    q_tok           : [period, n_layers, B, HQ, 128] bf16 (device or pinned host)
    k_tok / v_tok   : [period, n_layers, B, HKV, 128] bf16
    """

    def __init__(self, cfg, k_srcs, v_srcs, L0: int, device="cuda", prefetch_next: bool = False,
                 mode: str = "reselect", score: str = "logits"):
        if mode not in ("reselect", "frozen"):
            raise ValueError(f"mode must be 'reselect' or 'frozen', not {mode!r}")
        if score not in ("logits", "mass"):
            raise ValueError(f"score must be 'logits' or 'mass', not {score!r}")
        self.select = L.hyq_select_vertical_mass if score == "mass" else L.hyq_select_vertical
        self.cfg = cfg
        self.prefetch_next = prefetch_next
        self.frozen = mode == "frozen"
        self.tail0 = None
        self.n_layers = len(k_srcs)
        self.k_srcs, self.v_srcs = k_srcs, v_srcs
        self.L0 = L0
        self.L_end = L0 + cfg.period
        self.layers = [HybridLayer(cfg, device) for _ in k_srcs]
        self.ws_sel = workspace(cfg, L.OP_SELECT_MASS if score == "mass" else L.OP_SELECT, self.L_end, device)
        self.ws_dec = workspace(cfg, L.OP_DECODE, self.L_end, device)
        kmax = max(1, L.hyq_vl_count(cfg, max(0, cfg.capacity - cfg.window)))
        self.idx = [torch.zeros(cfg.batch, cfg.num_kv_heads, kmax, dtype=torch.int32, device=device)
                    for _ in k_srcs]
        B, HQ, HKV, T = cfg.batch, cfg.num_q_heads, cfg.num_kv_heads, cfg.period
        self.q_tok = torch.zeros(T, self.n_layers, B, HQ, 128, dtype=torch.bfloat16, device=device)
        self.k_tok = torch.zeros(T, self.n_layers, B, HKV, 128, dtype=torch.bfloat16, device=device)
        self.v_tok = torch.zeros_like(self.k_tok)
        self.out = torch.zeros(T, self.n_layers, B, HQ, 128, dtype=torch.bfloat16, device=device)
        self.counts0 = None
        self.graphs = None
        self.launches_per_period = 0

    def freeze(self, q_tail: torch.Tensor):
        """Build every layer's layout for the first L0 positions, choosing the
        vertical-line set from ``q_tail`` [n_layers, B, HQ, T, 128]."""
        for li, lay in enumerate(self.layers):
            lay.reset()
            k = self.select(self.cfg, q_tail[li], q_tail.shape[3], self.k_srcs[li], self.L0, self.idx[li],
                            self.ws_sel)
            L.hyq_rebuild(self.cfg, self.k_srcs[li], self.v_srcs[li], self.L0, self.idx[li], k, lay.c)
        torch.cuda.synchronize()
        self.counts0 = torch.stack([lay.counts().clone() for lay in self.layers])
        if self.frozen:
            self.tail0 = [(lay.tail_k().clone(), lay.tail_v().clone()) for lay in self.layers]

    # --- the per-token work, as eager calls (captured below) ---------------
    def _reset(self):
        for li, lay in enumerate(self.layers):
            lay.counts().copy_(self.counts0[li])
            if self.tail0 is not None:
                lay.tail_k().copy_(self.tail0[li][0])
                lay.tail_v().copy_(self.tail0[li][1])

    def _appends(self, t):
        n = 0
        for li, lay in enumerate(self.layers):
            L.hyq_decode_append(self.cfg, self.q_tok[t, li], self.k_tok[t, li], self.v_tok[t, li], lay.c,
                                self.k_srcs[li], self.v_srcs[li])
            n += 1
            if t == self.cfg.period - 1 and self.frozen:
                L.hyq_age_tail(self.cfg, lay.c)
                n += 3
            elif t == self.cfg.period - 1:
                ring = lay.q_ring()
                k = self.select(self.cfg, ring, ring.shape[2], self.k_srcs[li], self.L_end, self.idx[li],
                                self.ws_sel)
                L.hyq_rebuild(self.cfg, self.k_srcs[li], self.v_srcs[li], self.L_end, self.idx[li], k, lay.c)
                if self.select is L.hyq_select_vertical_mass:
                    # two passes and the top-k, plus a group-sum kernel when
                    # the proxy rows of a KV group exceed one 256-row group
                    rows = self.cfg.num_q_heads // self.cfg.num_kv_heads * ring.shape[2]
                    n_sel = 3 if rows <= 256 else 4
                else:
                    n_sel = 6 if self.cfg.vl_mode == L.VL_PER_QUERY_HEAD else 3
                n += (n_sel if k > 0 else 0) + \
                    (3 if self.L_end - self.cfg.window > 0 else 1)  # rows, marks, gather
        return n

    def _decodes(self, t):
        for li, lay in enumerate(self.layers):
            L.hyq_decode_attention(self.cfg, self.q_tok[t, li], lay.c, self.out[t, li], self.ws_dec, self.L_end)
        return self.n_layers

    def _steps(self, t):
        for li, lay in enumerate(self.layers):
            if self.prefetch_next:
                nxt = self.layers[(li + 1) % self.n_layers].c
                L.hyq_decode_step_prefetch(self.cfg, self.q_tok[t, li], self.k_tok[t, li], self.v_tok[t, li],
                                           lay.c, nxt, self.out[t, li], self.ws_dec, self.k_srcs[li],
                                           self.v_srcs[li], self.L_end)
            else:
                L.hyq_decode_step(self.cfg, self.q_tok[t, li], self.k_tok[t, li], self.v_tok[t, li], lay.c,
                                  self.out[t, li], self.ws_dec, self.k_srcs[li], self.v_srcs[li], self.L_end)
        return self.n_layers

    def _fused(self, t):
        return t < self.cfg.period - 1

    def capture(self):
        """Run one period eagerly (warm-up, attributes), then capture graphs."""
        s = torch.cuda.Stream()
        s.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(s):
            self._reset()
            for t in range(self.cfg.period):
                if self._fused(t):
                    self._steps(t)
                else:
                    self._appends(t)
                    self._decodes(t)
        torch.cuda.synchronize()
        self.g_reset = torch.cuda.CUDAGraph()
        with torch.cuda.graph(self.g_reset):
            self._reset()
        self.g_app, self.g_dec = [], []
        n = 0
        for t in range(self.cfg.period):
            gd = torch.cuda.CUDAGraph()
            if self._fused(t):
                ga = None
                with torch.cuda.graph(gd):
                    n += self._steps(t)
            else:
                ga = torch.cuda.CUDAGraph()
                with torch.cuda.graph(ga):
                    n += self._appends(t)
                with torch.cuda.graph(gd):
                    n += self._decodes(t)
            self.g_app.append(ga)
            self.g_dec.append(gd)
        self.launches_per_period = n
        torch.cuda.synchronize()

    def run_period(self, dec_events=None):
        """Replay one period.  ``dec_events`` (optional) is a list of
        (start, end) CUDA event pairs, one per token, recorded around the
        decode graph of that token (fused steps, or the attention alone at
        the maintenance token)."""
        self.g_reset.replay()
        for t in range(self.cfg.period):
            if self.g_app[t] is not None:
                self.g_app[t].replay()
            if dec_events is not None:
                dec_events[t][0].record()
            self.g_dec[t].replay()
            if dec_events is not None:
                dec_events[t][1].record()

    def run_period_host(self, q_host, k_host, v_host, out_host):
        """One period with inputs and outputs in (pinned) host memory: every
        token's inputs are copied in before its kernels and its outputs
        copied out after them."""
        self.g_reset.replay()
        for t in range(self.cfg.period):
            self.q_tok[t].copy_(q_host[t], non_blocking=True)
            self.k_tok[t].copy_(k_host[t], non_blocking=True)
            self.v_tok[t].copy_(v_host[t], non_blocking=True)
            if self.g_app[t] is not None:
                self.g_app[t].replay()
            self.g_dec[t].replay()
            out_host[t].copy_(self.out[t], non_blocking=True)
